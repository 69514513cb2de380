"""Pins for the oracle's quantiser (bf16 -> NVFP4) that do not go through
its own arithmetic: torch's float8_e4m3fn cast, the e2m1 table's midpoints
written out by hand, hand-worked blocks, and the round-trip error bound."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_linear_gb300.inputs import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_e4m3_round_matches_torch_float8_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([np.exp2(rng.uniform(-12, 8.8, 4000)).astype(np.float32),
                        np.float32([0.0, 2.0 ** -9, 2.0 ** -10, 1.5 * 2.0 ** -10, 448.0, 416.0,
                                    432.0, 440.0, 9.5, 10.5, 0.0546875])])
    v = v[v <= 448.0]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_round(x) for x in v], np.uint8)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


def test_e4m3_round_saturates():
    for v in (448.0, 449.0, 464.0, 1e6, float("inf")):
        assert oracle.e4m3_round(v) == 0x7E


# |t| -> code magnitude, including every midpoint of the e2m1 grid
# {0, 0.5, 1, 1.5, 2, 3, 4, 6}: ties go to the even code (mantissa bit 0).
E2M1_CASES = [(0.0, 0), (0.2, 0), (0.25, 0), (0.26, 1), (0.5, 1), (0.75, 2), (0.74, 1),
              (1.0, 2), (1.25, 2), (1.26, 3), (1.5, 3), (1.75, 4), (2.0, 4), (2.5, 4),
              (2.51, 5), (3.0, 5), (3.5, 6), (3.49, 5), (4.0, 6), (5.0, 6), (5.01, 7),
              (6.0, 7), (6.5, 7), (1e9, 7)]


@pytest.mark.parametrize("t,code", E2M1_CASES)
def test_e2m1_round_table(t, code):
    assert oracle.e2m1_round(t) == code
    assert oracle.e2m1_round(-t) == code | 8


def test_e2m1_round_keeps_sign_of_zero():
    assert oracle.e2m1_round(-0.0) == 8
    assert oracle.e2m1_round(-0.1) == 8
    assert oracle.e2m1_round(0.0) == 0


def _bits(rows):
    return f32_to_bf16_bits(np.asarray(rows, np.float32))


def test_hand_worked_blocks():
    doc = json.load(open(os.path.join(GOLDEN, "quantize_blocks.json")))
    for c in doc["cases"]:
        wp, ws, gs = oracle.quantize(_bits(c["w"]))
        assert gs == np.float32(c["global_scale"]), c["name"]
        assert np.array_equal(ws, np.asarray(c["scale"], np.uint8)), c["name"]
        codes = np.stack([wp & 0xF, wp >> 4], -1).reshape(c["N"], c["K"])
        assert np.array_equal(codes, np.asarray(c["codes"], np.uint8)), c["name"]


def test_round_trip_error_bound():
    """Dequantising the quantiser's output with the pinned decoders gives
    every weight back within its block's e2m1 half-step (at most 1 unit of
    s/gs, the gap between 4 and 6 halved), and the block maximum maps to a
    code of magnitude >= 4 whenever the block scale did not round to 0."""
    rng = np.random.default_rng(5)
    w = rng.standard_normal((24, 256)).astype(np.float32)
    w[3] *= 50.0
    w[7, :16] = 0.0
    w[9] *= 1e-3
    bits = f32_to_bf16_bits(w)
    wv = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    wp, ws, gs = oracle.quantize(bits)
    e2m1 = np.array([oracle.e2m1(c) for c in range(16)])
    codes = np.stack([wp & 0xF, wp >> 4], -1).reshape(w.shape)
    scale = np.repeat(torch.from_numpy(ws).view(torch.float8_e4m3fn).float().numpy()
                      .astype(np.float64), 16, axis=1)
    deq = e2m1[codes] * scale / np.float64(gs)
    step = scale / np.float64(gs)
    err = np.abs(deq - wv)
    assert gs == np.float32(448.0) / np.float32(np.abs(wv).max())
    # Blocks with a normal e4m3 scale (>= 2^-6): the scale is within 1/16 of
    # (amax_block * gs) / 6, so the block maximum lands within [5.6, 6.4]
    # and every weight is within the widest e2m1 half-gap (1) of a code.
    normal = np.repeat(scale.reshape(24, 16, 16)[..., 0] >= 2.0 ** -6, 16, axis=1)
    assert np.all(err[normal] <= step[normal] + 1e-12)
    # Subnormal or zero scales (tiny blocks next to a large tensor maximum):
    # the format's coarse scale grid only bounds the error by the block's
    # own magnitude plus one step.
    amax_b = np.repeat(np.abs(wv).reshape(24, 16, 16).max(-1), 16, axis=1)
    assert np.all(err <= amax_b + step + 1e-12)
    blocks = np.abs(wv).reshape(24, 16, 16)
    mag = (codes & 7).reshape(24, 16, 16)
    top = np.take_along_axis(mag, blocks.argmax(-1)[..., None], -1)[..., 0]
    nrm = scale.reshape(24, 16, 16)[..., 0] >= 2.0 ** -6
    assert nrm.sum() > 300
    assert np.all(top[nrm] == 7)        # the block maximum maps to 6 (code 7)
    assert np.all(codes.reshape(24, 16, 16)[ws == 0] == 0)


def test_bad_shapes():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((2, 20), np.uint16))
