"""Pins for the oracle's format decoders and rounding.

Every expectation here comes from outside the oracle: the printed e2m1 table,
the OCP e4m3 special values, torch's own float8_e4m3fn / bfloat16 decoders and
conversion (library routines), or properties of the formats.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_e2m1_matches_printed_table():
    table = _load("e2m1_table.json")["code_to_value"]
    e2m1, _ = oracle.decode_tables()
    for code, value in table.items():
        got = e2m1[int(code)]
        assert got == value, (code, got, value)
        # -0 has its sign bit set: code 8 must decode to a negative zero
        assert math.copysign(1.0, got) == math.copysign(1.0, value)
    assert oracle.e2m1(7) == 6.0 and oracle.e2m1(15) == -6.0


def test_e2m1_table_properties():
    e2m1, _ = oracle.decode_tables()
    # sign bit symmetry and strict increase of the magnitudes 0..7
    assert np.all(e2m1[8:] == -e2m1[:8])
    assert np.all(np.diff(e2m1[:8]) > 0)
    # every value is exactly representable in bf16 (at most 2 significant bits)
    assert np.all(np.float64(torch.tensor(e2m1).to(torch.bfloat16).double().numpy())
                  == e2m1)


def test_e4m3_all_patterns_match_torch_float8():
    _, e4m3 = oracle.decode_tables()
    bits = torch.arange(256, dtype=torch.uint8)
    ref = bits.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(e4m3), nan)
    assert nan.sum() == 2                          # 0x7f and 0xff only
    assert np.array_equal(e4m3[~nan], ref[~nan])
    # signed zeros agree too
    assert np.array_equal(np.signbit(e4m3[~nan]), np.signbit(ref[~nan]))


def test_e4m3_printed_specials():
    spec = _load("e4m3_specials.json")
    for b, v in spec["bits_to_value"].items():
        got = oracle.e4m3(int(b, 16))
        assert got == v and math.copysign(1, got) == math.copysign(1, v), b
    for b in spec["nan_bits"]:
        assert math.isnan(oracle.e4m3(int(b, 16)))


def test_e4m3_monotone_and_max():
    _, e4m3 = oracle.decode_tables()
    pos = e4m3[:0x7f]
    assert np.all(np.diff(pos) > 0)
    assert pos.max() == 448.0
    # the synthetic scale range 0x20..0x50 is exactly [2^-3, 2^3]
    assert e4m3[0x20] == 0.125 and e4m3[0x50] == 8.0


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(123)
    bits = np.concatenate([rng.integers(0, 65536, 20000, dtype=np.int64),
                           [0, 0x8000, 0x0001, 0x7f7f, 0x7f80, 0xff80]])
    ref = torch.from_numpy(bits.astype(np.uint16).view(np.int16)) \
        .view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _torch_bf16_bits(vals32):
    t = torch.from_numpy(np.asarray(vals32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rne_matches_torch_random_and_ties():
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)
    # force exact ties (low half 0x8000) on both parities, and near-ties
    ties = (u[:2000] & 0xffff0000) | 0x8000
    near = (u[2000:4000] & 0xffff0000) | np.uint32(0x7fff)
    vals = np.concatenate([u, ties.astype(np.uint32), near.astype(np.uint32)]).view(
        np.float32)
    finite = np.isfinite(vals)
    vals = vals[finite]
    ref = _torch_bf16_bits(vals)
    got = oracle.to_bf16_bits(vals.astype(np.float64))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("value,expected", [
    (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
    (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
    # 1 + 2^-8 is the exact midpoint between 1 and 1 + 2^-7: ties to even -> 1
    (1.0 + 2.0**-8, 0x3F80),
    # 1 + 3*2^-8 is the midpoint between 1+2^-7 (odd) and 1+2^-6: rounds up
    (1.0 + 3 * 2.0**-8, 0x3F82),
    # the largest float32 rounds up to infinity in bf16
    (float(np.finfo(np.float32).max), 0x7F80),
])
def test_rne_special_values(value, expected):
    assert oracle.f32_to_bf16(value) == expected


def test_rne_nan_stays_nan():
    b = oracle.f32_to_bf16(float("nan"))
    assert (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0
