"""Pins for the oracle's linear layer and SwiGLU.

The expectations come from hand-worked examples (tests/golden/hand_blocks.json),
closed forms, exact rational arithmetic on tiny inputs with decoders that do
not go through the oracle (the printed e2m1 table and torch's float8 decoder),
and symmetries of the definition.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_linear_gb300.inputs import make_linear, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


E2M1 = {int(k): v for k, v in _golden("e2m1_table.json")["code_to_value"].items()}


def _e4m3_torch(b):
    return float(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn)
                 .to(torch.float64)[0])


def _bf16_torch(bits):
    return float(torch.tensor([int(bits)], dtype=torch.int32).to(torch.int16)
                 .view(torch.bfloat16).to(torch.float64)[0])


def exact_linear(x_bits, w_packed, w_scale, gs):
    """y in exact rationals, decoding with the printed table and torch."""
    M, K = x_bits.shape
    N = w_packed.shape[0]
    gsf = Fraction(float(np.float32(gs)))
    y = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        w = []
        for k in range(K):
            byte = int(w_packed[n, k // 2])
            code = (byte >> (4 * (k % 2))) & 0xF
            w.append(Fraction(E2M1[code]) * Fraction(_e4m3_torch(int(w_scale[n, k // 16])))
                     / gsf)
        for m in range(M):
            y[m][n] = sum(Fraction(_bf16_torch(x_bits[m, k])) * w[k] for k in range(K))
    return y


@pytest.mark.parametrize("case", _golden("hand_blocks.json")["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked_examples(case):
    x = np.array(case["x_bits"], np.uint16)
    wp = np.array(case["w_packed"], np.uint8)
    ws = np.array(case["w_scale"], np.uint8)
    y, a = oracle.linear_f64(x, wp, ws, case["global_scale"], threads=1)
    assert np.array_equal(y, np.array(case["y"], np.float64)), (y, case["y"])
    assert np.all(a >= np.abs(y))


def test_closed_form_equal_codes_and_scales():
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 64
    x_bits = f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    for code in (1, 5, 7, 9, 14):
        for sbits in (0x20, 0x38, 0x4b, 0x01):
            byte = code | (code << 4)
            wp = np.full((N, K // 2), byte, np.uint8)
            ws = np.full((N, K // 16), sbits, np.uint8)
            gs = np.float32(448.0 / 6.0)
            y, _ = oracle.linear_f64(x_bits, wp, ws, gs, threads=2)
            xs = np.array([[_bf16_torch(b) for b in row] for row in x_bits])
            coef = E2M1[code] * _e4m3_torch(sbits) / float(gs)
            expect = coef * xs.sum(axis=1)
            # fp64 rounding of K-term sums: well inside 1e-12 relative
            np.testing.assert_allclose(y, np.repeat(expect[:, None], N, 1),
                                       rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("seed,M,N,K", [(0, 1, 4, 16), (1, 3, 8, 64), (2, 2, 3, 48),
                                         (3, 3, 5, 32)])
def test_brute_force_exact_rationals(seed, M, N, K):
    t = make_linear(M, N, K, seed)
    y, a = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale,
                             threads=1)
    exact = exact_linear(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    for m in range(M):
        for n in range(N):
            # each of the K products and sums rounds once in fp64
            bound = 4 * K * 2.0**-53 * a[m, n] + 1e-300
            assert abs(Fraction(y[m, n]) - exact[m][n]) <= Fraction(bound), (m, n)


def test_sign_flip_negates_exactly():
    t = make_linear(4, 16, 256, 5)
    y, _ = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    y_neg, _ = oracle.linear_f64(t.x_bits, t.w_packed ^ np.uint8(0x88), t.w_scale,
                                 t.global_scale)
    assert np.array_equal(y_neg, -y)


def test_nibble_order_single_nonzero():
    K, N = 32, 1
    x = np.zeros((1, K), np.uint16)
    x[0, 0] = 0x3F80          # 1.0 at k = 0
    x[0, 1] = 0x4000          # 2.0 at k = 1
    ws = np.full((N, K // 16), 0x38, np.uint8)
    lo = np.zeros((N, K // 2), np.uint8)
    lo[0, 0] = 0x07           # code 7 (6.0) in the low nibble -> k = 0
    hi = np.zeros((N, K // 2), np.uint8)
    hi[0, 0] = 0x70           # code 7 in the high nibble -> k = 1
    y_lo, _ = oracle.linear_f64(x, lo, ws, 1.0)
    y_hi, _ = oracle.linear_f64(x, hi, ws, 1.0)
    assert y_lo[0, 0] == 6.0 and y_hi[0, 0] == 12.0


def test_block_scale_index_is_k_over_16():
    # scale j must apply to k in [16j, 16j+16) only
    K, N = 64, 1
    x = np.full((1, K), 0x3F80, np.uint16)
    wp = np.full((N, K // 2), 0x22, np.uint8)     # code 2 = 1.0 everywhere
    for j in range(K // 16):
        ws = np.full((N, K // 16), 0x38, np.uint8)
        ws[0, j] = 0x40                          # block j doubled
        y, _ = oracle.linear_f64(x, wp, ws, 1.0)
        assert y[0, 0] == 64.0 + 16.0


def test_points_agree_with_full():
    t = make_linear(5, 40, 512, 9)
    y, a = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    rng = np.random.default_rng(0)
    mi = rng.integers(0, 5, 30)
    ni = rng.integers(0, 40, 30)
    yp, ap = oracle.linear_points_f64(t.x_bits, t.w_packed, t.w_scale,
                                      t.global_scale, mi, ni)
    assert np.array_equal(yp, y[mi, ni]) and np.array_equal(ap, a[mi, ni])


def test_threads_do_not_change_results():
    t = make_linear(3, 37, 256, 4)
    y1, a1 = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale, 1)
    y8, a8 = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale, 8)
    assert np.array_equal(y1, y8) and np.array_equal(a1, a8)


def test_empty_shapes():
    x = np.zeros((0, 32), np.uint16)
    y, a = oracle.linear_f64(x, np.zeros((4, 16), np.uint8),
                             np.zeros((4, 2), np.uint8), 1.0)
    assert y.shape == (0, 4)


def test_swiglu_closed_forms():
    assert oracle.swiglu(0.0, 5.0) == 0.0
    assert oracle.swiglu(3.0, 0.0) == 0.0
    # silu(g) = g * sigmoid(g); sigmoid(0) = 1/2 gives silu'(0) = 1/2: check
    # silu(1) = 1/(1+e^-1) exactly as printed in textbooks
    assert oracle.swiglu(1.0, 1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)),
                                                    rel=1e-15)
    # large positive gate: silu(g) -> g; large negative: -> 0
    assert oracle.swiglu(50.0, 2.0) == pytest.approx(100.0, rel=1e-15)
    assert abs(oracle.swiglu(-50.0, 2.0)) < 1e-19
    # odd-part identity: silu(g) - silu(-g) = g
    for g in (0.3, 1.7, -2.5):
        assert oracle.swiglu(g, 1) - oracle.swiglu(-g, 1) == pytest.approx(g, rel=1e-14)


def test_swiglu_rows_layout():
    # gate columns first, up columns second
    y = np.array([[1.0, -2.0, 3.0, 4.0]])
    out = oracle.swiglu_f64(y)
    s = lambda g: g / (1 + math.exp(-g))
    assert out[0, 0] == pytest.approx(s(1.0) * 3.0, rel=1e-15)
    assert out[0, 1] == pytest.approx(s(-2.0) * 4.0, rel=1e-15)


def test_bf16_chain_is_fp64_to_fp32_to_bf16():
    # 1 + 2^-8 + 2^-40 rounds to 1 + 2^-8 in fp32 (an exact bf16 tie), which
    # then rounds to even (1.0); rounding fp64 straight to bf16 would give
    # 1 + 2^-7.  The reading is the literal chain through fp32.
    v = 1.0 + 2.0**-8 + 2.0**-40
    assert oracle.to_bf16_bits(np.array([v]))[0] == 0x3F80
