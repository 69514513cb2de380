"""The oracle's pins have teeth: plant a plausible mistake in a copy of the C
oracle, build the copy, and check that the pins reject it.

Mistakes are planted only in a temporary copy of oracle/nvfp4_oracle.c, on the
CPU; the real oracle is untouched.
"""
import ctypes
import json
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nvfp4_oracle.c")
GOLDEN = os.path.join(ROOT, "tests", "golden")

MUTANTS = {
    "nibble_order_swapped": ("unsigned code = (k % 2 == 0) ? (byte & 0x0fu) : (byte >> 4);",
                             "unsigned code = (k % 2 == 0) ? (byte >> 4) : (byte & 0x0fu);"),
    "e2m1_bias_off_by_one": ("mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);",
                             "mag = ldexp(1.0 + 0.5 * (double)m, (int)e);"),
    "e2m1_sign_dropped": ("    unsigned s = (code >> 3) & 1u;", "    unsigned s = 0u * code;"),
    "e4m3_bias_8": ("mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
                    "mag = ldexp(1.0 + (double)m / 8.0, (int)e - 8);"),
    "e4m3_subnormal_as_normal": ("mag = ldexp((double)m / 8.0, -6);",
                                 "mag = ldexp(1.0 + (double)m / 8.0, -6);"),
    "scale_block_index_dropped": ("double scale = oracle_e4m3(w_scale[n * (K / 16) + k / 16]);",
                                  "double scale = oracle_e4m3(w_scale[n * (K / 16)]);"),
    "global_scale_multiplied": ("return oracle_e2m1(code) * scale / global_scale;",
                                "return oracle_e2m1(code) * scale * global_scale;"),
    "abs_sum_signed": ("abs_sum += fabs(prod);", "abs_sum += prod;"),
    "rne_ties_away": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))",
                      "if (lower >= 0x8000u)"),
    "swiglu_no_sigmoid": ("return gate / (1.0 + exp(-gate)) * up;", "return gate * up;"),
    "quant_block_divisor_4": ("const float s_f = (amax_b * gs) / 6.0f;",
                              "const float s_f = (amax_b * gs) / 4.0f;"),
    "quant_global_scale_inverted": ("const float gs = amax > 0.0f ? 448.0f / amax : 1.0f;",
                                    "const float gs = amax > 0.0f ? amax / 448.0f : 1.0f;"),
    "quant_e2m1_ties_odd": ("if (d < best_d || (d == best_d && (c & 1u) == 0)) {",
                            "if (d < best_d || (d == best_d && (c & 1u) == 1)) {"),
    "quant_e4m3_ties_odd": ("if (d < best_d || (d == best_d && (b & 1u) == 0)) {",
                            "if (d < best_d || (d == best_d && (b & 1u) == 1)) {"),
    "quant_codes_use_unrounded_scale": ("const float s = (float)oracle_e4m3(sbyte);",
                                        "const float s = s_f;"),
    "fp8_scale_divides": ("const float p = v * scale_inv[(n / block) * kb + k / block];",
                          "const float p = v / scale_inv[(n / block) * kb + k / block];"),
    "fp8_row_blocks_ignored": ("const float p = v * scale_inv[(n / block) * kb + k / block];",
                               "const float p = v * scale_inv[k / block];"),
    "fp8_scale_dropped": ("const float p = v * scale_inv[(n / block) * kb + k / block];",
                          "const float p = v;"),
    "quant_nibbles_swapped": ("w_packed[n * (K / 2) + b * 8 + j / 2] = (uint8_t)(c[0] | (c[1] << 4));",
                              "w_packed[n * (K / 2) + b * 8 + j / 2] = (uint8_t)(c[1] | (c[0] << 4));"),
}


def _build(tmp_path, name, source):
    c = tmp_path / (name + ".c")
    c.write_text(source)
    so = tmp_path / (name + ".so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so),
                    str(c), "-lm", "-lpthread"], check=True)
    lib = ctypes.CDLL(str(so))
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.oracle_linear_f64.argtypes = [P, P, P, ctypes.c_float, i64, i64, i64, P, P,
                                      ctypes.c_int]
    lib.oracle_decode_tables.argtypes = [P, P]
    lib.oracle_f64_to_bf16_array.argtypes = [P, P, i64]
    lib.oracle_swiglu.restype = ctypes.c_double
    lib.oracle_swiglu.argtypes = [ctypes.c_double, ctypes.c_double]
    lib.oracle_quantize.restype = ctypes.c_int
    lib.oracle_quantize.argtypes = [P, i64, i64, P, P, P]
    lib.oracle_e2m1_round.restype = ctypes.c_uint
    lib.oracle_e2m1_round.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_round.restype = ctypes.c_uint
    lib.oracle_e4m3_round.argtypes = [ctypes.c_float]
    lib.oracle_fp8_to_bf16.restype = ctypes.c_int
    lib.oracle_fp8_to_bf16.argtypes = [P, P, i64, i64, i64, P]
    return lib


def fp8_torch_case(N=200, K=272, block=128, seed=5):
    """A ragged block-scaled FP8 tensor with distinct non-power-of-two
    scales per block, and its bf16 image by torch's own e4m3 decode, fp32
    multiply and bf16 rounding."""
    rng = np.random.default_rng(seed)
    w8 = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x3A                     # no NaN codes
    nb, kb = -(-N // block), -(-K // block)
    sinv = np.exp(rng.uniform(-6, 6, size=(nb, kb))).astype(np.float32)
    x = torch.from_numpy(w8).view(torch.float8_e4m3fn).to(torch.float32)
    s_full = torch.from_numpy(sinv).repeat_interleave(block, 0)[:N] \
        .repeat_interleave(block, 1)[:, :K]
    want = (x * s_full).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return w8, sinv, want


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _pins_pass(lib) -> bool:
    """A compact re-run of the pins in test_oracle_*.py against ``lib``."""
    e2m1 = np.zeros(16)
    e4m3 = np.zeros(256)
    lib.oracle_decode_tables(_p(e2m1), _p(e4m3))
    table = json.load(open(os.path.join(GOLDEN, "e2m1_table.json")))["code_to_value"]
    if any(e2m1[int(c)] != v for c, v in table.items()):
        return False
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()
    ok = ~np.isnan(ref)
    if not np.array_equal(e4m3[ok], ref[ok]):
        return False
    for case in json.load(open(os.path.join(GOLDEN, "hand_blocks.json")))["cases"]:
        x = np.ascontiguousarray(case["x_bits"], np.uint16)
        wp = np.ascontiguousarray(case["w_packed"], np.uint8)
        ws = np.ascontiguousarray(case["w_scale"], np.uint8)
        M, K = x.shape
        N = wp.shape[0]
        y = np.zeros((M, N))
        a = np.zeros((M, N))
        lib.oracle_linear_f64(_p(x), _p(wp), _p(ws), case["global_scale"], M, N, K,
                              _p(y), _p(a), 1)
        if not np.array_equal(y, np.array(case["y"])) or np.any(a < np.abs(y)):
            return False
        # every output here has A = sum |x w| computable by hand only for the
        # sign-uniform cases; the sign-mixed first case must give A > |y|
        if case["name"] == "all_codes_cancel" and not a[0, 0] == 36.0:
            return False
    ties = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8])
    out = np.zeros(2, np.uint16)
    lib.oracle_f64_to_bf16_array(_p(ties), _p(out), 2)
    if list(out) != [0x3F80, 0x3F82]:
        return False
    if abs(lib.oracle_swiglu(1.0, 1.0) - 1.0 / (1.0 + np.exp(-1.0))) > 1e-15:
        return False
    # quantiser: the e2m1 midpoint table, torch's e4m3 cast on ties, and the
    # hand-worked blocks
    for t, code in ((0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
                    (7.0, 7)):
        if lib.oracle_e2m1_round(t) != code:
            return False
    ev = np.float32([9.5, 10.5, 0.0546875, 1.0 + 1.0 / 16, 448.0])
    want = torch.from_numpy(ev).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if [lib.oracle_e4m3_round(float(v)) for v in ev] != list(want):
        return False
    w8, sinv, want = fp8_torch_case()
    got = np.zeros(w8.shape, np.uint16)
    lib.oracle_fp8_to_bf16(_p(w8), _p(sinv), 128, w8.shape[0], w8.shape[1], _p(got))
    if not np.array_equal(got, want):
        return False
    for case in json.load(open(os.path.join(GOLDEN, "quantize_blocks.json")))["cases"]:
        w = torch.tensor(case["w"], dtype=torch.float32).to(torch.bfloat16) \
            .view(torch.int16).numpy().view(np.uint16)
        w = np.ascontiguousarray(w)
        N, K = w.shape
        wp = np.zeros((N, K // 2), np.uint8)
        ws = np.zeros((N, K // 16), np.uint8)
        gs = np.zeros(1, np.float32)
        lib.oracle_quantize(_p(w), N, K, _p(wp), _p(ws), _p(gs))
        codes = np.stack([wp & 0xF, wp >> 4], -1).reshape(N, K)
        if (gs[0] != np.float32(case["global_scale"])
                or not np.array_equal(ws, np.asarray(case["scale"], np.uint8))
                or not np.array_equal(codes, np.asarray(case["codes"], np.uint8))):
            return False
    return True


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_control_unmutated_passes(tmp_path, source):
    assert _pins_pass(_build(tmp_path, "control", source))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, source, name):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, "mutation anchor not found: " + name
    assert not _pins_pass(_build(tmp_path, name, source.replace(old, new)))


def test_gcc_available():
    assert shutil.which("gcc")
