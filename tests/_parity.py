"""Comparison helpers for the GPU-vs-oracle parity tests (test infrastructure).

Tolerances (the accuracy contract of the layer):
  * fp32 results:  |y_gpu - y64| <= 1e-4 * A + 1e-6, where y64 is the oracle's
    fp64 result and A = sum_k |x w| (the oracle's companion output).
  * bf16 results:  within 1 bf16 ulp of RNE_bf16(fp32(y64)); only near zero,
    where the fp32 bound above exceeds one bf16 ulp of that rounded value, an
    output may pass instead by lying within the fp32 bound plus half a bf16
    ulp (the final rounding).  +0 and -0 are equal.  The count of outputs
    that pass only that way (the strict-fail count) is returned.
  * SwiGLU (out = silu(g) * u): the accumulator errors propagate through
    d out = silu'(g) u dg + silu(g) du with |silu'| <= 1.1, plus a relative
    1e-5 for the fp32 exp/divide/multiply of the epilogue.
"""
import numpy as np


def tol_f32(a):
    return 1e-4 * np.asarray(a, np.float64) + 1e-6


def bf16_bits_to_f64(bits):
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _ordered(bits):
    """Map bf16 bit patterns to integers ordered like the values (+0 == -0)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (binary32 exponent, 7 fraction bits)."""
    v = np.abs(np.asarray(v, np.float64))
    v = np.maximum(v, np.float64(2.0) ** -126)
    return np.float64(2.0) ** (np.floor(np.log2(v)) - 7)


def check_f32(y_gpu, y64, a, what=""):
    y_gpu = np.asarray(y_gpu, np.float64)
    err = np.abs(y_gpu - y64)
    tol = tol_f32(a)
    bad = ~(err <= tol)
    assert not bad.any(), "%s: %d/%d fp32 outputs outside 1e-4*A+1e-6; worst excess %g at %s" % (
        what, bad.sum(), bad.size, float(np.max(err - tol)), np.argwhere(bad)[:3].tolist())
    return float(np.max(err / tol)) if err.size else 0.0


def near_zero(ref_bits, a):
    """Outputs whose fp32 error bound 1e-4*A+1e-6 exceeds one bf16 ulp of the
    oracle's rounded value: there the fp32 accumulation the bound allows can
    move the result by more than one bf16 ulp (cancellation, |y| << A)."""
    return tol_f32(a) > bf16_ulp(bf16_bits_to_f64(ref_bits))


def check_bf16(bits_gpu, y64, a, ref_bits, what=""):
    """Returns (strict_fail_count, combined_fail_count); asserts combined == 0.

    Strict: within 1 bf16 ulp of the oracle's RNE_bf16(fp32(y64)).  Only where
    the output is near zero in the sense of near_zero() may an output outside
    1 ulp pass instead by lying within the fp32 bound plus half a bf16 ulp (the
    final rounding); everywhere else the 1-ulp rule alone applies.  NaN must
    match NaN."""
    bits_gpu = np.asarray(bits_gpu, np.uint16)
    ulps = np.abs(_ordered(bits_gpu) - _ordered(ref_bits))
    strict_ok = ulps <= 1
    val = bf16_bits_to_f64(bits_gpu)
    with np.errstate(invalid="ignore"):
        loose_ok = near_zero(ref_bits, a) & (np.abs(val - y64) <= tol_f32(a) + 0.5 * bf16_ulp(val))
    ok = strict_ok | loose_ok
    nan_ref = np.isnan(y64)
    ok = np.where(nan_ref, np.isnan(val), ok)
    strict_fail = int((~strict_ok & ~nan_ref).sum())
    fail = int((~ok).sum())
    assert fail == 0, "%s: %d/%d bf16 outputs outside 1 ulp (and, near zero, outside the fp32 " \
        "tolerance); first at %s (gpu %s, oracle %s)" % (
            what, fail, ok.size, np.argwhere(~ok)[:3].tolist(), val[~ok][:3], y64[~ok][:3])
    return strict_fail, fail


def record(what, **counts):
    """Append one JSON line of parity counts to $NVFP4_PARITY_LOG, if set."""
    import json
    import os
    path = os.environ.get("NVFP4_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(what=what, **counts)) + "\n")


def swiglu_tol(y64_gate, y64_up, a_gate, a_up, out64):
    g, u = y64_gate, y64_up
    silu = g / (1.0 + np.exp(-g))
    return (1.1 * tol_f32(a_gate) * np.abs(u) + np.abs(silu) * tol_f32(a_up)
            + 1e-5 * np.abs(out64) + 1e-30)


def check_swiglu_f32(y_gpu, y64, a, out64, what=""):
    H = y64.shape[1] // 2
    tol = swiglu_tol(y64[:, :H], y64[:, H:], a[:, :H], a[:, H:], out64)
    err = np.abs(np.asarray(y_gpu, np.float64) - out64)
    bad = ~(err <= tol)
    assert not bad.any(), "%s: %d/%d SwiGLU outputs outside tolerance; first at %s" % (
        what, bad.sum(), bad.size, np.argwhere(bad)[:3].tolist())


def check_swiglu_bf16(bits_gpu, y64, a, out64, ref_bits, what=""):
    """As check_bf16 with the SwiGLU bound: the looser rule only where that
    bound exceeds one bf16 ulp of the rounded oracle value.  Returns the
    strict-fail count among outputs in fp32's normal range (|out| >= 2^-126;
    below it fp32 itself holds fewer significant bits than bf16, and silu of
    a very negative gate lands there)."""
    H = y64.shape[1] // 2
    tol = swiglu_tol(y64[:, :H], y64[:, H:], a[:, :H], a[:, H:], out64)
    bits_gpu = np.asarray(bits_gpu, np.uint16)
    ulps = np.abs(_ordered(bits_gpu) - _ordered(ref_bits))
    val = bf16_bits_to_f64(bits_gpu)
    near = tol > bf16_ulp(bf16_bits_to_f64(ref_bits))
    ok = (ulps <= 1) | (near & (np.abs(val - out64) <= tol + 0.5 * bf16_ulp(val)))
    assert ok.all(), "%s: %d/%d SwiGLU bf16 outputs outside tolerance; first at %s" % (
        what, (~ok).sum(), ok.size, np.argwhere(~ok)[:3].tolist())
    return int(((ulps > 1) & (np.abs(out64) >= 2.0 ** -126)).sum())
