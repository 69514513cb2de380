"""CPU oracle for the NVFP4 W4A16 block-scaled linear layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product path (``nvfp4_block_scaled_linear_gb300``) never imports it, and the
two share no code: this package wraps ``nvfp4_oracle.c``, a plain fp64 C
implementation that decodes every weight from its bits at the point of use.

Definition followed (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", section 1
"Model dependencies", checkpoint condition 2, the nvfp4-pack-quantized schema;
and the section 1 table: NVFP4 W4A16):

    w[n,k] = e2m1(code[n,k]) * e4m3(scale[n,k//16]) / global_scale
    y[m,n] = sum_k x[m,k] * w[n,k]

Every function below has pins in ``tests/test_oracle_*.py`` that do not go
through this package's own arithmetic (printed values, closed forms, library
decoders, brute force in exact rationals).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_e2m1.restype = ctypes.c_double
    lib.oracle_e2m1.argtypes = [ctypes.c_uint]
    lib.oracle_e4m3.restype = ctypes.c_double
    lib.oracle_e4m3.argtypes = [ctypes.c_uint]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_linear_f64.restype = ctypes.c_int
    lib.oracle_linear_f64.argtypes = [P, P, P, ctypes.c_float, i64, i64, i64,
                                      P, P, ctypes.c_int]
    lib.oracle_linear_points_f64.restype = ctypes.c_int
    lib.oracle_linear_points_f64.argtypes = [P, P, P, ctypes.c_float, i64, i64,
                                             i64, P, P, i64, P, P]
    lib.oracle_swiglu.restype = ctypes.c_double
    lib.oracle_swiglu.argtypes = [ctypes.c_double, ctypes.c_double]
    lib.oracle_f64_to_bf16_array.restype = None
    lib.oracle_f64_to_bf16_array.argtypes = [P, P, i64]
    lib.oracle_swiglu_rows.restype = ctypes.c_int
    lib.oracle_swiglu_rows.argtypes = [P, i64, i64, P]
    lib.oracle_decode_tables.restype = None
    lib.oracle_decode_tables.argtypes = [P, P]
    lib.oracle_e4m3_round.restype = ctypes.c_uint
    lib.oracle_e4m3_round.argtypes = [ctypes.c_float]
    lib.oracle_e2m1_round.restype = ctypes.c_uint
    lib.oracle_e2m1_round.argtypes = [ctypes.c_float]
    lib.oracle_quantize.restype = ctypes.c_int
    lib.oracle_quantize.argtypes = [P, i64, i64, P, P, P]
    lib.oracle_fp8_to_bf16.restype = ctypes.c_int
    lib.oracle_fp8_to_bf16.argtypes = [P, P, i64, i64, i64, P]
    _lib = lib
    return lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def e2m1(code: int) -> float:
    """Value of a 4-bit e2m1 code (sign, 2 exponent bits, 1 mantissa bit)."""
    return _load().oracle_e2m1(int(code))


def e4m3(bits: int) -> float:
    """Value of an 8-bit e4m3 (E4M3FN) pattern; NaN for S.1111.111."""
    return _load().oracle_e4m3(int(bits))


def decode_tables():
    """(e2m1 values for codes 0..15, e4m3 values for bytes 0..255) as fp64."""
    a = np.zeros(16, np.float64)
    b = np.zeros(256, np.float64)
    _load().oracle_decode_tables(_ptr(a), _ptr(b))
    return a, b


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits))


def f32_to_bf16(value: float) -> int:
    """bf16 bits of a binary32 value, round to nearest even."""
    return int(_load().oracle_f32_to_bf16_rne(float(value)))


def _check(x_bits, w_packed, w_scale, M=None):
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w_packed = np.ascontiguousarray(w_packed, dtype=np.uint8)
    w_scale = np.ascontiguousarray(w_scale, dtype=np.uint8)
    if x_bits.ndim != 2 or w_packed.ndim != 2 or w_scale.ndim != 2:
        raise ValueError("x, w_packed and w_scale must be 2-D")
    M, K = x_bits.shape
    N = w_packed.shape[0]
    if w_packed.shape != (N, K // 2) or w_scale.shape != (N, K // 16) or K % 16:
        raise ValueError("shape mismatch: x %s, w_packed %s, w_scale %s"
                         % (x_bits.shape, w_packed.shape, w_scale.shape))
    return x_bits, w_packed, w_scale, M, N, K


def linear_f64(x_bits, w_packed, w_scale, global_scale, threads=None):
    """fp64 y[M,N] and A[M,N] = sum_k |x w| for bf16 bits x[M,K]."""
    x_bits, w_packed, w_scale, M, N, K = _check(x_bits, w_packed, w_scale)
    y = np.zeros((M, N), np.float64)
    a = np.zeros((M, N), np.float64)
    rc = _load().oracle_linear_f64(_ptr(x_bits), _ptr(w_packed), _ptr(w_scale),
                                   float(np.float32(global_scale)), M, N, K,
                                   _ptr(y), _ptr(a),
                                   threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_linear_f64 rejected its arguments")
    return y, a


def linear_points_f64(x_bits, w_packed, w_scale, global_scale, m_idx, n_idx):
    """fp64 y and A at the listed (m, n) points only."""
    x_bits, w_packed, w_scale, M, N, K = _check(x_bits, w_packed, w_scale)
    m_idx = np.ascontiguousarray(m_idx, dtype=np.int64)
    n_idx = np.ascontiguousarray(n_idx, dtype=np.int64)
    if m_idx.shape != n_idx.shape:
        raise ValueError("m_idx and n_idx differ in shape")
    y = np.zeros(m_idx.shape, np.float64)
    a = np.zeros(m_idx.shape, np.float64)
    rc = _load().oracle_linear_points_f64(
        _ptr(x_bits), _ptr(w_packed), _ptr(w_scale),
        float(np.float32(global_scale)), M, N, K, _ptr(m_idx), _ptr(n_idx),
        m_idx.size, _ptr(y), _ptr(a))
    if rc != 0:
        raise ValueError("oracle_linear_points_f64 rejected its arguments")
    return y, a


def to_bf16_bits(y64):
    """bf16 bits of RNE(fp32(y64)): the literal fp64 -> fp32 -> bf16 chain."""
    y64 = np.ascontiguousarray(y64, dtype=np.float64)
    out = np.zeros(y64.shape, np.uint16)
    _load().oracle_f64_to_bf16_array(_ptr(y64), _ptr(out), y64.size)
    return out


def swiglu_f64(y64):
    """silu(gate) * up from fp64 accumulators laid out [M, gate | up]."""
    y64 = np.ascontiguousarray(y64, dtype=np.float64)
    M, N = y64.shape
    out = np.zeros((M, N // 2), np.float64)
    if _load().oracle_swiglu_rows(_ptr(y64), M, N, _ptr(out)) != 0:
        raise ValueError("swiglu needs an even number of columns")
    return out


def swiglu(gate: float, up: float) -> float:
    return _load().oracle_swiglu(float(gate), float(up))


def e4m3_round(v):
    """Nearest e4m3 code (bits) to a non-negative fp32 value (ties to even,
    saturating at 448)."""
    return int(_load().oracle_e4m3_round(float(v)))


def e2m1_round(t):
    """Nearest e2m1 code (sign | magnitude code) to an fp32 value (ties to
    the even code, saturating at 6)."""
    return int(_load().oracle_e2m1_round(float(t)))


def quantize(w_bits):
    """bf16 [N, K] (bits) -> (w_packed [N, K/2] u8, w_scale [N, K/16] u8,
    global_scale fp32), per the quantiser reading in nvfp4_oracle.c."""
    w_bits = np.ascontiguousarray(w_bits, np.uint16)
    N, K = w_bits.shape
    wp = np.zeros((N, K // 2), np.uint8)
    ws = np.zeros((N, K // 16), np.uint8)
    gs = np.zeros(1, np.float32)
    if _load().oracle_quantize(_ptr(w_bits), N, K, _ptr(wp), _ptr(ws), _ptr(gs)) != 0:
        raise ValueError("bad shape for the quantiser: %s" % (w_bits.shape,))
    return wp, ws, np.float32(gs[0])


def fp8_to_bf16(w8, scale_inv, block=128):
    """Block-scaled FP8 e4m3 [N, K] (bits) with fp32 scale_inv [ceil(N/B),
    ceil(K/B)] -> bf16 bits [N, K]: RNE_bf16(fp32(e4m3 * scale_inv)), per
    nvfp4_oracle.c."""
    w8 = np.ascontiguousarray(w8, np.uint8)
    N, K = w8.shape
    sinv = np.ascontiguousarray(scale_inv, np.float32)
    if sinv.shape != (-(-N // block), -(-K // block)):
        raise ValueError("scale_inv must be [ceil(N/%d), ceil(K/%d)]" % (block, block))
    out = np.zeros((N, K), np.uint16)
    if _load().oracle_fp8_to_bf16(_ptr(w8), _ptr(sinv), block, N, K, _ptr(out)) != 0:
        raise ValueError("bad shape")
    return out


def quantize_fp8(w8, scale_inv, block=128):
    """FP8 -> BF16 -> NVFP4: fp8_to_bf16, then quantize."""
    return quantize(fp8_to_bf16(w8, scale_inv, block))

