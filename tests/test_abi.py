"""The C ABI on the host: the library builds, loads, exports every function
include/nvfp4_linear.h declares, and rejects bad arguments before touching a
device.  No call here reaches a kernel (none of them gets past validation)."""
import ctypes

import pytest
import torch

from nvfp4_block_scaled_linear_gb300 import _lib
from nvfp4_block_scaled_linear_gb300 import build as cuda_build


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return _lib.load_library()


def test_exports_every_declared_function(lib):
    names = _lib.header_functions()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), "missing export " + n


def test_header_constants_match_binding():
    text = open(_lib.HEADER).read()
    for name, value in (("NVFP4_FLAG_SWIGLU", _lib.FLAG_SWIGLU),
                        ("NVFP4_FLAG_F32_OUT", _lib.FLAG_F32_OUT),
                        ("NVFP4_FLAG_FORCE_SMALLM", _lib.FLAG_FORCE_SMALLM),
                        ("NVFP4_FLAG_FORCE_TCGEMM", _lib.FLAG_FORCE_TCGEMM),
                        ("NVFP4_KERNEL_SMALLM", _lib.KERNEL_SMALLM),
                        ("NVFP4_KERNEL_TCGEMM", _lib.KERNEL_TCGEMM),
                        ("NVFP4_KERNEL_GEMV", _lib.KERNEL_GEMV),
                        ("NVFP4_KERNEL_GEMV_BF16", _lib.KERNEL_GEMV_BF16)):
        assert "#define %s %du" % (name, value) in text or "#define %s %d " % (name, value) in text
    assert "#define NVFP4_FLAG_BF16_MMA (1u << 17)" in text and _lib.FLAG_BF16_MMA == 1 << 17
    assert "#define NVFP4_FLAG_FORCE_GEMV (1u << 18)" in text and _lib.FLAG_FORCE_GEMV == 1 << 18
    assert "#define NVFP4_FLAG_TEST_STALL (1u << 19)" in text and _lib.FLAG_TEST_STALL == 1 << 19
    assert "#define NVFP4_FLAG_SPLIT_SHIFT 8" in text and _lib.FLAG_SPLIT(3) == 3 << 8
    assert "#define NVFP4_FLAG_GROUPS_SHIFT 13" in text and _lib.FLAG_GROUPS(5) == 5 << 13


def test_version_and_status_strings(lib):
    assert _lib.abi_version() == 1
    for st in (0, -1, -2, -3, -4, -5, -6, 7):
        s = _lib.status_string(st)
        assert isinstance(s, str) and s


@pytest.mark.parametrize("M,N,K,flags,expect", [
    (1, 256, 512, 0, _lib.KERNEL_SMALLM),
    (8, 256, 512, 0, _lib.KERNEL_SMALLM),
    (9, 256, 512, 0, _lib.KERNEL_SMALLM),
    (16, 256, 512, 0, _lib.KERNEL_SMALLM),
    (9, 34816, 5120, 0, _lib.KERNEL_GEMV_BF16),
    (8, 34816, 5120, 0, _lib.KERNEL_SMALLM),
    (17, 256, 512, 0, _lib.KERNEL_SMALLM),
    (32, 34816, 5120, 0, _lib.KERNEL_GEMV_BF16),                 # large layer, M = 17..32
    (17, 5120, 17408, 0, _lib.KERNEL_GEMV_BF16),
    (24, 8192, 5120, 0, _lib.KERNEL_SMALLM),                     # N * K < 2^26
    (16, 5120, 17408, 0, _lib.KERNEL_SMALLM),                    # M <= 16: N * K < 2^27
    (32, 5120, 6144, 0, _lib.KERNEL_GEMV_BF16),                  # M >= 25: N * K >= 3 * 2^23
    (32, 4096, 4096, 0, _lib.KERNEL_SMALLM),
    (16, 34816, 5120, 0, _lib.KERNEL_GEMV_BF16),
    (32, 34816, 5120, _lib.FLAG_BF16_MMA, _lib.KERNEL_GEMV_BF16),
    (16, 34816, 5120, _lib.FLAG_BF16_MMA, _lib.KERNEL_GEMV_BF16),
    (8, 34816, 5120, _lib.FLAG_BF16_MMA, _lib.KERNEL_SMALLM),
    (7, 256, 512, _lib.FLAG_FORCE_GEMV | _lib.FLAG_BF16_MMA, _lib.KERNEL_GEMV_BF16),
    (40, 256, 512, _lib.FLAG_FORCE_GEMV | _lib.FLAG_BF16_MMA, _lib.KERNEL_NONE),
    (1, 256, 512, _lib.FLAG_FORCE_SMALLM, _lib.KERNEL_SMALLM),
    (7, 256, 512, _lib.FLAG_BF16_MMA, _lib.KERNEL_SMALLM),
    (7, 256, 512, _lib.FLAG_FORCE_GEMV, _lib.KERNEL_GEMV),
    (40, 256, 512, _lib.FLAG_FORCE_GEMV, _lib.KERNEL_NONE),      # gemv needs M <= 32
    (7, 256, 512, _lib.FLAG_BF16_MMA | _lib.FLAG_FORCE_TCGEMM, _lib.KERNEL_NONE),
    (7, 256, 512, _lib.FLAG_FORCE_GEMV | _lib.FLAG_FORCE_TCGEMM, _lib.KERNEL_NONE),
    (7, 256, 512, _lib.FLAG_FORCE_GEMV | _lib.FLAG_FORCE_SMALLM, _lib.KERNEL_NONE),
    (33, 34816, 5120, 0, _lib.KERNEL_TCGEMM),
    (8192, 34816, 5120, _lib.FLAG_SWIGLU, _lib.KERNEL_TCGEMM),
    (7, 5120, 17408, _lib.FLAG_FORCE_TCGEMM, _lib.KERNEL_TCGEMM),
    (64, 256, 512, _lib.FLAG_FORCE_SMALLM, _lib.KERNEL_NONE),   # smallm needs M <= 32
    (1, 256, 500, 0, _lib.KERNEL_NONE),                          # K % 256
    (1, 200, 512, 0, _lib.KERNEL_NONE),                          # N % 128
    (0, 256, 512, 0, _lib.KERNEL_NONE),                          # empty: nothing launched
    (-1, 256, 512, 0, _lib.KERNEL_NONE),
    (1, 256, 512, 64, _lib.KERNEL_NONE),                         # unknown flag
    (1, 256, 512, _lib.FLAG_FORCE_SMALLM | _lib.FLAG_FORCE_TCGEMM, _lib.KERNEL_NONE),
    # the wait-limit test hook: warp-MMA kernel, split pinned to 1, only
    (7, 256, 512, _lib.FLAG_FORCE_SMALLM | _lib.FLAG_SPLIT(1) | _lib.FLAG_TEST_STALL,
     _lib.KERNEL_SMALLM),
    (7, 256, 512, _lib.FLAG_TEST_STALL, _lib.KERNEL_NONE),
    (7, 256, 512, _lib.FLAG_FORCE_SMALLM | _lib.FLAG_TEST_STALL, _lib.KERNEL_NONE),
    (7, 256, 512, _lib.FLAG_FORCE_SMALLM | _lib.FLAG_SPLIT(2) | _lib.FLAG_TEST_STALL,
     _lib.KERNEL_NONE),
    (7, 256, 512, _lib.FLAG_FORCE_GEMV | _lib.FLAG_SPLIT(1) | _lib.FLAG_TEST_STALL,
     _lib.KERNEL_NONE),
])
def test_kernel_choice(lib, M, N, K, flags, expect):
    assert _lib.kernel_for(M, N, K, flags) == expect


def _call(lib, x, wp, ws, y, M, N, K):
    return lib.nvfp4_linear(x, wp, ws, ctypes.c_float(1.0), y, M, N, K, None)


def test_rejects_before_any_device_work(lib):
    A = 0x10000           # fake, 16-byte aligned, never dereferenced
    assert _call(lib, None, A, A, A, 1, 256, 512) == -1
    assert _call(lib, A, None, A, A, 1, 256, 512) == -1
    assert _call(lib, A, A, None, A, 1, 256, 512) == -1
    assert _call(lib, A, A, A, None, 1, 256, 512) == -1
    assert _call(lib, A, A, A, A, -1, 256, 512) == -1
    assert _call(lib, A, A, A, A, 1, 0, 512) == -1
    assert _call(lib, A, A, A, A, 1, 256, 0) == -1
    assert _call(lib, A + 2, A, A, A, 1, 256, 512) == -2
    assert _call(lib, A, A + 8, A, A, 1, 256, 512) == -2
    assert _call(lib, A, A, A, A + 4, 1, 256, 512) == -2
    assert _call(lib, A, A, A, A, 1, 256, 384) == -3
    assert _call(lib, A, A, A, A, 1, 192, 512) == -3
    assert lib.nvfp4_linear_ex(A, A, A, ctypes.c_float(1.0), A, 1, 256, 512, 1 << 7, None) == -1
    assert lib.nvfp4_linear_ex(A, A, A, ctypes.c_float(1.0), A, 40, 256, 512,
                               _lib.FLAG_FORCE_SMALLM, None) == -1
    # M == 0 is a valid empty call: nothing to do, nothing launched; x and y
    # may be NULL (an empty tensor's data pointer)
    assert _call(lib, A, A, A, A, 0, 256, 512) == 0
    assert _call(lib, None, A, A, None, 0, 256, 512) == 0
    assert _call(lib, None, None, A, None, 0, 256, 512) == -1
    assert lib.nvfp4_linear_swiglu_gs(A, A, A, ctypes.c_float(1.0), ctypes.c_float(2.0), None,
                                      1, 256, 512, 0, None) == -1
    assert lib.nvfp4_linear_swiglu_gs(A, A, A, ctypes.c_float(1.0), ctypes.c_float(2.0), A,
                                      1, 256, 384, 0, None) == -3
    gs2 = (ctypes.c_float * 2)(1.0, 2.0)
    rows_ok = (ctypes.c_int64 * 2)(128, 128)
    rows_bad = (ctypes.c_int64 * 2)(128, 64)
    rows_zero = (ctypes.c_int64 * 2)(256, 0)
    seg = lib.nvfp4_linear_segmented
    assert seg(A, A, A, ctypes.cast(gs2, ctypes.c_void_p), ctypes.cast(rows_bad, ctypes.c_void_p),
               2, A, 1, 256, 512, 0, None) == -1                       # rows sum != N
    assert seg(A, A, A, ctypes.cast(gs2, ctypes.c_void_p), ctypes.cast(rows_zero, ctypes.c_void_p),
               2, A, 1, 256, 512, 0, None) == -1                       # empty segment
    assert seg(A, A, A, None, ctypes.cast(rows_ok, ctypes.c_void_p), 2, A, 1, 256, 512, 0,
               None) == -1
    assert seg(A, A, A, ctypes.cast(gs2, ctypes.c_void_p), ctypes.cast(rows_ok, ctypes.c_void_p),
               9, A, 1, 256, 512, 0, None) == -1                       # > 8 segments
    assert seg(A, A, A, ctypes.cast(gs2, ctypes.c_void_p), ctypes.cast(rows_ok, ctypes.c_void_p),
               2, A, 1, 256, 512, _lib.FLAG_SWIGLU, None) == -1
    q = lib.nvfp4_quantize
    F = 0x20000            # fake 16-byte aligned float address, never dereferenced
    assert q(None, 4, 64, A, A, F, None) == -1
    assert q(A, 4, 64, A, A, None, None) == -1
    assert q(A, 0, 64, A, A, F, None) == -1
    assert q(A, 4, 40, A, A, F, None) == -3                  # K % 16
    assert q(A + 8, 4, 64, A, A, F, None) == -2               # w not 16-byte aligned
    assert q(A, 4, 64, A + 4, A, F, None) == -2               # codes not 8-byte aligned
    q8 = lib.nvfp4_quantize_fp8
    assert q8(None, F, 128, 4, 64, A, A, F, None) == -1
    assert q8(A, None, 128, 4, 64, A, A, F, None) == -1
    assert q8(A, F, 0, 4, 64, A, A, F, None) == -1
    assert q8(A, F, 128, 4, 40, A, A, F, None) == -3           # K % 16
    assert q8(A, F, 100, 4, 64, A, A, F, None) == -3           # block % 16
    assert q8(A + 8, F, 128, 4, 64, A, A, F, None) == -2       # codes not 16-byte aligned
    assert q8(A, F + 2, 128, 4, 64, A, A, F, None) == -2       # scale_inv misaligned
    h = lib.nvfp4_linear_host
    H = 0x30000            # fake host address, never dereferenced
    assert h(None, A, A, A, ctypes.c_float(1.0), A, H, 1, 256, 512, 0, None) == -1
    assert h(H, A, A, A, ctypes.c_float(1.0), A, None, 1, 256, 512, 0, None) == -1
    assert h(H, None, A, A, ctypes.c_float(1.0), A, H, 1, 256, 512, 0, None) == -1
    assert h(H, A, A, A, ctypes.c_float(1.0), A + 2, H, 1, 256, 512, 0, None) == -2
    assert h(H, A, A, A, ctypes.c_float(1.0), A, H, 1, 256, 384, 0, None) == -3
    assert h(None, None, A, A, ctypes.c_float(1.0), None, None, 0, 256, 512, 0, None) == 0
    na = lib.nvfp4_linear_host_noalloc
    assert na(None, A, A, ctypes.c_float(1.0), H, 1, 256, 512, 0, None) == -1
    assert na(H, A, A, ctypes.c_float(1.0), None, 1, 256, 512, 0, None) == -1
    assert na(H, A, A, ctypes.c_float(1.0), H, -1, 256, 512, 0, None) == -1
    assert na(None, A, A, ctypes.c_float(1.0), None, 0, 256, 512, 0, None) == 0
    assert na(H, A, A, ctypes.c_float(1.0), H, 8192, 34816, 5120, 0, None) == -6   # too large
    assert _lib.status_string(-6) != _lib.status_string(99)
    # tuning overrides out of range
    assert lib.nvfp4_linear_ex(A, A, A, ctypes.c_float(1.0), A, 1, 256, 512,
                               _lib.FLAG_SPLIT(17), None) == -1
    assert lib.nvfp4_linear_ex(A, A, A, ctypes.c_float(1.0), A, 1, 256, 512,
                               _lib.FLAG_GROUPS(9), None) == -1


def test_binding_refuses_cpu_tensors(lib):
    x = torch.zeros(1, 512, dtype=torch.bfloat16)
    wp = torch.zeros(256, 256, dtype=torch.uint8)
    ws = torch.zeros(256, 32, dtype=torch.uint8)
    with pytest.raises(ValueError):
        _lib.linear(x, wp, ws, 1.0)
