"""nvfp4_linear_host_noalloc, the entry point for callers that cannot
allocate device memory (a plug-in inside an application that owns every
device allocation, a loop that may not take an allocation's implicit
device synchronisation, a process whose device memory is fully reserved).
It runs the layer on host activations into a host result, staging both
through a fixed scratch array that the library holds on the device, so the
caller passes no device buffer but the weights it already holds.

The test calls it through the C ABI and compares its output with that of the
existing entry point, nvfp4_linear_host, given device buffers of the
caller's own: the same kernels run on the same inputs, so the results must
agree bit for bit (well inside the parity tolerance).  Each case makes two
calls in a row on one stream with different activations, so the second call
must not see anything the first left in the shared scratch.

This file is named to be collected last; it also passes alone in a fresh
process (the first call on the device sets up the scratch's address)."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_linear_gb300 import _lib
from nvfp4_block_scaled_linear_gb300 import build as cuda_build
from nvfp4_block_scaled_linear_gb300.inputs import make_linear

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return _lib.load_library()


def _host(t, pinned):
    x = torch.from_numpy(t.x_bits.view(np.int16)).view(torch.bfloat16).clone()
    return x.pin_memory() if pinned else x


def _bits(y):
    return y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32)


# M = 1 and M = 7: the warp-MMA kernel in f16 (7 with SwiGLU); M = 20: the
# same in bf16, fp32 out, through pageable buffers (the copy path); M = 40:
# the tensor-core kernel and the output staging kernel.
@pytest.mark.parametrize("M,N,K,flags,pinned", [
    (1, 1024, 2048, 0, True),
    (7, 1024, 2048, _lib.FLAG_SWIGLU, True),
    (20, 512, 1024, _lib.FLAG_F32_OUT, False),
    (40, 512, 1024, 0, True)])
def test_no_alloc_call_matches_the_host_buffer_entry_point(lib, M, N, K, flags, pinned):
    ta = make_linear(M, N, K, seed=4000 + M)
    tb = make_linear(M, N, K, seed=4100 + M)          # other activations, same shapes
    wp = torch.from_numpy(ta.w_packed).to(DEV)
    ws = torch.from_numpy(ta.w_scale).to(DEV)
    gs = float(ta.global_scale)
    n_out = N // 2 if flags & _lib.FLAG_SWIGLU else N
    dtype = torch.float32 if flags & _lib.FLAG_F32_OUT else torch.bfloat16
    stream = torch.cuda.Stream()

    # references: the existing entry point with device buffers of the caller's
    refs = []
    for t in (ta, tb):
        hy = torch.empty((M, n_out), dtype=dtype)
        _lib.linear_host(_host(t, pinned), torch.empty((M, K), dtype=torch.bfloat16, device=DEV),
                         wp, ws, gs, torch.empty((M, n_out), dtype=dtype, device=DEV), hy,
                         flags, stream=stream)
        stream.synchronize()
        refs.append(hy)

    # two calls in a row through the C ABI, no device buffer of ours
    outs = []
    for t in (ta, tb):
        hx = _host(t, pinned)
        hy = torch.full((M, n_out), float("nan"), dtype=dtype)
        hy = hy.pin_memory() if pinned else hy
        st = lib.nvfp4_linear_host_noalloc(hx.data_ptr(), wp.data_ptr(), ws.data_ptr(),
                                           ctypes.c_float(gs), hy.data_ptr(), M, N, K, flags,
                                           ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, _lib.status_string(st)
        outs.append((hx, hy))
    stream.synchronize()
    for (hx, hy), ref in zip(outs, refs):
        assert torch.equal(_bits(hy), _bits(ref))
    assert not torch.equal(_bits(outs[0][1]), _bits(outs[1][1]))
    assert _lib.device_error(clear=False) == 0


def test_no_alloc_rejects_what_does_not_fit(lib):
    # a prefill chunk: 84 MB of activations alone; rejected before any launch
    hx = torch.zeros(16, dtype=torch.bfloat16)
    hy = torch.zeros(16, dtype=torch.bfloat16)
    wp = torch.zeros((128, 128), dtype=torch.uint8, device=DEV)
    ws = torch.zeros((128, 16), dtype=torch.uint8, device=DEV)
    st = lib.nvfp4_linear_host_noalloc(hx.data_ptr(), wp.data_ptr(), ws.data_ptr(),
                                       ctypes.c_float(1.0), hy.data_ptr(), 8192, 34816, 5120, 0,
                                       None)
    assert st == _lib.ERR_TOO_LARGE
    assert "scratch" in _lib.status_string(st)
    # just past the limit: activations + result one byte-step beyond 8 MiB
    M, K = 16, 256
    n_over = (_lib.NOALLOC_SCRATCH_BYTES - M * K * 2) // (M * 2) + 128
    st = lib.nvfp4_linear_host_noalloc(hx.data_ptr(), wp.data_ptr(), ws.data_ptr(),
                                       ctypes.c_float(1.0), hy.data_ptr(), M, n_over, K, 0, None)
    assert st == _lib.ERR_TOO_LARGE
