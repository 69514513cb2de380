"""The bounded pipeline waits, made to run out on purpose through the
library's test hook (NVFP4_FLAG_TEST_STALL): the warp-MMA few-row kernel,
without a k split, never loads its last stage, so every wait for that stage
gives up after its 1 ms limit.  The kernel must wind down by itself -- no
fault, no hang -- report the time-out in the device error word, and leave the
context usable: the next ordinary call is correct and leaves the word clear.

The hook is accepted only where a stalled CTA holds nothing shared: no
thread-block cluster (split 1) and no TMEM (the warp-MMA kernel)."""
import numpy as np
import pytest
import torch

import oracle
from _parity import check_bf16, check_f32
from nvfp4_block_scaled_linear_gb300 import _lib
from nvfp4_block_scaled_linear_gb300 import build as cuda_build
from nvfp4_block_scaled_linear_gb300.inputs import make_linear

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SMALLM1 = _lib.FLAG_FORCE_SMALLM | _lib.FLAG_SPLIT(1)


@pytest.fixture(scope="module", autouse=True)
def built():
    cuda_build.build()
    _lib.load_library()
    _lib.device_error(clear=True)
    yield
    _lib.device_error(clear=True)


def _dev(t):
    x = torch.from_numpy(t.x_bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    return x, torch.from_numpy(t.w_packed).to(DEV), torch.from_numpy(t.w_scale).to(DEV)


# M = 1 (f16, one activation converter), M = 7 (f16, two converters),
# M = 12 (bf16, no converter); K = 256 is a single stage, K = 1024 four.
@pytest.mark.parametrize("M,K", [(1, 1024), (7, 1024), (12, 1024), (1, 256)])
def test_stalled_stage_times_out_and_is_reported(M, K):
    t = make_linear(M, 256, K, seed=2500 + M + K)
    x, wp, ws = _dev(t)
    assert _lib.device_error(clear=True) == 0
    _lib.linear_ex(x, wp, ws, float(t.global_scale), SMALLM1 | _lib.FLAG_TEST_STALL)
    torch.cuda.synchronize()                       # the kernel completed
    assert _lib.device_error(clear=True) & 1, "the stalled waits were not reported"
    assert _lib.device_error(clear=False) == 0, "the word was not cleared"
    # the context is still usable: an ordinary call right after is correct
    y32 = _lib.linear_ex(x, wp, ws, float(t.global_scale), SMALLM1 | _lib.FLAG_F32_OUT)
    ybf = _lib.linear_ex(x, wp, ws, float(t.global_scale), SMALLM1)
    torch.cuda.synchronize()
    y64, a = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    check_f32(y32.cpu().numpy(), y64, a, "after the stall, M=%d" % M)
    check_bf16(ybf.cpu().view(torch.int16).numpy().view(np.uint16), y64, a,
               oracle.to_bf16_bits(y64), "after the stall, M=%d" % M)
    assert _lib.device_error(clear=False) == 0


@pytest.mark.parametrize("flags", [
    _lib.FLAG_TEST_STALL,                                              # kernel not forced
    _lib.FLAG_FORCE_SMALLM | _lib.FLAG_TEST_STALL,                     # split not pinned to 1
    _lib.FLAG_FORCE_SMALLM | _lib.FLAG_SPLIT(2) | _lib.FLAG_TEST_STALL,
    _lib.FLAG_FORCE_GEMV | _lib.FLAG_BF16_MMA | _lib.FLAG_SPLIT(1) | _lib.FLAG_TEST_STALL,
    _lib.FLAG_FORCE_TCGEMM | _lib.FLAG_TEST_STALL])
def test_stall_hook_is_refused_where_a_cta_holds_shared_state(flags):
    t = make_linear(4, 256, 512, seed=2600)
    x, wp, ws = _dev(t)
    with pytest.raises(_lib.Nvfp4Error) as e:
        _lib.linear_ex(x, wp, ws, float(t.global_scale), flags)
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert _lib.device_error(clear=False) == 0
