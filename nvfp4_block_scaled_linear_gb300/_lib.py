"""ctypes binding of libnvfp4_linear.so (include/nvfp4_linear.h).

Argument marshalling only: shape/dtype/device checks, output allocation with
torch, the current CUDA stream, and the call.  Every step of the layer runs
in the library's kernels; there is no CPU or PyTorch fallback, and a missing
library or GPU raises.
"""
import contextlib
import ctypes
import os
import re

import torch

from . import build as _build

# Mirrors of the header's constants.
OK = 0
FLAG_SWIGLU = 1
FLAG_F32_OUT = 2
FLAG_FORCE_SMALLM = 4
FLAG_FORCE_TCGEMM = 8
FLAG_BF16_MMA = 1 << 17
FLAG_FORCE_GEMV = 1 << 18
FLAG_TEST_STALL = 1 << 19       # test hook of the wait limit (see the header)


def FLAG_SPLIT(n):
    """Few-row kernel: split k over n CTAs of one cluster (1..16)."""
    return (int(n) & 0x1F) << 8


def FLAG_GROUPS(n):
    """Few-row kernel: CTAs of 16*n weight rows (1..8)."""
    return (int(n) & 0xF) << 13


ERR_TOO_LARGE = -6                # nvfp4_linear_host_noalloc: beyond its scratch
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

KERNEL_NONE, KERNEL_SMALLM, KERNEL_TCGEMM, KERNEL_GEMV, KERNEL_GEMV_BF16 = 0, 1, 2, 3, 4
KERNEL_NAMES = {KERNEL_SMALLM: "smallm", KERNEL_TCGEMM: "tcgemm", KERNEL_GEMV: "gemv_tc",
                KERNEL_GEMV_BF16: "gemv_bf16"}

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "nvfp4_linear.h")

_lib = None


class Nvfp4Error(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        msg = library().nvfp4_status_string(status).decode() if _lib else str(status)
        super().__init__("%s failed: %s (status %d)" % (what or "nvfp4", msg, status))


def header_functions():
    """Names of the functions declared in include/nvfp4_linear.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(nvfp4_\w+)\s*\(",
                                 text, re.M)))


def load_library(path=None):
    """Load the built library (never builds it; __graft_entry__.build() or
    ``python -m nvfp4_block_scaled_linear_gb300.build`` does)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError("libnvfp4_linear.so is not built (%s); run "
                           "python -m nvfp4_block_scaled_linear_gb300.build" % path)
    lib = ctypes.CDLL(path)
    P, i64, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint
    lib.nvfp4_abi_version.restype = ctypes.c_int
    lib.nvfp4_abi_version.argtypes = []
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_status_string.argtypes = [ctypes.c_int]
    for name in ("nvfp4_linear", "nvfp4_linear_f32", "nvfp4_linear_swiglu",
                 "nvfp4_linear_swiglu_f32"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P, P, P, ctypes.c_float, P, i64, i64, i64, P]
    lib.nvfp4_linear_ex.restype = ctypes.c_int
    lib.nvfp4_linear_ex.argtypes = [P, P, P, ctypes.c_float, P, i64, i64, i64, u32, P]
    lib.nvfp4_linear_host.restype = ctypes.c_int
    lib.nvfp4_linear_host.argtypes = [P, P, P, P, ctypes.c_float, P, P, i64, i64, i64, u32, P]
    lib.nvfp4_linear_host_noalloc.restype = ctypes.c_int
    lib.nvfp4_linear_host_noalloc.argtypes = [P, P, P, ctypes.c_float, P, i64, i64, i64, u32, P]
    lib.nvfp4_linear_swiglu_gs.restype = ctypes.c_int
    lib.nvfp4_linear_swiglu_gs.argtypes = [P, P, P, ctypes.c_float, ctypes.c_float, P, i64, i64,
                                           i64, u32, P]
    lib.nvfp4_linear_segmented.restype = ctypes.c_int
    lib.nvfp4_linear_segmented.argtypes = [P, P, P, P, P, ctypes.c_int, P, i64, i64, i64, u32, P]
    lib.nvfp4_quantize.restype = ctypes.c_int
    lib.nvfp4_quantize.argtypes = [P, i64, i64, P, P, P, P]
    lib.nvfp4_quantize_fp8.restype = ctypes.c_int
    lib.nvfp4_quantize_fp8.argtypes = [P, P, i64, i64, i64, P, P, P, P]
    lib.nvfp4_linear_kernel_for.restype = ctypes.c_int
    lib.nvfp4_linear_kernel_for.argtypes = [i64, i64, i64, u32]
    lib.nvfp4_device_status.restype = ctypes.c_int
    lib.nvfp4_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
    _lib = lib
    return lib


def library():
    return load_library()


def abi_version() -> int:
    return library().nvfp4_abi_version()


def status_string(status: int) -> str:
    return library().nvfp4_status_string(int(status)).decode()


def kernel_for(M, N, K, flags=0) -> int:
    return library().nvfp4_linear_kernel_for(int(M), int(N), int(K), int(flags))


def device_error(clear: bool = True) -> int:
    """The device error word (bit 0: a pipeline wait timed out); synchronises."""
    bits = ctypes.c_uint(0)
    st = library().nvfp4_device_status(ctypes.byref(bits), 1 if clear else 0)
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_device_status")
    return bits.value


def _as_u8(t, name):
    if t.dtype == torch.uint8:
        return t
    if t.dtype in (torch.int8, torch.float8_e4m3fn):
        return t.view(torch.uint8)
    raise TypeError("%s must be uint8 (or float8_e4m3fn for scales), got %s" % (name, t.dtype))


def _check(x, w_packed, w_scale):
    if not (x.is_cuda and w_packed.is_cuda and w_scale.is_cuda):
        raise ValueError("x, w_packed and w_scale must be CUDA tensors")
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16, got %s" % x.dtype)
    w_packed = _as_u8(w_packed, "w_packed")
    w_scale = _as_u8(w_scale, "w_scale")
    if x.dim() != 2 or w_packed.dim() != 2 or w_scale.dim() != 2:
        raise ValueError("x, w_packed and w_scale must be 2-D")
    M, K = x.shape
    N = w_packed.shape[0]
    if tuple(w_packed.shape) != (N, K // 2) or tuple(w_scale.shape) != (N, K // 16):
        raise ValueError("shapes disagree: x %s, w_packed %s, w_scale %s"
                         % (tuple(x.shape), tuple(w_packed.shape), tuple(w_scale.shape)))
    if not (x.is_contiguous() and w_packed.is_contiguous() and w_scale.is_contiguous()):
        raise ValueError("x, w_packed and w_scale must be contiguous")
    if len({x.device, w_packed.device, w_scale.device}) != 1:
        raise ValueError("inputs live on different devices")
    return w_packed, w_scale, M, N, K


def _on_device(device):
    """Make `device` current for the call (the library works on the current
    device); no switch, and no cost, when it already is."""
    if device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def linear_ex(x, w_packed, w_scale, global_scale, flags=0, out=None, stream=None):
    """Call nvfp4_linear_ex; allocate ``out`` if not given and return it."""
    w_packed, w_scale, M, N, K = _check(x, w_packed, w_scale)
    n_out = N // 2 if flags & FLAG_SWIGLU else N
    dtype = torch.float32 if flags & FLAG_F32_OUT else torch.bfloat16
    if out is None:
        out = torch.empty((M, n_out), dtype=dtype, device=x.device)
    elif (out.dtype != dtype or tuple(out.shape) != (M, n_out) or not out.is_contiguous()
          or out.device != x.device):
        raise ValueError("out must be a contiguous %s tensor of shape %s on %s"
                         % (dtype, (M, n_out), x.device))
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with _on_device(x.device):
        st = library().nvfp4_linear_ex(x.data_ptr(), w_packed.data_ptr(), w_scale.data_ptr(),
                                       float(global_scale), out.data_ptr(), M, N, K,
                                       int(flags), ctypes.c_void_p(stream.cuda_stream))
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_linear_ex")
    return out


def linear_host(x_host, x_dev, w_packed, w_scale, global_scale, y_dev, y_host, flags=0,
                stream=None):
    """Call nvfp4_linear_host: move the host activations ``x_host`` into the
    device buffer ``x_dev``, run the layer into ``y_dev`` and move it to the
    host tensor ``y_host``, all enqueued on ``stream``.  Page-locked,
    16-byte aligned host tensors take the zero-copy transfer kernels;
    others are copied.  Returns ``y_host``."""
    w_packed, w_scale, M, N, K = _check(x_dev, w_packed, w_scale)
    n_out = N // 2 if flags & FLAG_SWIGLU else N
    dtype = torch.float32 if flags & FLAG_F32_OUT else torch.bfloat16
    for name, t, want_dev in (("x_host", x_host, False), ("y_host", y_host, False),
                              ("y_dev", y_dev, True)):
        shape = (M, K) if name == "x_host" else (M, n_out)
        tdt = torch.bfloat16 if name == "x_host" else dtype
        if (t.dtype != tdt or tuple(t.shape) != shape or not t.is_contiguous()
                or t.is_cuda != want_dev or (want_dev and t.device != x_dev.device)):
            raise ValueError("%s must be a contiguous %s tensor of shape %s %s"
                             % (name, tdt, shape, "on %s" % x_dev.device if want_dev
                                else "in host memory"))
    if stream is None:
        stream = torch.cuda.current_stream(x_dev.device)
    with _on_device(x_dev.device):
        st = library().nvfp4_linear_host(x_host.data_ptr(), x_dev.data_ptr(),
                                         w_packed.data_ptr(), w_scale.data_ptr(),
                                         float(global_scale), y_dev.data_ptr(),
                                         y_host.data_ptr(), M, N, K, int(flags),
                                         ctypes.c_void_p(stream.cuda_stream))
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_linear_host")
    return y_host


def linear_host_noalloc(x_host, w_packed, w_scale, global_scale, y_host, flags=0, stream=None):
    """Call nvfp4_linear_host_noalloc: the layer on host activations
    ``x_host`` into the host tensor ``y_host``, staged through the library's
    own fixed device scratch (no device buffer from the caller).  Returns
    ``y_host``."""
    if not (w_packed.is_cuda and w_scale.is_cuda):
        raise ValueError("w_packed and w_scale must be CUDA tensors")
    w_packed, w_scale = _as_u8(w_packed, "w_packed"), _as_u8(w_scale, "w_scale")
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("x_host and y_host must be in host memory")
    if x_host.dtype != torch.bfloat16 or x_host.dim() != 2 or not x_host.is_contiguous():
        raise TypeError("x_host must be a contiguous 2-D bfloat16 tensor")
    M, K = x_host.shape
    N = w_packed.shape[0]
    if tuple(w_packed.shape) != (N, K // 2) or tuple(w_scale.shape) != (N, K // 16):
        raise ValueError("shapes disagree: x %s, w_packed %s, w_scale %s"
                         % (tuple(x_host.shape), tuple(w_packed.shape), tuple(w_scale.shape)))
    n_out = N // 2 if flags & FLAG_SWIGLU else N
    dtype = torch.float32 if flags & FLAG_F32_OUT else torch.bfloat16
    if y_host.dtype != dtype or tuple(y_host.shape) != (M, n_out) or not y_host.is_contiguous():
        raise ValueError("y_host must be a contiguous %s tensor of shape %s" % (dtype, (M, n_out)))
    if stream is None:
        stream = torch.cuda.current_stream(w_packed.device)
    with _on_device(w_packed.device):
        st = library().nvfp4_linear_host_noalloc(
            x_host.data_ptr(), w_packed.data_ptr(), w_scale.data_ptr(), float(global_scale),
            y_host.data_ptr(), M, N, K, int(flags), ctypes.c_void_p(stream.cuda_stream))
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_linear_host_noalloc")
    return y_host


def linear(x, w_packed, w_scale, global_scale, out=None, stream=None):
    """y[M, N] bf16 = x[M, K] . W^T with W the dequantised NVFP4 weight."""
    return linear_ex(x, w_packed, w_scale, global_scale, 0, out, stream)


def linear_f32(x, w_packed, w_scale, global_scale, out=None, stream=None):
    """Same as ``linear`` with fp32 output (before the bf16 rounding)."""
    return linear_ex(x, w_packed, w_scale, global_scale, FLAG_F32_OUT, out, stream)


def linear_swiglu(x, w_packed, w_scale, global_scale, out=None, stream=None):
    """Fused gate/up: y[M, N/2] bf16 = silu(x W_gate^T) * (x W_up^T)."""
    return linear_ex(x, w_packed, w_scale, global_scale, FLAG_SWIGLU, out, stream)


def linear_swiglu_f32(x, w_packed, w_scale, global_scale, out=None, stream=None):
    return linear_ex(x, w_packed, w_scale, global_scale, FLAG_SWIGLU | FLAG_F32_OUT, out,
                     stream)


def linear_swiglu_gs(x, w_packed, w_scale, gate_global_scale, up_global_scale, flags=0,
                     out=None, stream=None):
    """nvfp4_linear_swiglu_gs: SwiGLU with separate gate and up global scales."""
    w_packed, w_scale, M, N, K = _check(x, w_packed, w_scale)
    dtype = torch.float32 if flags & FLAG_F32_OUT else torch.bfloat16
    if out is None:
        out = torch.empty((M, N // 2), dtype=dtype, device=x.device)
    elif (out.dtype != dtype or tuple(out.shape) != (M, N // 2) or not out.is_contiguous()
          or out.device != x.device):
        raise ValueError("out must be a contiguous %s tensor of shape %s on %s"
                         % (dtype, (M, N // 2), x.device))
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with _on_device(x.device):
        st = library().nvfp4_linear_swiglu_gs(
            x.data_ptr(), w_packed.data_ptr(), w_scale.data_ptr(), float(gate_global_scale),
            float(up_global_scale), out.data_ptr(), M, N, K, int(flags),
            ctypes.c_void_p(stream.cuda_stream))
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_linear_swiglu_gs")
    return out


def linear_segmented(x, w_packed, w_scale, global_scales, segment_rows, flags=0, out=None,
                     stream=None):
    """nvfp4_linear_segmented: one launch over stacked projections, each row
    segment with its own global scale; y holds the segments' outputs side by
    side."""
    w_packed, w_scale, M, N, K = _check(x, w_packed, w_scale)
    gs = (ctypes.c_float * len(global_scales))(*[float(g) for g in global_scales])
    rows = (ctypes.c_int64 * len(segment_rows))(*[int(r) for r in segment_rows])
    dtype = torch.float32 if flags & FLAG_F32_OUT else torch.bfloat16
    if out is None:
        out = torch.empty((M, N), dtype=dtype, device=x.device)
    elif (out.dtype != dtype or tuple(out.shape) != (M, N) or not out.is_contiguous()
          or out.device != x.device):
        raise ValueError("out must be a contiguous %s tensor of shape %s on %s"
                         % (dtype, (M, N), x.device))
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with _on_device(x.device):
        st = library().nvfp4_linear_segmented(
            x.data_ptr(), w_packed.data_ptr(), w_scale.data_ptr(), ctypes.cast(gs, ctypes.c_void_p),
            ctypes.cast(rows, ctypes.c_void_p), len(segment_rows), out.data_ptr(), M, N, K,
            int(flags), ctypes.c_void_p(stream.cuda_stream))
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_linear_segmented")
    return out


def quantize(w, stream=None):
    """nvfp4_quantize: bf16 weights [N, K] -> (w_packed [N, K/2] u8,
    w_scale [N, K/16] u8, global_scale [1] fp32), all on w's device."""
    if not w.is_cuda:
        raise ValueError("w must be a CUDA tensor")
    if w.dtype != torch.bfloat16 or w.dim() != 2 or not w.is_contiguous():
        raise TypeError("w must be a contiguous 2-D bfloat16 tensor")
    N, K = w.shape
    wp = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    ws = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    gs = torch.empty(1, dtype=torch.float32, device=w.device)
    if stream is None:
        stream = torch.cuda.current_stream(w.device)
    with _on_device(w.device):
        st = library().nvfp4_quantize(w.data_ptr(), N, K, wp.data_ptr(), ws.data_ptr(),
                                      gs.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_quantize")
    return wp, ws, gs


def quantize_fp8(w_fp8, scale_inv, block=128, stream=None):
    """nvfp4_quantize_fp8: a block-scaled FP8 tensor (e4m3 [N, K], as uint8
    or float8_e4m3fn, with fp32 scale_inv [ceil(N/block), ceil(K/block)])
    -> (w_packed, w_scale, global_scale) like ``quantize``."""
    if not (w_fp8.is_cuda and scale_inv.is_cuda) or w_fp8.device != scale_inv.device:
        raise ValueError("w_fp8 and scale_inv must be CUDA tensors on one device")
    if w_fp8.dtype == torch.float8_e4m3fn:
        w_fp8 = w_fp8.view(torch.uint8)
    if w_fp8.dtype != torch.uint8 or w_fp8.dim() != 2 or not w_fp8.is_contiguous():
        raise TypeError("w_fp8 must be a contiguous 2-D uint8 / float8_e4m3fn tensor")
    N, K = w_fp8.shape
    shape = (-(-N // block), -(-K // block))
    if (scale_inv.dtype != torch.float32 or tuple(scale_inv.shape) != shape
            or not scale_inv.is_contiguous()):
        raise ValueError("scale_inv must be a contiguous float32 tensor of shape %s" % (shape,))
    wp = torch.empty((N, K // 2), dtype=torch.uint8, device=w_fp8.device)
    ws = torch.empty((N, K // 16), dtype=torch.uint8, device=w_fp8.device)
    gs = torch.empty(1, dtype=torch.float32, device=w_fp8.device)
    if stream is None:
        stream = torch.cuda.current_stream(w_fp8.device)
    with _on_device(w_fp8.device):
        st = library().nvfp4_quantize_fp8(w_fp8.data_ptr(), scale_inv.data_ptr(), int(block),
                                          N, K, wp.data_ptr(), ws.data_ptr(), gs.data_ptr(),
                                          ctypes.c_void_p(stream.cuda_stream))
    if st != OK:
        raise Nvfp4Error(st, "nvfp4_quantize_fp8")
    return wp, ws, gs


def choose_plan(M, N, K, flags=0):
    """Name of the kernel a call would launch ('smallm' / 'tcgemm'), or None."""
    return KERNEL_NAMES.get(kernel_for(M, N, K, flags))
