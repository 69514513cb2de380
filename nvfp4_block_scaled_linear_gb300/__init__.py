"""GB300 (sm_103a) NVFP4 W4A16 block-scaled linear layer.

The compute lives in ``libnvfp4_linear.so`` (CUDA, built from ``csrc/``);
``linear``, ``linear_swiglu`` and friends are thin ctypes marshalling around
its C ABI (``include/nvfp4_linear.h``).  Nothing here computes on the CPU: if
the library or a GPU is missing, every call raises.
"""
from .inputs import WORKLOADS, LinearInputs, algorithmic_bytes, flops  # noqa: F401


def __getattr__(name):
    # The binding is imported lazily so that the input generators stay
    # importable on machines without the built library.
    if name in ("linear", "linear_f32", "linear_swiglu", "linear_swiglu_f32",
                "status_string", "abi_version", "device_error", "library",
                "Nvfp4Error", "load_library", "choose_plan"):
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
