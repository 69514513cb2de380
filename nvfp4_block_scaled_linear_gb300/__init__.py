"""GB300 (sm_103a) NVFP4 W4A16 block-scaled linear layer.

The compute lives in ``libnvfp4_linear.so`` (CUDA, built from ``csrc/``);
``linear``, ``linear_swiglu`` and friends are thin ctypes marshalling around
its C ABI (``include/nvfp4_linear.h``).  Nothing here computes on the CPU: if
the library or a GPU is missing, every call raises.
"""
from .inputs import WORKLOADS, LinearInputs, algorithmic_bytes, flops  # noqa: F401


def __getattr__(name):
    # The binding (every public name of _lib: the calls, the flag and kernel
    # constants) is imported lazily so that the input generators stay
    # importable on machines without the built library.
    if not name.startswith("_"):
        from . import _lib
        if hasattr(_lib, name):
            return getattr(_lib, name)
    raise AttributeError(name)
