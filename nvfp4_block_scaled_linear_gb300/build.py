"""Build libnvfp4_linear.so (sm_103a) in-tree with nvcc.

    python -m nvfp4_block_scaled_linear_gb300.build [--force] [--verbose]

Output: nvfp4_block_scaled_linear_gb300/_build/libnvfp4_linear.so (ignored by
git).  The CUDA runtime is linked as a shared library so that the process
shares one runtime (current device, streams) with PyTorch.
"""
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libnvfp4_linear.so")
MAIN = os.path.join(CSRC, "nvfp4_linear.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) +
                  glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(ROOT, "include", "*.h")))


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(s) for s in _sources())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-cudart", "shared",
           "-o", tmp, MAIN]
    if verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
