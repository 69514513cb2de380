"""Run one layer call a few times on seeded inputs, for a profiler.

    python -m nvfp4_block_scaled_linear_gb300.run_case M N K [flags] [calls]

Draws the inputs with the package's seeded generator (seed 11; 1% of the
activation rows scaled by 8 when M > 32, as in the prefill configuration),
makes `calls` calls of nvfp4_linear_ex with `flags` on cuda:0 through the C
ABI, synchronises, and prints the kernel the calls ran.  Profile commands
select the launches to capture with the profiler's own filters (kernel name,
number of launches skipped).
"""
import sys

import numpy as np
import torch

from . import _lib
from .inputs import make_linear


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    if len(argv) < 3:
        raise SystemExit(__doc__)
    M, N, K = (int(v) for v in argv[:3])
    flags = int(argv[3]) if len(argv) > 3 else 0
    calls = int(argv[4]) if len(argv) > 4 else 5
    _lib.load_library()
    t = make_linear(M, N, K, seed=11, big_row_frac=0.01 if M > 32 else 0.0)
    dev = torch.device("cuda:0")
    x = torch.from_numpy(t.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    wp = torch.from_numpy(t.w_packed).to(dev)
    ws = torch.from_numpy(t.w_scale).to(dev)
    y = None
    for _ in range(calls):
        y = _lib.linear_ex(x, wp, ws, float(t.global_scale), flags, out=y)
    torch.cuda.synchronize()
    print("%s: %d calls of M=%d N=%d K=%d flags=%d" % (_lib.choose_plan(M, N, K, flags), calls,
                                                         M, N, K, flags))


if __name__ == "__main__":
    main()
