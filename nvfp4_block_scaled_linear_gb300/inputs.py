"""Seeded synthetic inputs for the NVFP4 W4A16 linear layer.

This module only draws random numbers and stores them in the checkpoint's
layouts; it holds none of the layer's arithmetic (no decoding, no dot
products), so both the CUDA path's tests and the CPU oracle can take their
inputs from it.

Layouts (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", section 1, checkpoint
condition 2):
    x            bf16 bits, uint16 [M, K], row-major
    w_packed     uint8 [N, K/2]   two e2m1 codes per byte (low nibble = even k)
    w_scale      uint8 [N, K/16]  e4m3 bit patterns
    global_scale float32 scalar

Distributions (the synthetic stand-in for the checkpoint and prompts, which
are not available here):
    * packed bytes uniform over 0..255, so each nibble is uniform over the 16
      e2m1 codes, -0 included;
    * scale bytes uniform over the 49 patterns 0x20..0x50, which are exactly
      the finite positive e4m3 values in [2^-3, 2^3];
    * global scale float32(448 / 6), i.e. the "448 / amax" form with amax 6;
    * activations float32 N(0, 1) rounded to bf16 (round to nearest even, by
      torch's CPU conversion); optionally a fraction of rows scaled by 8
      before rounding (exact: a power of two), rows drawn without replacement.
Draw order from ``numpy.random.default_rng(seed)``: packed bytes, scales,
activations, big-row indices.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

GLOBAL_SCALE = np.float32(448.0 / 6.0)
SCALE_LO, SCALE_HI = 0x20, 0x50          # e4m3 2^-3 and 2^3, inclusive


@dataclass
class LinearInputs:
    x_bits: np.ndarray          # uint16 [M, K]
    w_packed: np.ndarray        # uint8 [N, K/2]
    w_scale: np.ndarray         # uint8 [N, K/16]
    global_scale: np.float32
    big_rows: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))
    name: str = ""

    @property
    def M(self):
        return self.x_bits.shape[0]

    @property
    def K(self):
        return self.x_bits.shape[1]

    @property
    def N(self):
        return self.w_packed.shape[0]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (torch's CPU conversion, RNE); return bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def draw_linear(rng: np.random.Generator, M: int, N: int, K: int,
                big_row_frac: float = 0.0, big_row_factor: float = 8.0,
                name: str = "") -> LinearInputs:
    if K % 16:
        raise ValueError("K must be a multiple of 16 (one scale per 16 inputs)")
    w_packed = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    w_scale = rng.integers(SCALE_LO, SCALE_HI + 1, size=(N, K // 16),
                           dtype=np.uint8)
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_big = int(round(big_row_frac * M))
    big = np.sort(rng.choice(M, size=n_big, replace=False)).astype(np.int64) \
        if n_big else np.zeros(0, np.int64)
    if n_big:
        x[big] *= np.float32(big_row_factor)
    return LinearInputs(f32_to_bf16_bits(x), w_packed, w_scale, GLOBAL_SCALE,
                        big, name)


def make_linear(M: int, N: int, K: int, seed: int, big_row_frac: float = 0.0,
                name: str = "") -> LinearInputs:
    return draw_linear(np.random.default_rng(seed), M, N, K, big_row_frac,
                       name=name)


@dataclass
class Workload:
    """One named synthetic configuration: one or more linears, one seed."""
    name: str
    shapes: List[tuple]                  # (M, N, K, label)
    seed: int
    big_row_frac: float = 0.0
    swiglu: bool = False
    description: str = ""

    def draw(self, max_rows: Optional[int] = None) -> List[LinearInputs]:
        rng = np.random.default_rng(self.seed)
        out = []
        for (M, N, K, label) in self.shapes:
            out.append(draw_linear(rng, M if max_rows is None else min(M, max_rows),
                                   N, K, self.big_row_frac, name=label))
        return out


# The five configurations: a tiny correctness case, the decode GEMV over the
# fused MLP gate+up of a 5120-wide model, the speculative-verify M = K+1 = 7
# down projection, one decoder layer's four NVFP4 linears at a continuous
# batch of 32, and a cold 8192-row prefill chunk of the gate+up projection
# (optionally with the SwiGLU epilogue).
WORKLOADS = {
    "tiny": Workload("tiny", [(1, 256, 512, "tiny")], seed=0,
                     description="M=1 K=512 N=256"),
    "decode_gate_up": Workload("decode_gate_up", [(1, 34816, 5120, "gate_up")],
                               seed=1, description="M=1 K=5120 N=34816"),
    "verify_down": Workload("verify_down", [(7, 5120, 17408, "down")], seed=2,
                            description="M=7 K=17408 N=5120"),
    "layer_m32": Workload("layer_m32", [(32, 34816, 5120, "gate_up"),
                                        (32, 5120, 17408, "down"),
                                        (32, 8192, 5120, "qkv"),
                                        (32, 5120, 6144, "o")], seed=3,
                          description="M=32: gate_up, down, q/k/v, o"),
    "prefill": Workload("prefill", [(8192, 34816, 5120, "gate_up")], seed=4,
                        big_row_frac=0.01,
                        description="M=8192 K=5120 N=34816, 1% rows x8"),
    "prefill_swiglu": Workload("prefill_swiglu", [(8192, 34816, 5120, "gate_up")],
                               seed=4, big_row_frac=0.01, swiglu=True,
                               description="as prefill, SwiGLU epilogue -> "
                                           "[8192, 17408]"),
}


# The load-time quantisers' inputs, on the decode gate+up weight shape: a
# bf16 weight of N(0, 0.02^2) values, and a block-scaled FP8 checkpoint
# tensor (e4m3 codes of N(0, 60^2) values by torch's round-to-nearest
# conversion -- values past 448 would become NaN codes, a 7.5-sigma event
# absent from these draws -- and one fp32 scale_inv per 128 x 128 tile,
# exp(U(-9, 2))).  CPU tensors, drawn from torch.Generator(seed).
def quantizer_weight(N: int = 34816, K: int = 5120, seed: int = 11) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16)


def fp8_checkpoint_tensor(N: int = 34816, K: int = 5120, block: int = 128, seed: int = 12):
    """(w8 float8_e4m3fn [N, K], scale_inv float32 [ceil(N/block), ceil(K/block)])."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    w8 = (torch.randn((N, K), generator=g) * 60.0).to(torch.float8_e4m3fn)
    sinv = torch.exp(torch.empty((-(-N // block), -(-K // block))).uniform_(-9, 2, generator=g))
    return w8, sinv


def algorithmic_bytes(M: int, N: int, K: int, swiglu: bool = False) -> int:
    """Bytes the layer must move: packed weights and scales once, x once,
    y once (bf16), the global scale once."""
    n_out = N // 2 if swiglu else N
    return N * K // 2 + N * K // 16 + 2 * M * K + 2 * M * n_out + 4


def flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
