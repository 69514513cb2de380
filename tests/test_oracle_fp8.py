"""Pins of the oracle's FP8 -> BF16 step (the first half of the FP8 -> BF16
-> NVFP4 load-time conversion): block-scaled e4m3 with one fp32 scale_inv
per B x B block, checked against torch's own float8_e4m3fn decode, fp32
multiply and bf16 rounding, and the block index on ragged edges."""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_mutants import fp8_torch_case


@pytest.mark.parametrize("N,K,block,seed", [(200, 272, 128, 5), (64, 48, 16, 6), (1, 16, 128, 7),
                                            (257, 129, 64, 8)])
def test_fp8_to_bf16_matches_torch(N, K, block, seed):
    w8, sinv, want = fp8_torch_case(N, K, block, seed)
    assert np.array_equal(oracle.fp8_to_bf16(w8, sinv, block), want)


def test_fp8_block_index_on_ragged_edges():
    # all codes 1.0; block (i, j) scaled by 2^(3i + j): every output names its block
    N, K, B = 300, 200, 128
    w8 = np.full((N, K), 0x38, np.uint8)
    sinv = np.float32([[2.0 ** (3 * i + j) for j in range(2)] for i in range(3)])
    out = oracle.fp8_to_bf16(w8, sinv, B)
    vals = (out.astype(np.uint32) << 16).view(np.float32)
    n = np.arange(N)[:, None] // B
    k = np.arange(K)[None, :] // B
    assert np.array_equal(vals, np.exp2(3 * n + k).astype(np.float32))


def test_fp8_rounding_to_bf16_is_nearest_even():
    # e4m3 1.875 (0x3F) times 1 + 2^-7 + 2^-9 -> 1.8896..., not representable in bf16:
    # the bf16 neighbours 1.875 and 1.8828125; RNE picks the nearer
    w8 = np.array([[0x3F, 0x38]], np.uint8)
    s = np.float32([[1.0 + 2.0 ** -7 + 2.0 ** -9]])
    out = oracle.fp8_to_bf16(w8, s, 128)
    want = torch.tensor([1.875 * float(s[0, 0]), float(s[0, 0])], dtype=torch.float32) \
        .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out[0], want)
    assert out[0, 1] == 0x3F81          # 1 + 2^-7 + 2^-9 -> 1 + 2^-7 (ties not involved)


def test_quantize_fp8_is_the_bf16_rule_on_the_converted_tensor():
    w8, sinv, _ = fp8_torch_case(64, 256, 128, 9)
    a = oracle.quantize_fp8(w8, sinv, 128)
    b = oracle.quantize(oracle.fp8_to_bf16(w8, sinv, 128))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


def test_scale_inv_shape_is_checked():
    with pytest.raises(ValueError):
        oracle.fp8_to_bf16(np.zeros((4, 32), np.uint8), np.ones((1, 2), np.float32), 128)
