"""The seeded input recipes and the bench's algorithmic accounting.

Byte and flop totals are pinned to numbers written out by hand from the
checkpoint layout (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", section 1,
condition 2: codes K/2 bytes per weight row, e4m3 scales K/16 bytes per row;
x and y bf16; one fp32 global scale) for each benchmarked shape, so that
the roofline's numerator cannot drift from the definition."""
import numpy as np
import torch

from nvfp4_block_scaled_linear_gb300.inputs import (GLOBAL_SCALE, SCALE_HI, SCALE_LO, WORKLOADS,
                                                     algorithmic_bytes, flops,
                                                     fp8_checkpoint_tensor, make_linear,
                                                     quantizer_weight)


def _total_bytes(name):
    w = WORKLOADS[name]
    return sum(algorithmic_bytes(M, N, K, w.swiglu) for (M, N, K, _) in w.shapes)


def test_algorithmic_bytes_of_the_benchmarked_shapes():
    # 34816*5120/2 + 34816*320 + 2*5120 + 2*34816 + 4
    assert _total_bytes("decode_gate_up") == 89_128_960 + 11_141_120 + 10_240 + 69_632 + 4
    # 5120*17408/2 + 5120*1088 + 2*7*17408 + 2*7*5120 + 4
    assert _total_bytes("verify_down") == 44_564_480 + 5_570_560 + 243_712 + 71_680 + 4
    assert _total_bytes("tiny") == 65_536 + 8_192 + 1_024 + 512 + 4
    assert _total_bytes("layer_m32") == 197_263_376
    # prefill: y is [8192, 34816] bf16, or [8192, 17408] after SwiGLU
    assert _total_bytes("prefill") == 100_270_080 + 83_886_080 + 570_425_344 + 4
    assert _total_bytes("prefill_swiglu") == 100_270_080 + 83_886_080 + 285_212_672 + 4


def test_flops_of_the_benchmarked_shapes():
    assert flops(1, 34816, 5120) == 2 * 34816 * 5120
    assert flops(8192, 34816, 5120) == 2_920_577_761_280


def test_linear_recipe_is_seeded_and_in_range():
    a = make_linear(3, 256, 512, seed=9, big_row_frac=0.34)
    b = make_linear(3, 256, 512, seed=9, big_row_frac=0.34)
    assert np.array_equal(a.x_bits, b.x_bits) and np.array_equal(a.w_packed, b.w_packed)
    assert np.array_equal(a.w_scale, b.w_scale)
    assert a.w_packed.shape == (256, 256) and a.w_scale.shape == (256, 32)
    assert a.w_scale.min() >= SCALE_LO and a.w_scale.max() <= SCALE_HI
    assert a.global_scale == GLOBAL_SCALE
    # every nibble value appears (codes uniform over the 16 e2m1 patterns)
    nib = np.concatenate([a.w_packed & 15, a.w_packed >> 4]).ravel()
    assert np.unique(nib).size == 16
    c = make_linear(3, 256, 512, seed=10)
    assert not np.array_equal(a.w_packed, c.w_packed)


def test_quantizer_recipes_are_seeded_and_in_range():
    w1, w2 = quantizer_weight(64, 256), quantizer_weight(64, 256)
    assert w1.dtype == torch.bfloat16 and w1.shape == (64, 256)
    assert torch.equal(w1.view(torch.int16), w2.view(torch.int16))
    w8, sinv = fp8_checkpoint_tensor(300, 256, 128)
    assert w8.dtype == torch.float8_e4m3fn and w8.shape == (300, 256)
    assert sinv.dtype == torch.float32 and sinv.shape == (3, 2)
    assert float(sinv.min()) >= np.exp(-9.0) * 0.999 and float(sinv.max()) <= np.exp(2.0) * 1.001
    bits = w8.view(torch.uint8).numpy()
    assert not ((bits & 0x7F) == 0x7F).any()
    w8b, sinvb = fp8_checkpoint_tensor(300, 256, 128)
    assert torch.equal(w8.view(torch.uint8), w8b.view(torch.uint8)) and torch.equal(sinv, sinvb)
