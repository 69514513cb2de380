"""GPU parity of the quantiser (nvfp4_quantize) with the oracle's: codes,
block scales and global scale bit for bit, on seeded weights shaped like a
checkpoint's projections, with outlier rows, all-zero and tiny blocks (e4m3
subnormal scales), weights that round to -0 and the saturation edge."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_linear_gb300 import _lib
from nvfp4_block_scaled_linear_gb300 import build as cuda_build
from nvfp4_block_scaled_linear_gb300.inputs import f32_to_bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    cuda_build.build()
    _lib.load_library()
    _lib.device_error(clear=True)
    yield
    assert _lib.device_error(clear=True) == 0


def _weights(N, K, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    if N > 3:
        w[1] *= 40.0                                   # an outlier row sets the tensor amax
        w[2, : min(K, 64)] = 0.0                       # all-zero blocks
        w[3] *= 1e-4                                   # tiny blocks: subnormal e4m3 scales
    w[0, 5] = -1e-6                                    # rounds to -0 next to larger weights
    return f32_to_bf16_bits(w)


def _gpu(bits):
    w = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    wp, ws, gs = _lib.quantize(w)
    torch.cuda.synchronize()
    return wp.cpu().numpy(), ws.cpu().numpy(), np.float32(gs.cpu().numpy()[0])


@pytest.mark.parametrize("N,K", [(1, 16), (7, 48), (64, 256), (300, 1024), (2048, 5120)])
def test_quantize_bit_exact(N, K):
    bits = _weights(N, K, seed=N * 3 + K)
    wp, ws, gs = _gpu(bits)
    wp_o, ws_o, gs_o = oracle.quantize(bits)
    assert gs == gs_o
    assert np.array_equal(ws, ws_o), np.argwhere(ws != ws_o)[:5]
    assert np.array_equal(wp, wp_o), np.argwhere(wp != wp_o)[:5]


def test_quantize_hand_values_and_saturation():
    # one row: the tensor maximum 6 in block 0; block 1 crosses the e2m1
    # midpoints of the oracle's table after scaling
    w = np.zeros((2, 32), np.float32)
    w[0, :8] = [6.0, 3.0, 1.5, -6.0, 0.5, 1.0, 2.0, 4.0]
    w[1, 16:24] = [0.75, -0.375, 0.1875, 0.0625, 0.03125, -0.015625, 5.0, -5.9]
    bits = f32_to_bf16_bits(w)
    wp, ws, gs = _gpu(bits)
    wp_o, ws_o, gs_o = oracle.quantize(bits)
    assert gs == gs_o and np.array_equal(ws, ws_o) and np.array_equal(wp, wp_o)


def test_all_zero_tensor():
    bits = np.zeros((4, 64), np.uint16)
    wp, ws, gs = _gpu(bits)
    assert gs == np.float32(1.0) and not wp.any() and not ws.any()


def test_quantised_weights_drive_the_linear():
    """Quantise on the GPU, then run the linear on the result: equal to the
    oracle's linear on the oracle's quantisation of the same weights."""
    from _parity import check_f32
    N, K, M = 512, 1024, 3
    bits = _weights(N, K, seed=77)
    w = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    wp, ws, gs = _lib.quantize(w)
    x_bits = f32_to_bf16_bits(np.random.default_rng(78).standard_normal((M, K)).astype(np.float32))
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    y = _lib.linear_f32(x, wp, ws, float(gs.item()))
    torch.cuda.synchronize()
    wp_o, ws_o, gs_o = oracle.quantize(bits)
    y64, a = oracle.linear_f64(x_bits, wp_o, ws_o, gs_o)
    check_f32(y.cpu().numpy(), y64, a, "quantise then linear")


# ------------------------------------------------------------------ FP8 source
def _fp8_case(N, K, block, seed):
    """Block-scaled FP8 weights shaped like a checkpoint tensor: e4m3 codes of
    N(0, 1) values (NaN codes excluded) and one fp32 scale_inv per block."""
    rng = np.random.default_rng(seed)
    w = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32) * 60.0)
    w8 = w.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    nb, kb = -(-N // block), -(-K // block)
    sinv = np.exp(rng.uniform(-9, 2, size=(nb, kb))).astype(np.float32)
    return np.ascontiguousarray(w8), sinv


# units of four 16-input blocks where K and block are multiples of 64
# (300/1024/128, 129/4096/64, 2048/5120/128, 33/384/192 with a block that is
# not a power of two), single blocks otherwise (the rest; 50/768/48: K is a
# multiple of 64, the block is not)
@pytest.mark.parametrize("N,K,block", [(1, 16, 16), (7, 48, 16), (200, 272, 128),
                                       (300, 1024, 128), (129, 4096, 64), (2048, 5120, 128),
                                       (33, 384, 192), (50, 768, 48)])
def test_quantize_fp8_bit_exact(N, K, block):
    w8, sinv = _fp8_case(N, K, block, seed=N + K + block)
    wp, ws, gs = _lib.quantize_fp8(torch.from_numpy(w8).to(DEV), torch.from_numpy(sinv).to(DEV),
                                   block)
    torch.cuda.synchronize()
    wp_o, ws_o, gs_o = oracle.quantize_fp8(w8, sinv, block)
    assert np.float32(gs.cpu().numpy()[0]) == gs_o
    assert np.array_equal(ws.cpu().numpy(), ws_o)
    assert np.array_equal(wp.cpu().numpy(), wp_o)


@pytest.mark.parametrize("N,K,block", [(70, 512, 128), (9, 272, 16)])
def test_quantize_fp8_edge_codes(N, K, block):
    """FP8 bytes at the edges of the format: +-0, +-448 (the largest finite
    e4m3), the smallest subnormals, whole zero units and blocks whose
    largest image sets the tensor maximum; with the smallest and largest
    tile scales."""
    w8, sinv = _fp8_case(N, K, block, seed=N * K + 5)
    w8[0, :64] = 0x80                                  # -0 everywhere in a unit
    w8[1, :16] = [0x7E, 0xFE, 0x01, 0x81, 0x00, 0x80] + [0x08] * 10
    w8[2, 16:32] = 0x01                                # subnormal-only block
    w8[3, :] = np.where(np.arange(K) % 2 == 0, 0x7E, 0xFE)   # +-448 row
    sinv[0, 0] = np.float32(2.0 ** -40)
    sinv[-1, -1] = np.float32(2.0 ** 6)
    wp, ws, gs = _lib.quantize_fp8(torch.from_numpy(w8).to(DEV), torch.from_numpy(sinv).to(DEV),
                                   block)
    torch.cuda.synchronize()
    wp_o, ws_o, gs_o = oracle.quantize_fp8(w8, sinv, block)
    assert np.float32(gs.cpu().numpy()[0]) == gs_o
    assert np.array_equal(ws.cpu().numpy(), ws_o)
    assert np.array_equal(wp.cpu().numpy(), wp_o)


def test_quantize_fp8_unaligned_scale_output_takes_the_single_block_path():
    """w_scale one byte into its allocation cannot take the four-block
    units' word stores: the call takes single blocks and writes the same
    bytes."""
    import ctypes
    N, K, block = 256, 1024, 128
    w8, sinv = _fp8_case(N, K, block, seed=41)
    w8_t = torch.from_numpy(w8).to(DEV)
    s_t = torch.from_numpy(sinv).to(DEV)
    wp_a, ws_a, gs_a = _lib.quantize_fp8(w8_t, s_t, block)
    wp = torch.empty((N, K // 2), dtype=torch.uint8, device=DEV)
    ws_buf = torch.full((N * (K // 16) + 16,), 0xAB, dtype=torch.uint8, device=DEV)
    gs = torch.empty(1, dtype=torch.float32, device=DEV)
    st = _lib.library().nvfp4_quantize_fp8(
        w8_t.data_ptr(), s_t.data_ptr(), block, N, K, wp.data_ptr(), ws_buf.data_ptr() + 1,
        gs.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(wp, wp_a) and torch.equal(gs, gs_a)
    ws_u = ws_buf.cpu().numpy()
    assert np.array_equal(ws_u[1:1 + N * (K // 16)], ws_a.cpu().numpy().ravel())
    assert ws_u[0] == 0xAB and (ws_u[1 + N * (K // 16):] == 0xAB).all()


def test_quantize_fp8_equals_bf16_quantiser_on_the_converted_tensor():
    """The FP8 entry point equals nvfp4_quantize applied to the bf16 tensor
    torch converts from the same FP8 codes and scales (both on the GPU)."""
    N, K, block = 384, 2048, 128
    w8, sinv = _fp8_case(N, K, block, seed=31)
    w8_t = torch.from_numpy(w8).to(DEV)
    s_t = torch.from_numpy(sinv).to(DEV)
    s_full = s_t.repeat_interleave(block, 0)[:N].repeat_interleave(block, 1)[:, :K]
    w_bf16 = (w8_t.view(torch.float8_e4m3fn).to(torch.float32) * s_full).to(torch.bfloat16)
    a = _lib.quantize_fp8(w8_t.view(torch.float8_e4m3fn), s_t, block)
    b = _lib.quantize(w_bf16.contiguous())
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ------------------------------------------------------------------ full size
def _sampled_rows(row_absmax, rng, count=509):
    """Random rows plus the first, the last and the one holding the tensor's
    largest magnitude (so that the global scale over the sample is the
    tensor's)."""
    N = row_absmax.shape[0]
    extra = [0, N - 1, int(np.argmax(row_absmax))]
    return np.unique(np.concatenate([rng.choice(N, count, replace=False), extra]))


def test_quantizers_at_the_benchmarked_size_on_sampled_rows():
    """The bench's quantiser inputs (34816 x 5120: the bf16 weight and the
    block-scaled FP8 tensor), checked bit for bit on sampled rows.  Rows
    quantise independently given the global scale, and the sample holds the
    row with the largest |w| (for FP8, the largest |bf16 image|), so the
    oracle's global scale over the sample is the whole tensor's."""
    from nvfp4_block_scaled_linear_gb300.inputs import fp8_checkpoint_tensor, quantizer_weight
    rng = np.random.default_rng(77)
    w = quantizer_weight()
    wp, ws, gs = _lib.quantize(w.to(DEV))
    torch.cuda.synchronize()
    rows = _sampled_rows(w.float().abs().amax(1).numpy(), rng)
    wp_o, ws_o, gs_o = oracle.quantize(w.view(torch.int16).numpy().view(np.uint16)[rows])
    assert np.float32(gs.cpu().numpy()[0]) == gs_o
    assert np.array_equal(ws.cpu().numpy()[rows], ws_o)
    assert np.array_equal(wp.cpu().numpy()[rows], wp_o)
    del w, wp, ws

    w8, sinv = fp8_checkpoint_tensor()
    w8_bits = w8.view(torch.uint8).numpy()
    assert not ((w8_bits & 0x7F) == 0x7F).any()          # no NaN codes in the draw
    wp, ws, gs = _lib.quantize_fp8(w8.to(DEV), sinv.to(DEV), 128)
    torch.cuda.synchronize()
    img = oracle.fp8_to_bf16(w8_bits, sinv.numpy(), 128)
    img_absmax = torch.from_numpy(img.view(np.int16)).view(torch.bfloat16).float().abs().amax(1)
    rows = _sampled_rows(img_absmax.numpy(), rng)
    wp_o, ws_o, gs_o = oracle.quantize(img[rows])
    assert np.float32(gs.cpu().numpy()[0]) == gs_o
    assert np.array_equal(ws.cpu().numpy()[rows], ws_o)
    assert np.array_equal(wp.cpu().numpy()[rows], wp_o)
