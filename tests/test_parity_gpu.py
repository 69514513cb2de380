"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element, on seeded inputs.  Tolerances are documented in _parity.py."""
import numpy as np
import pytest
import torch

import oracle
from _parity import (check_bf16, check_f32, check_swiglu_bf16, check_swiglu_f32, record)
from nvfp4_block_scaled_linear_gb300 import _lib
from nvfp4_block_scaled_linear_gb300 import build as cuda_build
from nvfp4_block_scaled_linear_gb300.inputs import (WORKLOADS, LinearInputs, draw_linear,
                                                    make_linear)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    cuda_build.build()
    _lib.load_library()
    _lib.device_error(clear=True)
    yield
    assert _lib.device_error(clear=True) == 0, "a kernel reported a wait timeout"


def to_dev(t: LinearInputs):
    x = torch.from_numpy(t.x_bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    return x, torch.from_numpy(t.w_packed).to(DEV), torch.from_numpy(t.w_scale).to(DEV)


def bf16_bits(y):
    return y.cpu().view(torch.int16).numpy().view(np.uint16)


def run(t, flags=0):
    x, wp, ws = to_dev(t)
    y = _lib.linear_ex(x, wp, ws, float(t.global_scale), flags)
    torch.cuda.synchronize()
    return y


def full_check(t, flags=0, what=""):
    y64, a = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    if flags & _lib.FLAG_SWIGLU:
        out64 = oracle.swiglu_f64(y64)
        y32 = run(t, flags | _lib.FLAG_F32_OUT).cpu().numpy()
        check_swiglu_f32(y32, y64, a, out64, what + " f32")
        ybf = bf16_bits(run(t, flags))
        return check_swiglu_bf16(ybf, y64, a, out64, oracle.to_bf16_bits(out64), what + " bf16")
    y32 = run(t, flags | _lib.FLAG_F32_OUT).cpu().numpy()
    check_f32(y32, y64, a, what + " f32")
    ybf = bf16_bits(run(t, flags))
    strict, _ = check_bf16(ybf, y64, a, oracle.to_bf16_bits(y64), what + " bf16")
    return strict


# ------------------------------------------------------------------ small M
# The few-row kernels, each forced (the default picks one by M): the tcgen05
# kernel in f16 and in bf16 (with two and with four lane groups) and the
# warp-MMA kernel.
GEMV_BF16 = _lib.FLAG_FORCE_GEMV | _lib.FLAG_BF16_MMA
FEW_ROW = [pytest.param(_lib.FLAG_FORCE_GEMV, id="gemv_tc"),
           pytest.param(GEMV_BF16 | _lib.FLAG_GROUPS(4), id="gemv_bf16_g4"),
           pytest.param(GEMV_BF16 | _lib.FLAG_GROUPS(2), id="gemv_bf16_g2"),
           pytest.param(_lib.FLAG_FORCE_SMALLM, id="smallm")]


@pytest.mark.parametrize("kflag", FEW_ROW)
@pytest.mark.parametrize("M", [1, 2, 5, 7, 8, 9, 16, 17, 24, 25, 31, 32])
def test_few_row_all_row_counts(M, kflag):
    t = make_linear(M, 384, 1024, seed=100 + M)
    want = {_lib.FLAG_FORCE_SMALLM: _lib.KERNEL_SMALLM, _lib.FLAG_FORCE_GEMV: _lib.KERNEL_GEMV}.get(
        kflag, _lib.KERNEL_GEMV_BF16)
    assert _lib.kernel_for(M, 384, 1024, kflag) == want
    assert _lib.kernel_for(M, 384, 1024) in (_lib.KERNEL_SMALLM, _lib.KERNEL_GEMV)
    full_check(t, kflag, what="few-row M=%d flags=%d" % (M, kflag))


@pytest.mark.parametrize("kflag", FEW_ROW)
@pytest.mark.parametrize("N,K", [(128, 256), (256, 768), (640, 4352), (1024, 2304)])
def test_few_row_shapes_and_uneven_splits(N, K, kflag):
    # K/256 stages split over clusters of CTAs, unevenly when they do not
    # divide
    t = make_linear(7, N, K, seed=N + K)
    full_check(t, kflag, what="few-row N=%d K=%d flags=%d" % (N, K, kflag))


@pytest.mark.parametrize("kflag", FEW_ROW)
@pytest.mark.parametrize("M", [1, 7, 16, 17, 32])
def test_few_row_swiglu(M, kflag):
    t = make_linear(M, 512, 1024, seed=300 + M)
    full_check(t, _lib.FLAG_SWIGLU | kflag, what="few-row swiglu M=%d flags=%d" % (M, kflag))


@pytest.mark.parametrize("M", [1, 7, 16, 32])
def test_gemv_tc_every_split(M):
    """The tcgen05 few-row kernel at every k split (one cluster of s CTAs,
    uneven when s does not divide the K/256 stages), forced."""
    N, K = 640, 4096
    t = make_linear(M, N, K, seed=1050 + M)
    y64, a = _oracle(t)
    for s in (1, 2, 3, 5, 7, 8, 16):
        _check_against(t, y64, a, _lib.FLAG_FORCE_GEMV | _lib.FLAG_SPLIT(s),
                       "gemv_tc M=%d split=%d" % (M, s))


@pytest.mark.parametrize("M", [1, 7, 16, 17, 32])
def test_gemv_bf16_every_split_and_group_count(M):
    """The bf16 tcgen05 few-row kernel at every k split, with two and with
    four lane groups: a CTA of 1..16 stages gives each group 1..64 jobs, so
    every TMEM ring position and every stage-barrier parity is exercised."""
    N, K = 640, 4096
    t = make_linear(M, N, K, seed=1070 + M)
    y64, a = _oracle(t)
    for g in (2, 4):
        for s in (1, 2, 3, 5, 7, 8, 16):
            _check_against(t, y64, a, GEMV_BF16 | _lib.FLAG_GROUPS(g) | _lib.FLAG_SPLIT(s),
                           "gemv_bf16 M=%d groups=%d split=%d" % (M, g, s))


@pytest.mark.parametrize("M", [9, 32])
def test_gemv_bf16_swiglu_every_split(M):
    """The k-split reduction of the bf16 tcgen05 few-row kernel with SwiGLU:
    two partial values (gate and up row) per output, pushed to the CTA that
    owns the output, for splits that divide the outputs unevenly."""
    t = make_linear(M, 640, 4096, seed=1090 + M)
    for g in (2, 4):
        for s in (1, 2, 3, 5, 16):
            full_check(t, _lib.FLAG_SWIGLU | GEMV_BF16 | _lib.FLAG_GROUPS(g) | _lib.FLAG_SPLIT(s),
                       what="gemv_bf16 swiglu M=%d groups=%d split=%d" % (M, g, s))


# ------------------------------------------------------------------ tcgen05
@pytest.mark.parametrize("M", [33, 64, 255, 256, 257, 600])
def test_tcgemm_row_counts_and_tails(M):
    t = make_linear(M, 384, 1024, seed=200 + M, big_row_frac=0.02)
    assert _lib.kernel_for(M, 384, 1024) == _lib.KERNEL_TCGEMM
    full_check(t, what="tcgemm M=%d" % M)


@pytest.mark.parametrize("N,K", [(128, 256), (256, 4096), (640, 512)])
def test_tcgemm_shapes(N, K):
    t = make_linear(100, N, K, seed=N * 7 + K)
    full_check(t, what="tcgemm N=%d K=%d" % (N, K))


@pytest.mark.parametrize("M", [40, 300])
def test_tcgemm_swiglu(M):
    t = make_linear(M, 512, 1024, seed=400 + M)
    full_check(t, _lib.FLAG_SWIGLU, what="tcgemm swiglu M=%d" % M)


@pytest.mark.parametrize("M", [1, 7, 32])
def test_every_kernel_at_small_m(M):
    t = make_linear(M, 256, 512, seed=500 + M)
    full_check(t, _lib.FLAG_FORCE_TCGEMM, what="forced tcgemm M=%d" % M)
    full_check(t, _lib.FLAG_FORCE_SMALLM, what="forced smallm M=%d" % M)
    full_check(t, _lib.FLAG_FORCE_GEMV, what="forced gemv_tc M=%d" % M)


def _oracle(t):
    y64, a = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    return y64, a


def _check_against(t, y64, a, flags, what):
    y32 = run(t, flags | _lib.FLAG_F32_OUT).cpu().numpy()
    check_f32(y32, y64, a, what + " f32")
    ybf = bf16_bits(run(t, flags))
    check_bf16(ybf, y64, a, oracle.to_bf16_bits(y64), what + " bf16")


@pytest.mark.parametrize("M", [1, 7, 16, 32])
def test_smallm_every_cta_height_and_split(M):
    """Every CTA height (16*g rows, g = 1..8; ragged row tails where 16*g
    does not divide N) and k split (one cluster of s CTAs, uneven when s
    does not divide the K/256 stages) of the warp-MMA kernel, forced."""
    N, K = 640, 4096
    t = make_linear(M, N, K, seed=1000 + M)
    y64, a = _oracle(t)
    g_max = 8 if M <= 16 else 4
    ran = 0
    for g in range(1, g_max + 1):
        for s in (1, 2, 3, 5, 8, 16):
            flags = _lib.FLAG_FORCE_SMALLM | _lib.FLAG_GROUPS(g) | _lib.FLAG_SPLIT(s)
            try:
                _check_against(t, y64, a, flags, "M=%d g=%d split=%d" % (M, g, s))
                ran += 1
            except _lib.Nvfp4Error as e:      # a layout that does not fit
                assert e.status == -1, str(e)
    assert ran >= 6 * g_max - 4, ran


@pytest.mark.parametrize("M", [1, 7, 32])
def test_smallm_swiglu_overrides(M):
    t = make_linear(M, 1024, 2048, seed=1100 + M)
    for g, s in ((1, 1), (2, 3), (4, 8)):
        full_check(t, _lib.FLAG_SWIGLU | _lib.FLAG_FORCE_SMALLM | _lib.FLAG_GROUPS(g) |
                   _lib.FLAG_SPLIT(s), what="swiglu M=%d g=%d split=%d" % (M, g, s))
    for s in (1, 3, 8):
        full_check(t, _lib.FLAG_SWIGLU | _lib.FLAG_FORCE_GEMV | _lib.FLAG_SPLIT(s),
                   what="gemv_tc swiglu M=%d split=%d" % (M, s))


@pytest.mark.parametrize("M", [1, 3, 8, 20])
def test_smallm_bf16_multiply_path(M):
    """The few-row kernels default to f16 operands; the warp-MMA kernel's
    bf16 path is kept as an option and must meet the same bound."""
    t = make_linear(M, 384, 2048, seed=1200 + M)
    full_check(t, _lib.FLAG_BF16_MMA, what="bf16-mma M=%d" % M)
    full_check(t, 0, what="f16 M=%d" % M)
    full_check(t, _lib.FLAG_FORCE_GEMV, what="gemv_tc M=%d" % M)


def _wide_range_inputs(M, seed):
    """Activation rows that stress the f16 path's per-row power-of-two
    scaling: magnitudes spread over 2^-40..2^20 in one row, a row whose
    large values arrive only in the last k stages (the running maximum
    grows mid-row), a row scaled by 2^-60, and a sparse row of values near
    3e5 (beyond f16's range before scaling)."""
    rng = np.random.default_rng(seed)
    N, K = 256, 2048
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0] = np.sign(rng.standard_normal(K)) * np.exp2(rng.uniform(-40, 20, K))
    if M > 1:
        x[1] *= np.float32(1e-3)
        x[1, -300:] = rng.standard_normal(300).astype(np.float32) * np.float32(4e4)
    if M > 2:
        x[2] *= np.float32(2.0 ** -60)
    if M > 3:
        x[3] = 0.0
        idx = rng.choice(K, 12, replace=False)
        x[3, idx] = rng.uniform(2.5e5, 3.5e5, 12).astype(np.float32) * np.sign(
            rng.standard_normal(12)).astype(np.float32)
    wp = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    ws = rng.integers(0x20, 0x51, size=(N, K // 16), dtype=np.uint8)
    from nvfp4_block_scaled_linear_gb300.inputs import GLOBAL_SCALE, f32_to_bf16_bits
    return LinearInputs(f32_to_bf16_bits(x), wp, ws, GLOBAL_SCALE)


@pytest.mark.parametrize("M,flags", [(4, 0), (8, 0), (12, 0), (32, 0), (4, _lib.FLAG_BF16_MMA),
                                     (40, 0), (4, _lib.FLAG_FORCE_GEMV | _lib.FLAG_SPLIT(1)),
                                     (4, _lib.FLAG_FORCE_GEMV | _lib.FLAG_SPLIT(8)),
                                     (8, _lib.FLAG_FORCE_GEMV | _lib.FLAG_SPLIT(3)),
                                     (32, _lib.FLAG_FORCE_GEMV),
                                     (4, _lib.FLAG_FORCE_SMALLM),
                                     (4, _lib.FLAG_FORCE_SMALLM | _lib.FLAG_SPLIT(8)),
                                     (8, _lib.FLAG_FORCE_SMALLM | _lib.FLAG_SPLIT(3)),
                                     (12, _lib.FLAG_FORCE_SMALLM),
                                     (4, GEMV_BF16), (32, GEMV_BF16 | _lib.FLAG_GROUPS(2)),
                                     (24, GEMV_BF16 | _lib.FLAG_SPLIT(3))])
def test_wide_dynamic_range_rows(M, flags):
    t = _wide_range_inputs(M, seed=1300 + M)
    y64, a = _oracle(t)
    _check_against(t, y64, a, flags, "wide-range M=%d flags=%d" % (M, flags))
    # the row scaled by 2^-60 is held to the relative bound alone (the
    # absolute 1e-6 would make its check vacuous)
    y32 = run(t, flags | _lib.FLAG_F32_OUT).cpu().numpy().astype(np.float64)
    err = np.abs(y32[2] - y64[2])
    assert np.all(err <= 1e-4 * a[2]), float(np.max(err / a[2]))
    assert np.all(np.abs(y64[2]) > 0) and np.all(np.abs(y32[2]) < 2.0 ** -40)


def _out_of_window_inputs(M, seed, N=256, K=2048):
    """Rows whose range exceeds the f16 window (2^31 below the running
    maximum): row 0 = [2^40, 1, 1, ...] (huge value first), row 1 =
    [1, ..., 1, 2^40] (huge value last, so the running maximum drops the
    scale only in the last stage), row 2 an ordinary N(0, 1) row, row 3 =
    [-2^100, N(0,1) * 2^60 ...], then the pattern again with other signs.
    Every weight row has code 0 at k = 0 and k = K - 1, so the huge values
    add nothing to y or to A = sum |x w|: the small values are all of the
    result and all of its tolerance."""
    rng = np.random.default_rng(seed)
    wp = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    wp[:, 0] &= 0xF0                  # k = 0: low nibble, code +0
    wp[:, -1] &= 0x0F                 # k = K - 1: high nibble, code +0
    ws = rng.integers(0x20, 0x51, size=(N, K // 16), dtype=np.uint8)
    x = np.ones((M, K), np.float32)
    for m in range(M):
        kind, sign = m % 4, np.float32(1.0 if (m // 4) % 2 == 0 else -1.0)
        if kind == 0:
            x[m] = sign
            x[m, 0] = np.float32(2.0 ** 40)
        elif kind == 1:
            x[m] = -sign
            x[m, -1] = np.float32(2.0 ** 40) * sign
        elif kind == 2:
            x[m] = rng.standard_normal(K).astype(np.float32)
        else:
            x[m] = rng.standard_normal(K).astype(np.float32) * np.float32(2.0 ** 60)
            x[m, 0] = np.float32(-2.0 ** 100) * sign
    from nvfp4_block_scaled_linear_gb300.inputs import GLOBAL_SCALE, f32_to_bf16_bits
    return LinearInputs(f32_to_bf16_bits(x), wp, ws, GLOBAL_SCALE)


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8])
@pytest.mark.parametrize("flags", [0, _lib.FLAG_FORCE_SMALLM | _lib.FLAG_SPLIT(3)],
                         ids=["default", "split3"])
def test_rows_beyond_the_f16_window_are_exact(M, flags):
    """The default M <= 8 kernel multiplies in f16 with a per-row power of
    two; a stage of a row holding values more than 2^31 below the row's
    running maximum is multiplied in bf16 instead.  Held to the fp32 and
    bf16 bounds; with a forced split, each row also equals the single-row
    call on that row bit for bit (the fallback is decided per row)."""
    t = _out_of_window_inputs(M, seed=1350 + M)
    assert _lib.kernel_for(M, t.N, t.K, flags) == _lib.KERNEL_SMALLM
    y64, a = _oracle(t)
    _check_against(t, y64, a, flags, "out-of-window M=%d flags=%d" % (M, flags))
    if flags & _lib.FLAG_SPLIT(31):          # the same split forced on both calls
        y = bf16_bits(run(t, flags))
        for i in range(M):
            ti = LinearInputs(t.x_bits[i:i + 1].copy(), t.w_packed, t.w_scale, t.global_scale)
            assert np.array_equal(bf16_bits(run(ti, flags))[0], y[i]), "row %d" % i


@pytest.mark.parametrize("M,flags", [(1, 0), (6, 0), (6, _lib.FLAG_BF16_MMA), (20, 0),
                                     (1, _lib.FLAG_FORCE_SMALLM), (6, _lib.FLAG_FORCE_SMALLM),
                                     (1, _lib.FLAG_FORCE_GEMV), (6, _lib.FLAG_FORCE_GEMV),
                                     (6, _lib.FLAG_FORCE_TCGEMM), (50, 0),
                                     (1, GEMV_BF16), (6, GEMV_BF16),
                                     (20, GEMV_BF16 | _lib.FLAG_GROUPS(2))])
def test_non_finite_values_propagate(M, flags):
    """An inf or NaN activation, or a NaN block scale (e4m3 S.1111.111),
    gives the non-finite outputs the exact sum gives (IEEE: inf * 0 = NaN,
    inf - inf = NaN); every other output is unaffected."""
    t = make_linear(M, 256, 1024, seed=1400 + M)
    x = t.x_bits.copy()
    if M > 1:
        x[0, 37] = 0x7F80                     # +inf (a whole output row non-finite)
    if M > 2:
        x[2, 600] = 0xFF80                    # -inf
        x[M - 1, 5] = 0x7FC0                  # NaN
    ws = t.w_scale.copy()
    ws[17, 3] = 0x7F                          # NaN scale: row 17, k in [48, 64)
    ws[200, 60] = 0xFF
    t = LinearInputs(x, t.w_packed, ws, t.global_scale)
    y64, a = _oracle(t)
    y32 = run(t, flags | _lib.FLAG_F32_OUT).cpu().numpy().astype(np.float64)
    fin = np.isfinite(y64)
    assert (~fin).any() and fin.any()
    assert np.array_equal(np.isnan(y32), np.isnan(y64))
    assert np.array_equal(y32[np.isinf(y64)], y64[np.isinf(y64)])
    check_f32(y32[fin], y64[fin], a[fin], "non-finite M=%d" % M)
    ybf = bf16_bits(run(t, flags))
    check_bf16(ybf[fin], y64[fin], a[fin], oracle.to_bf16_bits(y64[fin]), "non-finite bf16")
    vb = oracle.to_bf16_bits(y64)
    assert np.array_equal(ybf[np.isinf(y64)], vb[np.isinf(y64)])
    assert np.all((ybf[np.isnan(y64)] & 0x7FFF) > 0x7F80)


@pytest.mark.parametrize("M,kflag", [(1, 0), (7, _lib.FLAG_FORCE_SMALLM), (12, 0), (24, 0),
                                     (7, _lib.FLAG_FORCE_GEMV), (64, 0), (300, 0),
                                     (7, GEMV_BF16), (24, GEMV_BF16 | _lib.FLAG_GROUPS(2))])
def test_swiglu_separate_gate_up_global_scales(M, kflag):
    """Gate rows with one global scale, up rows with another: equal to the
    oracle's two half-linears combined by SwiGLU."""
    N, K = 512, 1024
    t = make_linear(M, N, K, seed=1800 + M)
    gs_gate, gs_up = np.float32(448.0 / 6.0), np.float32(448.0 / 1.5)
    H = N // 2
    g64, ga = oracle.linear_f64(t.x_bits, t.w_packed[:H], t.w_scale[:H], gs_gate)
    u64, ua = oracle.linear_f64(t.x_bits, t.w_packed[H:], t.w_scale[H:], gs_up)
    y64 = np.concatenate([g64, u64], 1)
    a = np.concatenate([ga, ua], 1)
    out64 = oracle.swiglu_f64(y64)
    x, wp, ws = to_dev(t)
    y32 = _lib.linear_swiglu_gs(x, wp, ws, gs_gate, gs_up, kflag | _lib.FLAG_F32_OUT)
    ybf = _lib.linear_swiglu_gs(x, wp, ws, gs_gate, gs_up, kflag)
    torch.cuda.synchronize()
    check_swiglu_f32(y32.cpu().numpy(), y64, a, out64, "swiglu_gs M=%d" % M)
    check_swiglu_bf16(bf16_bits(ybf), y64, a, out64, oracle.to_bf16_bits(out64),
                      "swiglu_gs M=%d" % M)
    # equal scales: the same bits as the one-scale entry point
    same = _lib.linear_swiglu_gs(x, wp, ws, t.global_scale, t.global_scale, kflag)
    ref = _lib.linear_ex(x, wp, ws, float(t.global_scale), _lib.FLAG_SWIGLU | kflag)
    torch.cuda.synchronize()
    assert torch.equal(same.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("M,kflag", [(1, 0), (7, 0), (7, _lib.FLAG_FORCE_GEMV), (12, 0),
                                     (32, 0), (100, 0), (7, GEMV_BF16),
                                     (32, GEMV_BF16 | _lib.FLAG_GROUPS(4))])
def test_segmented_qkv_global_scales(M, kflag):
    """q, k and v stacked into one launch, each with its own global scale:
    equal to three separate oracle linears side by side (segments of 384,
    128 and 128 rows: boundaries inside CTAs and tiles)."""
    K = 1024
    rows = [384, 128, 128]
    gss = [np.float32(448.0 / 6.0), np.float32(448.0 / 2.0), np.float32(448.0 / 11.0)]
    t = make_linear(M, sum(rows), K, seed=1900 + M)
    ys, As = [], []
    r0 = 0
    for r, g in zip(rows, gss):
        y64, a = oracle.linear_f64(t.x_bits, t.w_packed[r0:r0 + r], t.w_scale[r0:r0 + r], g)
        ys.append(y64)
        As.append(a)
        r0 += r
    y64, a = np.concatenate(ys, 1), np.concatenate(As, 1)
    x, wp, ws = to_dev(t)
    y32 = _lib.linear_segmented(x, wp, ws, gss, rows, kflag | _lib.FLAG_F32_OUT)
    ybf = _lib.linear_segmented(x, wp, ws, gss, rows, kflag)
    torch.cuda.synchronize()
    check_f32(y32.cpu().numpy(), y64, a, "segmented M=%d" % M)
    check_bf16(bf16_bits(ybf), y64, a, oracle.to_bf16_bits(y64), "segmented M=%d" % M)


# ------------------------------------------------------------------ exactness
def _exhaustive_products():
    """Rows n = every e4m3 scale byte; inputs k = 0..15 carry codes 0..15;
    x row m is one-hot at k = m, so y[m, n] = code(m) * scale(n) / gs: one
    exact product per output, which must match bit for bit."""
    N, K, M = 256, 256, 16
    wp = np.zeros((N, K // 2), np.uint8)
    codes = np.arange(K) % 16
    wp[:] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    ws = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 16, axis=1)
    x = np.zeros((M, K), np.uint16)
    x[np.arange(M), np.arange(M)] = 0x3F80
    return LinearInputs(x, wp, ws, np.float32(1.0))


@pytest.mark.parametrize("flags", [_lib.FLAG_FORCE_SMALLM, _lib.FLAG_FORCE_TCGEMM,
                                   _lib.FLAG_FORCE_GEMV, GEMV_BF16,
                                   GEMV_BF16 | _lib.FLAG_GROUPS(2)])
def test_every_code_times_every_scale_is_exact(flags):
    t = _exhaustive_products()
    y64, _ = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    y32 = run(t, flags | _lib.FLAG_F32_OUT).cpu().numpy().astype(np.float64)
    nan = np.isnan(y64)
    assert np.array_equal(np.isnan(y32), nan)
    assert np.array_equal(y32[~nan], y64[~nan])


@pytest.mark.parametrize("M,flags", [(5, 0), (12, 0), (30, 0), (70, 0),
                                     (5, _lib.FLAG_FORCE_TCGEMM), (5, _lib.FLAG_FORCE_GEMV),
                                     (5, GEMV_BF16), (30, GEMV_BF16 | _lib.FLAG_GROUPS(2))])
def test_exact_integer_inputs_are_bit_exact(M, flags):
    # small-integer activations, power-of-two scales, global scale 1: every
    # partial sum is an exactly representable fp32 number, so the result is
    # exact whatever the summation order
    rng = np.random.default_rng(9)
    N, K = 256, 1024
    xs = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    x = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wp = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    ws = rng.choice(np.array([0x30, 0x38, 0x40, 0x48], np.uint8), size=(N, K // 16))
    t = LinearInputs(x, wp, ws, np.float32(1.0))
    y64, _ = oracle.linear_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale)
    y32 = run(t, flags | _lib.FLAG_F32_OUT).cpu().numpy().astype(np.float64)
    assert np.array_equal(y32, y64)


@pytest.mark.parametrize("M,flags", [(3, 0), (3, _lib.FLAG_FORCE_GEMV), (50, 0), (3, GEMV_BF16)])
def test_sign_flip_negates_exactly(M, flags):
    t = make_linear(M, 256, 512, seed=600 + M)
    y = run(t, _lib.FLAG_F32_OUT | flags).cpu().numpy()
    flipped = LinearInputs(t.x_bits, t.w_packed ^ np.uint8(0x88), t.w_scale, t.global_scale)
    y_neg = run(flipped, _lib.FLAG_F32_OUT | flags).cpu().numpy()
    assert np.array_equal(y_neg, -y)


@pytest.mark.parametrize("M,flags", [(1, 0), (1, _lib.FLAG_FORCE_GEMV), (40, 0), (1, GEMV_BF16),
                                     (32, GEMV_BF16)])
def test_nibble_order(M, flags):
    K, N = 256, 128
    x = np.zeros((M, K), np.uint16)
    x[:, 0] = 0x3F80          # 1.0 at k = 0
    x[:, 1] = 0x4000          # 2.0 at k = 1
    ws = np.full((N, K // 16), 0x38, np.uint8)
    lo = np.zeros((N, K // 2), np.uint8)
    lo[:, 0] = 0x07           # 6.0 at k = 0 (low nibble)
    hi = np.zeros((N, K // 2), np.uint8)
    hi[:, 0] = 0x70           # 6.0 at k = 1 (high nibble)
    y_lo = run(LinearInputs(x, lo, ws, np.float32(1.0)), _lib.FLAG_F32_OUT | flags).cpu().numpy()
    y_hi = run(LinearInputs(x, hi, ws, np.float32(1.0)), _lib.FLAG_F32_OUT | flags).cpu().numpy()
    assert np.all(y_lo == 6.0) and np.all(y_hi == 12.0)


@pytest.mark.parametrize("kflag", FEW_ROW)
def test_row_batch_invariance_verify_vs_decode(kflag):
    # greedy decode (M = 1) and speculative verify (M = 7) see the same rows:
    # each verify row must equal the single-row call on that row, bit for bit
    # (same k split forced on both)
    t = make_linear(7, 1024, 2048, seed=700)
    fl = kflag | _lib.FLAG_SPLIT(4)
    y7 = bf16_bits(run(t, fl))
    for i in range(7):
        ti = LinearInputs(t.x_bits[i:i + 1].copy(), t.w_packed, t.w_scale, t.global_scale)
        assert np.array_equal(bf16_bits(run(ti, fl))[0], y7[i]), "row %d" % i


# ------------------------------------------------------------------ edges
def test_empty_m_is_a_no_op():
    x = torch.zeros((0, 512), dtype=torch.bfloat16, device=DEV)
    wp = torch.zeros((256, 256), dtype=torch.uint8, device=DEV)
    ws = torch.zeros((256, 32), dtype=torch.uint8, device=DEV)
    y = _lib.linear(x, wp, ws, 1.0)
    assert tuple(y.shape) == (0, 256)


def test_errors_on_device_buffers():
    x = torch.zeros((1, 512 + 8), dtype=torch.bfloat16, device=DEV)
    wp = torch.zeros((256, 256), dtype=torch.uint8, device=DEV)
    ws = torch.zeros((256, 32), dtype=torch.uint8, device=DEV)
    lib = _lib.library()
    y = torch.empty((1, 256), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    import ctypes
    # x starting 2 bytes into an allocation: misaligned
    st = lib.nvfp4_linear(x.data_ptr() + 2, wp.data_ptr(), ws.data_ptr(), ctypes.c_float(1.0),
                          y.data_ptr(), 1, 256, 512, ctypes.c_void_p(s))
    assert st == -2
    st = lib.nvfp4_linear(x.data_ptr(), wp.data_ptr(), ws.data_ptr(), ctypes.c_float(1.0),
                          y.data_ptr(), 1, 256, 520, ctypes.c_void_p(s))
    assert st == -3


@pytest.mark.parametrize("M", [3, 20, 45])
def test_output_guard_rows_untouched(M):
    t = make_linear(M, 256, 512, seed=800 + M)
    x, wp, ws = to_dev(t)
    big = torch.full((M + 2, 256), 12345.0, dtype=torch.float32, device=DEV)
    out = big[1:M + 1]
    _lib.linear_f32(x, wp, ws, float(t.global_scale), out=out)
    torch.cuda.synchronize()
    assert torch.all(big[0] == 12345.0) and torch.all(big[M + 1] == 12345.0)


def test_repeated_calls_are_deterministic():
    t = make_linear(7, 512, 4096, seed=900)
    a = bf16_bits(run(t))
    for _ in range(3):
        assert np.array_equal(bf16_bits(run(t)), a)


def test_concurrent_calls_from_two_threads_on_two_streams():
    """Every call shares the library's host state (device set-up, plan and
    descriptor caches): two threads calling at once, each on its own
    stream, with shapes that take different kernels and plans, get the
    outputs of calls made one at a time, bit for bit."""
    import threading
    cases = [(make_linear(1, 1024, 2048, seed=3000), 0),
             (make_linear(20, 768, 1024, seed=3001), 0),
             (make_linear(12, 512, 2048, seed=3002), GEMV_BF16 | _lib.FLAG_SPLIT(2)),
             (make_linear(5, 640, 1024, seed=3003), _lib.FLAG_SWIGLU)]
    refs = [bf16_bits(run(t, fl)) for t, fl in cases]
    failures = []

    def worker(items):
        s = torch.cuda.Stream()
        dev = [(to_dev(t), t, fl, ref) for (t, fl), ref in items]
        for i in range(40):
            for (x, wp, ws), t, fl, ref in dev:
                y = _lib.linear_ex(x, wp, ws, float(t.global_scale), fl, stream=s)
                s.synchronize()
                if not np.array_equal(bf16_bits(y), ref):
                    failures.append((t.M, fl, i))
                    return

    pairs = list(zip(cases, refs))
    threads = [threading.Thread(target=worker, args=(pairs[k::2],)) for k in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not failures, failures


@pytest.mark.parametrize("M,flags,pinned", [
    (1, 0, True), (7, _lib.FLAG_SWIGLU, True), (20, _lib.FLAG_F32_OUT, False),
    (20, _lib.FLAG_F32_OUT, True), (12, _lib.FLAG_SWIGLU | _lib.FLAG_F32_OUT, True),
    (20, _lib.FLAG_FORCE_GEMV | _lib.FLAG_BF16_MMA, True), (12, _lib.FLAG_FORCE_GEMV, True),
    (9, _lib.FLAG_FORCE_GEMV | _lib.FLAG_BF16_MMA | _lib.FLAG_SWIGLU | _lib.FLAG_F32_OUT |
     _lib.FLAG_SPLIT(1), True),
    (32, _lib.FLAG_FORCE_GEMV | _lib.FLAG_BF16_MMA | _lib.FLAG_SWIGLU | _lib.FLAG_SPLIT(3), True),
    (40, 0, True)])
def test_host_buffer_call_equals_device_call(M, flags, pinned):
    """nvfp4_linear_host (activations and result in host memory, page-locked
    or not) gives the device call's output bit for bit: with page-locked
    buffers each few-row kernel (the warp-MMA kernel in f16 and bf16, both
    tcgen05 few-row kernels) also writes the result into the host buffer from
    its epilogue, and at M > 32 the output staging kernel moves it."""
    t = make_linear(M, 512, 1024, seed=3100 + M)
    x, wp, ws = to_dev(t)
    ref = _lib.linear_ex(x, wp, ws, float(t.global_scale), flags).cpu()
    hx = x.cpu()
    hy = torch.empty(ref.shape, dtype=ref.dtype)
    if pinned:
        hx, hy = hx.pin_memory(), hy.pin_memory()
    dx = torch.empty_like(x)
    dy = torch.empty(ref.shape, dtype=ref.dtype, device=x.device)
    s = torch.cuda.Stream()
    _lib.linear_host(hx, dx, wp, ws, float(t.global_scale), dy, hy, flags, stream=s)
    s.synchronize()
    assert torch.equal(hy.view(torch.int16) if hy.dtype == torch.bfloat16 else hy,
                       ref.view(torch.int16) if ref.dtype == torch.bfloat16 else ref)
    assert torch.equal(dx.cpu().view(torch.int16), x.cpu().view(torch.int16))


@pytest.mark.parametrize("M", [1, 40])
def test_host_buffer_calls_chained_on_one_stream(M):
    """Back-to-back nvfp4_linear_host calls on one stream sharing x_dev and
    y_dev, each with its own page-locked input and output (the zero-copy
    path, whose transfers are kernels chained by programmatic dependent
    launch): every call reads its own activations and returns its own
    result, bit for bit the device call's."""
    n = 4
    ts = [make_linear(M, 512, 1024, seed=3200 + 10 * M + i) for i in range(n)]
    x0, wp, ws = to_dev(ts[0])
    gs = float(ts[0].global_scale)
    refs = []
    hxs, hys = [], []
    for t in ts:
        x = torch.from_numpy(t.x_bits.view(np.int16)).view(torch.bfloat16)
        refs.append(_lib.linear_ex(x.to(DEV), wp, ws, gs, 0).cpu())
        hxs.append(x.clone().pin_memory())
        hys.append(torch.full((M, 512), float("nan"), dtype=torch.bfloat16).pin_memory())
    dx = torch.empty_like(x0)
    dy = torch.empty((M, 512), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    for rep in range(3):
        for i in range(n):
            _lib.linear_host(hxs[i], dx, wp, ws, gs, dy, hys[i], 0, stream=s)
    s.synchronize()
    for i in range(n):
        assert torch.equal(hys[i].view(torch.int16), refs[i].view(torch.int16)), "call %d" % i


def test_host_buffers_off_16_byte_alignment_take_the_copies():
    """Page-locked buffers 2 bytes into their allocation cannot take the
    16-byte staging kernels: the call copies instead, same result."""
    M, N, K = 3, 512, 1024
    t = make_linear(M, N, K, seed=3300)
    x, wp, ws = to_dev(t)
    ref = _lib.linear_ex(x, wp, ws, float(t.global_scale), 0).cpu()
    big_x = torch.empty(M * K + 8, dtype=torch.bfloat16).pin_memory()
    big_y = torch.empty(M * N + 8, dtype=torch.bfloat16).pin_memory()
    hx = big_x[1:1 + M * K].view(M, K)
    hy = big_y[1:1 + M * N].view(M, N)
    hx.copy_(x.cpu())
    dx = torch.empty_like(x)
    dy = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    _lib.linear_host(hx, dx, wp, ws, float(t.global_scale), dy, hy, 0, stream=s)
    s.synchronize()
    assert torch.equal(hy.view(torch.int16), ref.view(torch.int16))


def test_cuda_graph_capture_and_replay():
    """Calls captured into a CUDA graph (both kernels, SwiGLU and plain)
    give on replay what the same calls give eagerly, bit for bit, also after
    the inputs are overwritten in place between replays."""
    shapes = [(1, 512, 1024, 0), (7, 384, 2048, 0), (32, 512, 1024, _lib.FLAG_SWIGLU),
              (100, 256, 1024, 0)]
    ts = [make_linear(M, N, K, seed=1500 + i) for i, (M, N, K, _) in enumerate(shapes)]
    devs = [to_dev(t) for t in ts]
    outs = [torch.empty((M, N // 2 if f else N), dtype=torch.bfloat16, device=DEV)
            for (M, N, K, f) in shapes]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for (x, wp, ws), t, o, (_, _, _, f) in zip(devs, ts, outs, shapes):   # warm-up
            _lib.linear_ex(x, wp, ws, float(t.global_scale), f, out=o, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        for (x, wp, ws), t, o, (_, _, _, f) in zip(devs, ts, outs, shapes):
            _lib.linear_ex(x, wp, ws, float(t.global_scale), f, out=o, stream=st)
    for rep in range(2):
        if rep:
            for (x, _, _) in devs:
                x.mul_(-2.0)
        for o in outs:
            o.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        for (x, wp, ws), t, o, (_, _, _, f) in zip(devs, ts, outs, shapes):
            ref = _lib.linear_ex(x, wp, ws, float(t.global_scale), f)
            torch.cuda.synchronize()
            assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    # and the eager result is the oracle's
    t0 = LinearInputs(devs[1][0].cpu().view(torch.int16).numpy().view(np.uint16),
                      ts[1].w_packed, ts[1].w_scale, ts[1].global_scale)
    y64, a = _oracle(t0)
    check_bf16(bf16_bits(outs[1]), y64, a, oracle.to_bf16_bits(y64), "graph replay")


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_chained_calls_read_the_previous_output(M):
    """y1 = L1(x); y2 = L2(y1); y3 = L3(y2) back to back on one stream: each
    call's activations are the previous call's output, written by the kernel
    just before it (the calls overlap their weight prefetch with it).  Equal,
    bit for bit, to the same calls separated by synchronisation."""
    K0 = 1024
    dims = [(512, K0), (768, 512), (256, 768)]
    rng = np.random.default_rng(1600 + M)
    layers = []
    for i, (N, K) in enumerate(dims):
        t = draw_linear(rng, 1, N, K)
        layers.append((torch.from_numpy(t.w_packed).to(DEV),
                       torch.from_numpy(t.w_scale).to(DEV), float(t.global_scale)))
    x = torch.from_numpy(make_linear(M, 128, K0, seed=1700 + M).x_bits.view(np.int16)).view(
        torch.bfloat16).to(DEV)
    for _ in range(3):
        h = x
        for wp, ws, gs in layers:
            h = _lib.linear(h, wp, ws, gs)
        chained = h.clone()
        h = x
        for wp, ws, gs in layers:
            h = _lib.linear(h, wp, ws, gs)
            torch.cuda.synchronize()
        assert torch.equal(chained.view(torch.int16), h.view(torch.int16))


# ------------------------------------------------------------------ full size
# The benchmarked configurations, in the benchmark's launch configuration
# (the same entry points and plans).  tiny, decode_gate_up, verify_down and
# the four linears of layer_m32 are checked at every output; prefill (with and
# without SwiGLU) at every output of the rows where its tiles have edges or
# its values are extreme, and at every output column on a weight-tile edge
# for a row sample.  The strict 1-ulp fail counts (outputs that pass only
# through the near-zero rule) are bounded here and logged when
# NVFP4_PARITY_LOG names a file.

def _strict_bound(n):
    # near-zero outputs (|y| well below A / 100) are a few percent of a
    # Gaussian sum; the ones the fp32 summation moves by over an ulp are
    # fewer
    return max(8, n // 100)


@pytest.mark.parametrize("name", ["tiny", "decode_gate_up", "verify_down", "layer_m32"])
def test_full_size_workloads_every_output(name):
    w = WORKLOADS[name]
    for t in w.draw():
        x, wp, ws = to_dev(t)
        y32 = _lib.linear_ex(x, wp, ws, float(t.global_scale), _lib.FLAG_F32_OUT)
        ybf = _lib.linear_ex(x, wp, ws, float(t.global_scale), 0)
        torch.cuda.synchronize()
        y64, a = _oracle(t)
        what = "%s/%s" % (name, t.name)
        ratio = check_f32(y32.cpu().numpy(), y64, a, what)
        strict, _ = check_bf16(bf16_bits(ybf), y64, a, oracle.to_bf16_bits(y64), what)
        record(what, outputs=int(y64.size), strict_fail=strict, worst_f32_over_tol=ratio,
               kernel=_lib.choose_plan(t.M, t.N, t.K))
        assert strict <= _strict_bound(y64.size), (what, strict)
        del x, wp, ws, y32, ybf
        torch.cuda.empty_cache()


_PREFILL_CACHE = {}


def _prefill_reference():
    """Inputs of the prefill configuration, the checked rows and columns, and
    the oracle's fp64 results there (shared by the plain and SwiGLU tests)."""
    if "ref" in _PREFILL_CACHE:
        return _PREFILL_CACHE["ref"]
    t = WORKLOADS["prefill"].draw()[0]
    M, N = t.M, t.N
    tile_x = 256                      # activation rows per tensor-core tile
    edges = [r for j in range(1, M // tile_x) for r in (tile_x * j - 1, tile_x * j)]
    rows = np.unique(np.concatenate([[0, M - 1], t.big_rows, edges])).astype(np.int64)
    y64, a = oracle.linear_f64(t.x_bits[rows], t.w_packed, t.w_scale, t.global_scale)
    rng = np.random.default_rng(4321)
    sample = np.sort(rng.choice(M, size=64, replace=False)).astype(np.int64)
    ref = dict(t=t, rows=rows, y64=y64, a=a, sample=sample)
    _PREFILL_CACHE["ref"] = ref
    return ref


def _col_edges(n_out, tile):
    return np.array([c for j in range(1, n_out // tile) for c in (tile * j - 1, tile * j)]
                    + [0, n_out - 1], np.int64)


@pytest.mark.parametrize("swiglu", [False, True], ids=["prefill", "prefill_swiglu"])
def test_prefill_rows_and_tile_edges(swiglu):
    ref = _prefill_reference()
    t, rows, y64, a, sample = ref["t"], ref["rows"], ref["y64"], ref["a"], ref["sample"]
    name = "prefill_swiglu" if swiglu else "prefill"
    assert len(t.big_rows) == 82
    x, wp, ws = to_dev(t)
    flags = _lib.FLAG_SWIGLU if swiglu else 0
    y32 = _lib.linear_ex(x, wp, ws, float(t.global_scale), flags | _lib.FLAG_F32_OUT)
    ybf = _lib.linear_ex(x, wp, ws, float(t.global_scale), flags)
    torch.cuda.synchronize()
    ridx = torch.from_numpy(rows).to(DEV)
    r32 = y32.index_select(0, ridx).cpu().numpy()
    rbf = bf16_bits(ybf.index_select(0, ridx))
    # whole output columns on the edges of the weight tiles (128 weight rows;
    # 64 gate + 64 up rows, i.e. 64 outputs, with SwiGLU), for a row sample
    n_out = t.N // 2 if swiglu else t.N
    cols = _col_edges(n_out, 64 if swiglu else 128)
    mi = np.repeat(sample, cols.size)
    ni = np.tile(cols, sample.size)
    c32 = y32[torch.from_numpy(mi).to(DEV), torch.from_numpy(ni).to(DEV)].cpu().numpy()
    cbf = bf16_bits(ybf[torch.from_numpy(mi).to(DEV), torch.from_numpy(ni).to(DEV)])
    if swiglu:
        H = t.N // 2
        out64 = oracle.swiglu_f64(y64)
        check_swiglu_f32(r32, y64, a, out64, name + " rows")
        strict = check_swiglu_bf16(rbf, y64, a, out64, oracle.to_bf16_bits(out64), name + " rows")
        g64, ga = oracle.linear_points_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale,
                                           mi, ni)
        u64, ua = oracle.linear_points_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale,
                                           mi, ni + H)
        cy, ca = np.stack([g64, u64], 1), np.stack([ga, ua], 1)
        cout = oracle.swiglu_f64(cy)
        check_swiglu_f32(c32[:, None], cy, ca, cout, name + " columns")
        strict_c = check_swiglu_bf16(cbf[:, None], cy, ca, cout, oracle.to_bf16_bits(cout),
                                     name + " columns")
    else:
        check_f32(r32, y64, a, name + " rows")
        strict, _ = check_bf16(rbf, y64, a, oracle.to_bf16_bits(y64), name + " rows")
        cy, ca = oracle.linear_points_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale,
                                          mi, ni)
        check_f32(c32, cy, ca, name + " columns")
        strict_c, _ = check_bf16(cbf, cy, ca, oracle.to_bf16_bits(cy), name + " columns")
    n_checked = rbf.size + cbf.size
    record(name, outputs=int(n_checked), rows=int(rows.size), columns=int(cols.size),
           sample_rows=int(sample.size), strict_fail=int(strict + strict_c))
    assert strict + strict_c <= _strict_bound(n_checked), (name, strict, strict_c)


@pytest.mark.parametrize("M,swiglu", [(20, False), (32, True)])
def test_bf16_few_row_kernel_is_the_default_on_large_layers(M, swiglu):
    """M = 17..32 on a weight matrix of N * K = 2^26 runs the bf16 tcgen05
    few-row kernel by default (two lane groups: 128 row blocks fill the
    SMs); sampled outputs against the oracle."""
    N, K = 16384, 4096
    flags = _lib.FLAG_SWIGLU if swiglu else 0
    assert _lib.kernel_for(M, N, K, flags) == _lib.KERNEL_GEMV_BF16
    t = make_linear(M, N, K, seed=2100 + M)
    x, wp, ws = to_dev(t)
    y32 = _lib.linear_ex(x, wp, ws, float(t.global_scale), flags | _lib.FLAG_F32_OUT)
    ybf = _lib.linear_ex(x, wp, ws, float(t.global_scale), flags)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2200 + M)
    n_out = y32.shape[1]
    mi = rng.integers(0, M, size=800)
    ni = rng.integers(0, n_out, size=800)
    y32s = y32.cpu().numpy()[mi, ni].astype(np.float64)
    ybs = bf16_bits(ybf)[mi, ni]
    if swiglu:
        H = N // 2
        g64, ga = oracle.linear_points_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale, mi, ni)
        u64, ua = oracle.linear_points_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale, mi,
                                           ni + H)
        y64, a = np.stack([g64, u64], 1), np.stack([ga, ua], 1)
        out64 = oracle.swiglu_f64(y64)[:, 0]
        check_swiglu_f32(y32s[:, None], y64, a, out64[:, None], "bf16 default swiglu")
        check_swiglu_bf16(ybs[:, None], y64, a, out64[:, None],
                          oracle.to_bf16_bits(out64)[:, None], "bf16 default swiglu")
    else:
        y64, a = oracle.linear_points_f64(t.x_bits, t.w_packed, t.w_scale, t.global_scale, mi, ni)
        check_f32(y32s, y64, a, "bf16 default M=%d" % M)
        check_bf16(ybs, y64, a, oracle.to_bf16_bits(y64), "bf16 default M=%d" % M)
