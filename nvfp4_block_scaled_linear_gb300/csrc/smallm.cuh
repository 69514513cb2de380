// smallm.cuh -- NVFP4 W4A16 linear for few activation rows (M <= 32):
// decode (M = 1), speculative verify (M = K+1, FlashRT docs section 3) and
// small continuous batches.  At these sizes the layer is bound by streaming
// the packed weights and scales from HBM once; every design choice below is
// about keeping that stream at full rate.
//
//  * One CTA owns G groups of 16 weight rows (G = 1..8, chosen per call) and
//    a contiguous range of k.  A producer warp streams 256-k stages (packed
//    weights, block scales, activations) into a shared-memory ring with TMA;
//    an L2 evict-first hint keeps the once-read weights from displacing the
//    activations.  The weights of the first ring-full are requested before
//    the kernel waits on the preceding kernel in the stream (programmatic
//    dependent launch); the activations only after.
//  * Eight consumer warps: warp (kq, rp) takes the 64-k quarter kq of every
//    stage for the row groups rp, rp+2, rp+4, rp+6 of the CTA.  The weights
//    are dequantised in registers straight into the A fragments of the
//    register-fed m16n8k16 warp MMA (weights as the 16-row operand,
//    activations as the 8-wide one), so dequantised weights never touch
//    shared memory.  (The tcgen05 MMA reads both of its operands from shared
//    memory or TMEM; at N = 8..32 that round trip would cost more shared-memory
//    bandwidth than the weight stream itself.)
//  * bf16 path (any M <= 32): the dequantiser's (k, k+4) pairing is matched
//    by building the activation fragments with the same k permutation, so
//    the dot products are unchanged.
//  * f16 path (M <= 8, the default there): the weights are dequantised by the
//    hardware e2m1 -> f16 conversion, about half the instructions of the bf16
//    bit manipulation, so the MMA runs in f16 and a converter warp brings the
//    activations to f16 each stage with a power-of-two scale per activation
//    row, taken from that row's running maximum |x|.  Every activation within
//    2^31 of its row's running maximum converts exactly, nothing overflows,
//    and the fp32 accumulators are rescaled by exact powers of two when a
//    row's maximum grows.  A row whose stage holds a nonzero value below that
//    window is flagged by its converter: the consumers get zeros for it, and
//    the converter itself multiplies that row's stage in bf16 (the bf16
//    path's exact weights, the activations as given) into the CTA's partial
//    sums, so the product is exact for every finite bf16 row while the
//    consumers' loop, and every unflagged row, are exactly those of the plain
//    f16 path.
//  * Split-K: CTAs that share rows but not k form one thread-block cluster.
//    Partials are reduced warp -> CTA in shared memory and then across the
//    cluster through distributed shared memory.  No global workspace, no
//    atomics, no spin-waits on other CTAs.
//  * The host picks G, the split and the ring depth so that the whole grid is
//    resident at once and the busiest SM carries as little work as possible.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace smallm {

constexpr int kGroupRows = 16;        // rows of one MMA row group
constexpr int kMaxGroups = 8;         // up to 128 weight rows per CTA
constexpr int kStageK = 256;          // k per pipeline stage
constexpr int kKQuarters = 4;         // 64-k quarters of a stage
constexpr int kWays = 2;              // row-group ways of the default layout
constexpr int kMaxSplit = 16;         // cluster size limit (non-portable above 8)
constexpr int kF16MaxRows = 8;        // the f16 path serves M <= 8

// Consumer warps: (k quarter, row-group way) for `ways` row-group ways.
__host__ __device__ constexpr int consumer_warps(int ways) { return kKQuarters * ways; }
// Consumers, the TMA producer and (f16 path) cv activation converters.
__host__ __device__ constexpr int threads_for(int cv, int ways = kWays) {
  return (consumer_warps(ways) + 1 + cv) * 32;
}

// Row groups one consumer warp may hold: all of its accumulators live in
// registers, so the widest activation tiles get fewer.
__host__ __device__ constexpr int max_groups(int mt) { return mt <= 2 ? 8 : 4; }
__host__ __device__ constexpr int groups_per_warp(int mt, int ways = kWays) {
  return max_groups(mt) / ways;
}

// Shared-memory layout of one launch (byte offsets from the 1024-aligned
// base), computed on the host per call.  Stage: packed weights
// [16G rows][128 B] (128B-swizzled), block scales [16G rows][16 B], then the
// activations: for M <= 8 one plain box [M rows][256 k] bf16 and (f16 path)
// its f16 copy [M rows][256 k] plus the rows' exponents; for larger M four
// 128B-swizzled boxes [MT*8 rows][64 k].
struct SmemLayout {
  int stages;
  int stage_bytes;
  int s_off;        // scales, within a stage
  int x_off;        // bf16 activations, within a stage
  int x_box_bytes;  // one activation box
  int x_tx;         // activation bytes a stage receives
  int x16_off;      // f16 activation tile, within a stage (f16 path)
  int exp_off;      // int[8] activation exponents, within a stage (f16 path)
  int part_off;     // CTA partials [MT*8][16G + kRedPad] f32
  int lut_off;      // 256 scale pairs
  int bar_off;      // full[stages], conv[stages], empty[stages], abort flag
  int total;        // dynamic shared memory to request (includes alignment slack)
};

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Partial sums in shared memory are column-major, [activation row m][weight
// row j] with a row pitch of 16G + kRedPad floats: the warps' paired stores
// (weight rows ra, ra + 1 of one column) then take the minimum two
// wavefronts, and the readers (consecutive j) none more than one.
constexpr int kRedPad = 8;
__host__ __device__ constexpr int red_pitch(int groups) {
  return groups * kGroupRows + kRedPad;
}

__host__ __device__ constexpr SmemLayout make_layout(int mt, int groups, int stages,
                                                     bool f16, int m_rows) {
  SmemLayout l{};
  const int w_bytes = groups * kGroupRows * (kStageK / 2);
  const int s_end = w_bytes + groups * kGroupRows * (kStageK / 16);
  int end = 0;
  l.stages = stages;
  l.s_off = w_bytes;
  if (mt == 1) {
    l.x_off = align_up(s_end, 128);
    l.x_box_bytes = m_rows * kStageK * 2;
    l.x_tx = l.x_box_bytes;
    l.x16_off = align_up(l.x_off + l.x_box_bytes, 128);
    l.exp_off = l.x16_off + (f16 ? m_rows * kStageK * 2 : 0);
    end = l.exp_off + (f16 ? 8 * 4 : 0);
  } else {
    l.x_off = align_up(s_end, 1024);
    l.x_box_bytes = mt * 8 * 128;
    l.x_tx = kKQuarters * l.x_box_bytes;
    end = l.x_off + kKQuarters * l.x_box_bytes;
    l.x16_off = l.exp_off = end;
  }
  l.stage_bytes = align_up(end, 1024);
  l.part_off = stages * l.stage_bytes;
  l.lut_off = l.part_off + mt * 8 * red_pitch(groups) * 4;
  l.bar_off = l.lut_off + 256 * 4;
  l.total = l.bar_off + 3 * stages * 8 + 16 + 1024;
  return l;
}

// The cross-warp reduction reuses the ring; it must fit.
__host__ __device__ constexpr bool layout_ok(const SmemLayout& l, int mt, int groups) {
  return kKQuarters * mt * 8 * red_pitch(groups) * 4 <= l.stages * l.stage_bytes;
}

struct Params {
  void* y;              // [M, N] (or [M, N/2] with swiglu), bf16 or f32
  void* y_host;         // nullptr, or the same output again in host memory mapped
                        // into the device (the host-buffer entry point)
  int64_t M, N, K;
  float out_scale;      // fp32(2^10 / global_scale) (bf16 path), 1 / global_scale (f16)
  float out_scale_up;   // the same for the up rows of SwiGLU (their own global scale)
  int stages_total;     // K / 256
  int split;            // CTAs per cluster along k
  int out_f32;          // 1: write f32 (before the bf16 rounding)
  int swiglu;           // 1: rows [0,N/2) gate, [N/2,N) up, y = silu(g)*u
  SmemLayout lay;
  SegScales seg;        // per-segment scales (seg.n == 0: out_scale for every column)
  unsigned int* err;    // device error word
  uint64_t wait_ns;     // limit of every pipeline wait (kWaitTimeoutNs)
  int test_stall;       // test hook: 1 = never load the last stage, so that the
                        // waits for it run out (split 1 only)
};

// 2^a as fp32, a in [-126, 127].
__device__ __forceinline__ float pow2f(int a) { return __int_as_float((a + 127) << 23); }

// Output (m, n) from its accumulated sums: v (row n, or the gate row with
// SwiGLU) and u (the up row), both before the global scale.  Columns past
// the output width (the last CTA's padding rows) are skipped.
__device__ __forceinline__ void store_output(const Params& p, int m, int64_t n, float v,
                                             float u) {
  const int64_t n_out = p.swiglu ? p.N / 2 : p.N;
  if (n >= n_out) return;
  float yv = v * (p.seg.n ? seg_scale(p.seg, n) : p.out_scale);
  if (p.swiglu) yv = silu_mul(yv, u * p.out_scale_up);
  const int64_t off = static_cast<int64_t>(m) * n_out + n;
  if (p.out_f32) {
    static_cast<float*>(p.y)[off] = yv;
    if (p.y_host) static_cast<float*>(p.y_host)[off] = yv;
  } else {
    const __nv_bfloat16 yb = __float2bfloat16_rn(yv);
    static_cast<__nv_bfloat16*>(p.y)[off] = yb;
    if (p.y_host) static_cast<__nv_bfloat16*>(p.y_host)[off] = yb;
  }
}

// Next position in a ring of `stages` slots; flips the barrier parity on
// wrap-around.
__device__ __forceinline__ int next_slot(int slot, int stages, uint32_t& parity) {
  if (++slot == stages) {
    parity ^= 1u;
    return 0;
  }
  return slot;
}

// The exact products of one stage for the flagged rows (bit m of `mine`) of
// one converter warp, in bf16 on the warp MMA: the same fragment layout as
// the consumers' bf16 path -- weights code * scale * 2^-10, activations as
// given, paired (k, k+4) -- over all 16G rows and 256 k of the stage.  The
// sums of the flagged rows' columns are added to the CTA's partials
// [8][16G + kRedPad] (still carrying 2^-10; the consumers' reduction scales them
// by 2^10); other columns stay zero and are not written.  Slow (about the
// consumers' whole stage in one warp), taken only for rows outside the f16
// window, and kept out of line so that it costs the converter's loop nothing
// otherwise.
template <int G>
__device__ __noinline__ void flagged_rows_bf16(const uint8_t* st, uint32_t mine,
                                               const SmemLayout& L, float* part, int lane) {
  constexpr int P = red_pitch(G);
  const int g = lane >> 2, t = lane & 3;
  const bool col_g = (mine >> g) & 1u;                  // B column g
  const bool own0 = (mine >> (2 * t)) & 1u;             // D columns 2t, 2t + 1
  const bool own1 = (mine >> (2 * t + 1)) & 1u;
#pragma unroll 1
  for (int r = 0; r < G; ++r) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int kq = 0; kq < kKQuarters; ++kq) {
      uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
      if (col_g) {
        const uint8_t* xr = st + L.x_off + g * 512 + kq * 128 + t * 32;
        c0 = *reinterpret_cast<const uint4*>(xr);
        c1 = *reinterpret_cast<const uint4*>(xr + 16);
      }
      const uint32_t b[8] = {prmt(c0.x, c0.z, 0x5410u), prmt(c0.x, c0.z, 0x7632u),
                             prmt(c0.y, c0.w, 0x5410u), prmt(c0.y, c0.w, 0x7632u),
                             prmt(c1.x, c1.z, 0x5410u), prmt(c1.x, c1.z, 0x7632u),
                             prmt(c1.y, c1.w, 0x5410u), prmt(c1.y, c1.w, 0x7632u)};
      uint32_t pw[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = kGroupRows * r + 2 * g + h;
        const int chunk = 2 * kq + (t >> 1);
        const uint2 w = *reinterpret_cast<const uint2*>(
            st + row * 128 + ((chunk ^ (row & 7)) << 4) + ((t & 1) << 3));
        const uint32_t sc = scale_pair_from_e4m3(st[L.s_off + row * 16 + 4 * kq + t]);
        dequant8_strided(w.x, sc, &pw[h][0]);
        dequant8_strided(w.y, sc, &pw[h][4]);
      }
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4)
        mma_bf16_16816(d, pw[0][2 * s4], pw[1][2 * s4], pw[0][2 * s4 + 1], pw[1][2 * s4 + 1],
                       b[2 * s4], b[2 * s4 + 1]);
    }
    const int ra = kGroupRows * r + 2 * g;
    if (own0) {
      part[2 * t * P + ra] += d[0];
      part[2 * t * P + ra + 1] += d[2];
    }
    if (own1) {
      part[(2 * t + 1) * P + ra] += d[1];
      part[(2 * t + 1) * P + ra + 1] += d[3];
    }
  }
}

// CV: 0 for the bf16 path; 1, 2 or 4 for the f16 path with that many
// activation converter warps (the host picks more as M grows).
// W: row-group ways -- 4 * W consumer warps, warp (k quarter, way w) taking
// the row groups w, w + W, ... of the CTA (2: eight consumers; 4: sixteen,
// for the bf16 path, with a quarter of the accumulators each).
template <int MT, int G, int CV, int W = kWays>
__global__ void __launch_bounds__(threads_for(CV, W), CV > 0 ? 2 : 1)
    smallm_kernel(const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_x, const Params p) {
  constexpr bool F16 = CV > 0;
  constexpr int kThreads = threads_for(CV, W);
  constexpr int kConsumerWarps = consumer_warps(W);
  constexpr int RG = groups_per_warp(MT, W);
  constexpr int C = MT * 8;
  constexpr int rows = G * kGroupRows;
  constexpr int half_rows = rows / 2;
  constexpr int P = red_pitch(G);
  static_assert(G >= 1 && G <= max_groups(MT), "row groups per CTA out of range");
  static_assert(W == kWays || !F16, "the f16 path keeps the default consumer layout");
  static_assert(!F16 || MT == 1, "the f16 path serves M <= 8");
  const SmemLayout& L = p.lay;
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base, formed by arithmetic on the shared array itself so
  // that every access through it stays a shared-memory access
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + L.lut_off);
  float* part = reinterpret_cast<float*>(smem + L.part_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* conv = full + L.stages;
  uint64_t* empty = conv + L.stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + L.stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = p.split;
  const int z = blockIdx.y;                                  // k-slice index
  const int st_begin = static_cast<int>((int64_t)p.stages_total * z / split);
  const int st_end = static_cast<int>((int64_t)p.stages_total * (z + 1) / split);
  const int n_stages = st_end - st_begin;

  // Weight rows of this CTA, as two boxes of 8G rows: consecutive rows, or
  // (SwiGLU) 8G gate rows and the 8G matching up rows.
  int row0, row1;
  if (p.swiglu) {
    row0 = blockIdx.x * half_rows;
    row1 = static_cast<int>(p.N / 2) + blockIdx.x * half_rows;
  } else {
    row0 = blockIdx.x * rows;
    row1 = row0 + half_rows;
  }

  for (int i = threadIdx.x; i < 256; i += kThreads)
    lut[i] = F16 ? scale_pair_f16_from_e4m3(i) : scale_pair_from_e4m3(i);
  // f16 path: the converters add the bf16 products of flagged rows into the
  // CTA's partials during the loop (the consumers' sums join them after it)
  if (F16)
    for (int i = threadIdx.x; i < C * P; i += kThreads) part[i] = 0.f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv[s], CV > 0 ? CV : 1);
      mbar_init(&empty[s], kConsumerWarps + CV);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Let the next kernel in the stream launch now: its CTAs take the SM room
  // this grid leaves free and prefetch their weights while this one runs.
  // (They read this kernel's results only after griddepcontrol.wait, which
  // waits for the whole grid to complete.)
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_s);
      prefetch_tensormap(&tm_x);
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      const uint32_t tx =
          static_cast<uint32_t>(rows * (kStageK / 2 + kStageK / 16) + L.x_tx);
      auto issue_weights = [&](int it, int slot) {
        uint8_t* st = smem + slot * L.stage_bytes;
        const int k0 = (st_begin + it) * kStageK;
        tma_load_2d_hint(st, &tm_w, &full[slot], k0 / 2, row0, pol_stream);
        tma_load_2d_hint(st + half_rows * 128, &tm_w, &full[slot], k0 / 2, row1, pol_stream);
        tma_load_2d_hint(st + L.s_off, &tm_s, &full[slot], k0 / 16, row0, pol_stream);
        tma_load_2d_hint(st + L.s_off + half_rows * 16, &tm_s, &full[slot], k0 / 16, row1,
                         pol_stream);
      };
      auto issue_acts = [&](int it, int slot) {
        uint8_t* st = smem + slot * L.stage_bytes;
        const int k0 = (st_begin + it) * kStageK;
        if (MT == 1) {
          tma_load_2d_hint(st + L.x_off, &tm_x, &full[slot], k0, 0, pol_keep);
        } else {
#pragma unroll
          for (int q = 0; q < kKQuarters; ++q)
            tma_load_2d_hint(st + L.x_off + q * L.x_box_bytes, &tm_x, &full[slot],
                             k0 + 64 * q, 0, pol_keep);
        }
      };
      // Test hook: the last stage is never loaded, so every wait for it
      // runs out (the host allows this only without a k split).
      const int skipped = p.test_stall ? n_stages - 1 : -1;
      // The weights do not depend on the preceding kernel in the stream:
      // fill the ring with them first, then wait for that kernel before
      // touching the activations.
      const int pre = n_stages < L.stages ? n_stages : L.stages;
      for (int it = 0; it < pre; ++it) {
        if (it == skipped) continue;
        mbar_arrive_expect_tx(&full[it], tx);
        issue_weights(it, it);
      }
      griddep_wait();
      for (int it = 0; it < pre; ++it)
        if (it != skipped) issue_acts(it, it);
      int issued = pre;
      int slot = pre == L.stages ? 0 : pre;
      uint32_t par = pre == L.stages ? 0u : 1u;
      for (int it = pre; it < n_stages; ++it) {
        if (!mbar_wait(&empty[slot], par, abort_flag, p.wait_ns)) break;
        if (it != skipped) {
          mbar_arrive_expect_tx(&full[slot], tx);
          issue_weights(it, slot);
          issue_acts(it, slot);
        }
        ++issued;
        slot = next_slot(slot, L.stages, par);
      }
      // Drain: never leave a copy in flight into this CTA's shared memory.
      const int first = issued > L.stages ? issued - L.stages : 0;
      for (int it = first; it < issued; ++it) {
        if (it == skipped) continue;
        volatile int no_abort = 0;
        if (!mbar_wait(&full[it % L.stages], (it / L.stages) & 1, &no_abort))
          atomicOr(p.err, kErrWaitTimeout);
      }
    }
  } else if (F16 && warp > kConsumerWarps) {
    // ------------------------------------------------------------ converters
    // Converter c takes activation rows c, c + CV, ...: one converter up to
    // M = 3, row after row; two from M = 4, each converting all of its rows
    // at once so that their load -> max -> convert chains overlap (one warp
    // for all the rows bounded the verify launch).  Lane l takes the 16-byte
    // chunk l (8 consecutive k) of each row of every stage.  a_run[i] is the
    // exponent of row c + CV * i: x is stored as f16(x * 2^a_run), with
    // a_run the largest value keeping the row's running maximum below 2^15
    // (so no f16 overflow).  A bf16 value of biased exponent e converts to
    // f16 exactly when e + a_run >= 110 (its last significant bit, at
    // 2^(e - 134 + a_run), is then at or above f16's smallest step 2^-24).
    // A row whose stage holds a nonzero value with a smaller exponent is
    // flagged: it goes to the consumers as zeros, and this warp adds the
    // row's exact bf16 products for the stage to the CTA's partials.
    constexpr int kConvWarps = CV > 0 ? CV : 1;
    constexpr int kRowsPer = kF16MaxRows / kConvWarps;
    const int c = warp - kConsumerWarps - 1;
    const int M = static_cast<int>(p.M);
    // this converter's rows (warp-uniform); the warp-wide maximum is not
    // cheap, and the conversion is on every stage's critical path: rows
    // past M are skipped, not processed as zeros
    const int n_rows = M > c ? (M - c + kConvWarps - 1) / kConvWarps : 0;
    // row m of the stage (this lane's 8 k) -> f16(x * 2^a) in the swizzled
    // operand tile; lane 0 records the row's exponent.  (max * 2^a < 2^15.)
    auto convert_row = [&](uint8_t* st, int m, const uint4& v, int a) {
      const float f = pow2f(a);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = f32x2_to_f16x2(__uint_as_float(w4[j] << 16) * f,
                              __uint_as_float(w4[j] & 0xFFFF0000u) * f);
      *reinterpret_cast<uint4*>(st + L.x16_off + m * 512 + ((lane ^ (m & 7)) << 4)) =
          make_uint4(o[0], o[1], o[2], o[3]);
      if (lane == 0) reinterpret_cast<int*>(st + L.exp_off)[m] = a;
    };
    // Warp-wide max |x| and (smallest nonzero |x|) - 1 of one row's 256 k, as
    // bf16 magnitude bits.  Per 16-bit lane of a word of magnitudes,
    // (h + 0x7FFF) & 0x7FFF is h - 1 for h > 0 and 0x7FFF for h = 0 (no carry
    // crosses lanes: h <= 0x7FFF).
    auto row_range = [&](const uint4& v, uint32_t& mx, uint32_t& mn) {
      const uint32_t a0 = v.x & 0x7FFF7FFFu, a1 = v.y & 0x7FFF7FFFu;
      const uint32_t a2 = v.z & 0x7FFF7FFFu, a3 = v.w & 0x7FFF7FFFu;
      mx = max_u16x2(max_u16x2(a0, a1), max_u16x2(a2, a3));
      mn = min_u16x2(min_u16x2((a0 + 0x7FFF7FFFu) & 0x7FFF7FFFu,
                               (a1 + 0x7FFF7FFFu) & 0x7FFF7FFFu),
                     min_u16x2((a2 + 0x7FFF7FFFu) & 0x7FFF7FFFu,
                               (a3 + 0x7FFF7FFFu) & 0x7FFF7FFFu));
      mx = __reduce_max_sync(0xffffffffu, max(mx & 0xFFFFu, mx >> 16));
      mn = __reduce_min_sync(0xffffffffu, min(mn & 0xFFFFu, mn >> 16));
    };
    // flagged: a nonzero magnitude below (110 - a) << 7
    auto out_of_window = [](uint32_t mn, int a) {
      return static_cast<int>(mn) < (110 - a) * 128 - 1;
    };
    int a_run[kRowsPer];
#pragma unroll
    for (int i = 0; i < kRowsPer; ++i) a_run[i] = 126;
    int slot = 0;                 // ring position, stepped without a divide
    uint32_t par = 0;
    for (int it = 0; it < n_stages; ++it, slot = next_slot(slot, L.stages, par)) {
      if (!mbar_wait(&full[slot], par, abort_flag, p.wait_ns)) break;
      uint8_t* st = smem + slot * L.stage_bytes;
      uint32_t mine = 0;             // this converter's flagged rows (warp-uniform)
      if constexpr (CV == 1) {
        // one converter (M <= 3): row after row
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          if (i >= n_rows) break;
          const uint4 v = *reinterpret_cast<const uint4*>(st + L.x_off + i * 512 + lane * 16);
          uint32_t mx, mn;
          row_range(v, mx, mn);
          a_run[i] = min(a_run[i], max(-126, 141 - static_cast<int>(mx >> 7)));
          mine |= out_of_window(mn, a_run[i]) ? 1u << i : 0u;
          convert_row(st, i, v, a_run[i]);
        }
      } else {
        // several converters (M >= 4): each converts all of its rows at once
        uint4 v[kRowsPer];
        int e_max[kRowsPer];
        uint32_t mn[kRowsPer];
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          if (i >= n_rows) break;
          v[i] = *reinterpret_cast<const uint4*>(st + L.x_off + (c + kConvWarps * i) * 512 +
                                                 lane * 16);
        }
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          if (i >= n_rows) break;
          uint32_t mx;
          row_range(v[i], mx, mn[i]);
          e_max[i] = static_cast<int>(mx >> 7);                // biased bf16 exponent
        }
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
          if (i >= n_rows) break;
          a_run[i] = min(a_run[i], max(-126, 141 - e_max[i]));
          mine |= out_of_window(mn[i], a_run[i]) ? 1u << (c + kConvWarps * i) : 0u;
          convert_row(st, c + kConvWarps * i, v[i], a_run[i]);
        }
      }
      // rows past M: a fixed exponent (their columns hold zeros)
      if (c == 0 && lane >= M && lane < kF16MaxRows)
        reinterpret_cast<int*>(st + L.exp_off)[lane] = 126;
      if (mine) {
        // rare: the flagged rows go to the consumers as zeros (this lane's
        // 16 bytes of each), and their exact products come from here
        for (int m = 0; m < kF16MaxRows; ++m)
          if ((mine >> m) & 1u)
            *reinterpret_cast<uint4*>(st + L.x16_off + m * 512 + ((lane ^ (m & 7)) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv[slot]);
      if (mine) flagged_rows_bf16<G>(st, mine, L, part, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    // the flagged rows' products are in the partials
    asm volatile("bar.arrive 2, %0;" ::"n"((kConsumerWarps + CV) * 32) : "memory");
  } else if (warp < kConsumerWarps) {
    // ------------------------------------------------------------ consumers
    // warp = (k quarter kq, row-group way rp): 64 k of every stage for
    // the row groups rp, rp + W, ... of this CTA.
    const int kq = warp & 3, rp = warp >> 2;
    const int g = lane >> 2, t = lane & 3;
    float acc[RG][MT][4];
#pragma unroll
    for (int i = 0; i < RG; ++i)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][mt][c] = 0.f;
    int a_col[2] = {126, 126};            // f16 path: exponents of columns 2t, 2t+1

    // MMA rows g and g+8 of group r are weight rows 16r+2g and 16r+2g+1:
    // with the 128B swizzle this makes the weight loads bank-conflict free.
    // Row 16r+2g+h has swizzle phase (2g+h) & 7 for every r, so each load
    // below is a per-thread base plus a compile-time offset for r.
    const int chunk = 2 * kq + (t >> 1);
    int w_base[2], s_base[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = kGroupRows * rp + 2 * g + h;
      w_base[h] = row * 128 + ((chunk ^ (row & 7)) << 4) + ((t & 1) << 3);
      s_base[h] = L.s_off + row * 16 + 4 * kq + t;
    }
    // Activations for MMA column g: elements [16t, 16t+16) of this warp's
    // 64-k quarter.  bf16: paired (k, k+4) like the bit trick's weights;
    // f16: the converter's tile, consecutive pairs.  Rows >= M are zero.
    const bool x_row = MT > 1 || g < static_cast<int>(p.M);
    int x_off[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int m = mt * 8 + g;
      if (MT == 1 && F16) {
        const int c = 8 * kq + 2 * t;
        x_off[mt][0] = L.x16_off + m * 512 + ((c ^ (m & 7)) << 4);
        x_off[mt][1] = L.x16_off + m * 512 + (((c + 1) ^ (m & 7)) << 4);
      } else if (MT == 1) {
        x_off[mt][0] = L.x_off + m * 512 + kq * 128 + t * 32;
        x_off[mt][1] = x_off[mt][0] + 16;
      } else {
        const int box = L.x_off + kq * L.x_box_bytes + m * 128;
        x_off[mt][0] = box + (((2 * t) ^ (m & 7)) << 4);
        x_off[mt][1] = box + (((2 * t + 1) ^ (m & 7)) << 4);
      }
    }

    int slot = 0;
    uint32_t par = 0;
    for (int it = 0; it < n_stages; ++it, slot = next_slot(slot, L.stages, par)) {
      // f16 path: the converter waited for the copies before releasing the
      // stage, so its barrier alone orders them before the loads below
      if (!F16 && !mbar_wait(&full[slot], par, abort_flag, p.wait_ns)) break;
      if (F16 && !mbar_wait(&conv[slot], par, abort_flag, p.wait_ns)) break;
      const uint8_t* st = smem + slot * L.stage_bytes;

      uint32_t bx[MT][8];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
        if (x_row) {
          c0 = *reinterpret_cast<const uint4*>(st + x_off[mt][0]);
          c1 = *reinterpret_cast<const uint4*>(st + x_off[mt][1]);
        }
        if (F16) {
          bx[mt][0] = c0.x; bx[mt][1] = c0.y; bx[mt][2] = c0.z; bx[mt][3] = c0.w;
          bx[mt][4] = c1.x; bx[mt][5] = c1.y; bx[mt][6] = c1.z; bx[mt][7] = c1.w;
        } else {
          bx[mt][0] = prmt(c0.x, c0.z, 0x5410u);
          bx[mt][1] = prmt(c0.x, c0.z, 0x7632u);
          bx[mt][2] = prmt(c0.y, c0.w, 0x5410u);
          bx[mt][3] = prmt(c0.y, c0.w, 0x7632u);
          bx[mt][4] = prmt(c1.x, c1.z, 0x5410u);
          bx[mt][5] = prmt(c1.x, c1.z, 0x7632u);
          bx[mt][6] = prmt(c1.y, c1.w, 0x5410u);
          bx[mt][7] = prmt(c1.y, c1.w, 0x7632u);
        }
      }
      if (F16) {
        // A column's exponent only ever decreases; rescale its running sums
        // (exactly, by a power of two) when it does.
        // The drop d lies in [-252, 0]: apply 2^d as two factors, each a
        // normal fp32 power of two, so that the product underflows as the
        // exact one would (one factor 2^d is not representable below -126).
        const int2 an = *reinterpret_cast<const int2*>(st + L.exp_off + 8 * t);
        if (an.x != a_col[0] || an.y != a_col[1]) {
          const int d0 = an.x - a_col[0], d1 = an.y - a_col[1];
          const float f0a = pow2f(d0 >> 1), f0b = pow2f(d0 - (d0 >> 1));
          const float f1a = pow2f(d1 >> 1), f1b = pow2f(d1 - (d1 >> 1));
#pragma unroll
          for (int i = 0; i < RG; ++i) {
            acc[i][0][0] = acc[i][0][0] * f0a * f0b;
            acc[i][0][2] = acc[i][0][2] * f0a * f0b;
            acc[i][0][1] = acc[i][0][1] * f1a * f1b;
            acc[i][0][3] = acc[i][0][3] * f1a * f1b;
          }
          a_col[0] = an.x;
          a_col[1] = an.y;
        }
      }

      // one row group: its weights dequantised, then its MMA chain
      auto group_operands = [&](int i, uint32_t (&pa)[8], uint32_t (&pb)[8]) {
        const uint2 wa =
            *reinterpret_cast<const uint2*>(st + w_base[0] + i * W * kGroupRows * 128);
        const uint2 wb =
            *reinterpret_cast<const uint2*>(st + w_base[1] + i * W * kGroupRows * 128);
        const uint32_t sa = lut[st[s_base[0] + i * W * kGroupRows * 16]];
        const uint32_t sb = lut[st[s_base[1] + i * W * kGroupRows * 16]];
        if (F16) {
          dequant8_f16(wa.x, sa, &pa[0]);
          dequant8_f16(wa.y, sa, &pa[4]);
          dequant8_f16(wb.x, sb, &pb[0]);
          dequant8_f16(wb.y, sb, &pb[4]);
        } else {
          dequant8_strided(wa.x, sa, &pa[0]);
          dequant8_strided(wa.y, sa, &pa[4]);
          dequant8_strided(wb.x, sb, &pb[0]);
          dequant8_strided(wb.y, sb, &pb[4]);
        }
      };
      auto group_mma = [&](int i, int s, const uint32_t (&pa)[8], const uint32_t (&pb)[8]) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          if (F16)
            mma_f16_16816(acc[i][mt], pa[2 * s], pb[2 * s], pa[2 * s + 1], pb[2 * s + 1],
                          bx[mt][2 * s], bx[mt][2 * s + 1]);
          else
            mma_bf16_16816(acc[i][mt], pa[2 * s], pb[2 * s], pa[2 * s + 1], pb[2 * s + 1],
                           bx[mt][2 * s], bx[mt][2 * s + 1]);
        }
      };
      if constexpr (G == W * RG && RG % 2 == 0) {
        // a full CTA: two groups at a time, their MMA chains interleaved
#pragma unroll
        for (int i = 0; i < RG; i += 2) {
          uint32_t pa0[8], pb0[8], pa1[8], pb1[8];
          group_operands(i, pa0, pb0);
          group_operands(i + 1, pa1, pb1);
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            group_mma(i, s4, pa0, pb0);
            group_mma(i + 1, s4, pa1, pb1);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < RG; ++i) {
          const int r = rp + W * i;
          if (G != W * RG && r >= G) break;      // uniform; never when G fills the ways
          uint32_t pa[8], pb[8];
          group_operands(i, pa, pb);
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) group_mma(i, s4, pa, pb);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (F16) {
      // back to the activations' own units: divide column c by 2^a_col
      const float u0 = pow2f(-a_col[0]), u1 = pow2f(-a_col[1]);
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        acc[i][0][0] *= u0;
        acc[i][0][2] *= u0;
        acc[i][0][1] *= u1;
        acc[i][0][3] *= u1;
      }
    }

    // Warp partials -> ring (free now: every stage has been consumed once
    // all consumer warps -- and, on the f16 path, the converters, which read
    // the ring for flagged rows -- pass the barrier below).  Only the
    // columns that hold activation rows are kept.
    if (F16)
      asm volatile("bar.sync 2, %0;" ::"n"((kConsumerWarps + CV) * 32) : "memory");
    else
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    const int M = static_cast<int>(p.M);
    float* red = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int i = 0; i < RG; ++i) {
      const int r = rp + W * i;
      if (G != W * RG && r >= G) break;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int ra = kGroupRows * r + 2 * g, col = mt * 8 + 2 * t;
        float* base = red + kq * C * P + ra;
        if (col < M)
          *reinterpret_cast<float2*>(base + col * P) = make_float2(acc[i][mt][0], acc[i][mt][2]);
        if (col + 1 < M)
          *reinterpret_cast<float2*>(base + (col + 1) * P) =
              make_float2(acc[i][mt][1], acc[i][mt][3]);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    // the four k quarters' sums of (weight row j, activation row m), and on
    // the f16 path the flagged rows' bf16 products (carrying 2^-10)
    auto quarter_sum = [&](int j, int m) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < kKQuarters; ++q) s += red[(q * C + m) * P + j];
      return F16 ? s + part[m * P + j] * kWeightPow2 : s;
    };
    if (split == 1) {
      // the CTA holds whole sums: write the outputs from here
      if (*abort_flag && threadIdx.x == 0) atomicOr(p.err, kErrWaitTimeout);
      if (p.swiglu) {
        const int64_t n_base = static_cast<int64_t>(blockIdx.x) * half_rows;
        for (int i = threadIdx.x; i < half_rows * M; i += kConsumerWarps * 32) {
          const int m = i / half_rows, j = i % half_rows;
          store_output(p, m, n_base + j, quarter_sum(j, m), quarter_sum(half_rows + j, m));
        }
      } else {
        const int64_t n_base = static_cast<int64_t>(blockIdx.x) * rows;
        for (int i = threadIdx.x; i < rows * M; i += kConsumerWarps * 32) {
          const int m = i / rows, j = i % rows;
          store_output(p, m, n_base + j, quarter_sum(j, m), 0.f);
        }
      }
      return;
    }
    for (int i = threadIdx.x; i < rows * M; i += kConsumerWarps * 32) {
      const int m = i / rows, j = i % rows;
      part[m * P + j] = quarter_sum(j, m);
    }
  }

  if (split == 1) return;             // producer and converters: nothing left
  if (*abort_flag && threadIdx.x == 0) atomicOr(p.err, kErrWaitTimeout);

  // ---------------------------------------------------------------- epilogue
  // (k split) Every CTA of the cluster finishes its partial; CTA z then
  // reduces a 1/split share of the outputs across the cluster's shared
  // memories.  (Reconverge each warp first: the cluster barrier is a
  // warp-aligned op.)
  __syncwarp();
  cluster_sync();
  {
    const int M = static_cast<int>(p.M);
    const int R = p.swiglu ? half_rows : rows;           // outputs per activation row
    const int items = R * M;
    const int i0 = static_cast<int>((int64_t)items * z / split);
    const int i1 = static_cast<int>((int64_t)items * (z + 1) / split);
    const uint32_t part_local = smem_addr(part);
    const int64_t n_base = static_cast<int64_t>(blockIdx.x) * R;
    for (int i = i0 + threadIdx.x; i < i1; i += kThreads) {
      const int m = i / R, j = i % R;
      const float v = cluster_sum_f32<kMaxSplit>(part_local, 4u * (m * P + j), split);
      const float u =
          p.swiglu ? cluster_sum_f32<kMaxSplit>(part_local, 4u * (m * P + half_rows + j), split)
                   : 0.f;
      store_output(p, m, n_base + j, v, u);
    }
  }
  __syncwarp();
  cluster_sync();   // keep every partial alive until all readers are done
}

}  // namespace smallm
}  // namespace nvfp4
