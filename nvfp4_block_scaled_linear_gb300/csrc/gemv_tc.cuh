// gemv_tc.cuh -- NVFP4 W4A16 linear for few activation rows (M <= 32):
// decode (M = 1), speculative verify (M = K+1, FlashRT docs section 3) and
// small continuous batches, on the tcgen05 tensor cores, in f16.  (Run when
// forced: the bf16 kernel of gemv_bf16.cuh and the warp-MMA kernel are the
// defaults; this one is kept for its f16 arithmetic and per-stage exponents.)
//
// At these sizes the layer is bound by streaming the packed weights and
// scales from HBM once.  What limits a kernel that keeps up with HBM is the
// instruction issue of the streaming multiprocessors: decoding 16 FP4 codes
// and applying their block scale costs a few instructions per weight, and
// register-fed warp MMAs add their own operand traffic on top.  Here the
// CUDA cores only dequantise; the tensor core does every multiply-add:
//
//  * One CTA owns 128 weight rows (the MMA's M; SwiGLU: 64 gate rows and
//    the 64 matching up rows) and a contiguous range of k.  A producer warp
//    streams 256-k stages -- packed codes (128B-swizzled), block scales and
//    the M activation rows -- into a shared-memory ring with TMA.  The codes
//    of the first ring-full are requested before the kernel waits on the
//    preceding kernel in the stream (programmatic dependent launch).
//  * Eight dequantisation warps turn the codes into f16 weights: the
//    hardware e2m1 -> f16x2 conversion and one f16x2 multiply by the block
//    scale give code * scale exactly.  Each thread owns one weight row (its
//    TMEM lane) and writes 64 k of it per half stage straight into tensor
//    memory with tcgen05.st: the weights never pass through shared memory.
//  * One thread issues tcgen05.mma kind::f16 with A = the dequantised
//    weights in TMEM, B = the activations (f16, 128B-swizzled K-major in
//    shared memory, N = 16 or 32 rows) and D = fp32 in TMEM: 16 MMAs of
//    K = 16 per stage.
//  * Two converter warps bring each stage's activation rows to f16 with a
//    power-of-two scale per row and stage, taken from that row's maximum
//    |x| within the stage (so the largest value stays below 2^15).  Every
//    activation within 2^31 of that maximum converts exactly, and nothing
//    overflows.  Because the scale differs per stage, each stage
//    accumulates into a fresh D (double-buffered in TMEM), and four
//    accumulator warps add D * 2^-scale into fp32 registers per row.
//  * Split-K: CTAs that share rows but not k form one thread-block cluster;
//    partials are reduced across the cluster through distributed shared
//    memory.  No global workspace, no atomics, no waits on other CTAs.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace gemvtc {

constexpr int kRows = 128;              // weight rows per CTA (the MMA's M)
constexpr int kHalfRows = kRows / 2;    // one TMA box of rows
constexpr int kStageK = 256;            // k per pipeline stage
constexpr int kASlots = 3;              // TMEM weight ring, 128 k (64 columns) each
constexpr int kAColsPerSlot = 64;
constexpr int kDCol = kASlots * kAColsPerSlot;   // D buffers start at column 192
constexpr int kMaxRows = 32;            // activation rows served
constexpr int kMaxSplit = 16;           // cluster size limit (non-portable above 8)

// Warp roles.  Two MMA issuers: a single thread issues at most one
// tcgen05.mma every ~30-60 ns whatever the MMA's N, far below what the
// tensor core accepts from several issuers, so half stage h of every stage
// is issued by warp kWarpMma + h into its own accumulator.  N = 32 (up to
// 32 activation rows) runs one CTA per SM and gets three converter warps.
template <int NM>
struct Roles {
  static constexpr int kWarpProducer = 0;
  static constexpr int kWarpMma = 1;                       // issuers: warps 1, 2
  static constexpr int kWarpConv = 3;
  static constexpr int kConvWarps = NM == 16 ? 1 : 3;
  static constexpr int kWarpDeq = kWarpConv + kConvWarps;  // eight dequantisation warps
  static constexpr int kDeqWarps = 8;
  static constexpr int kWarpAcc = kWarpDeq + kDeqWarps;   // four accumulator warps
  static constexpr int kAccWarps = 4;
  static constexpr int kThreads = (kWarpAcc + kAccWarps) * 32;
  // weight ring (192 columns) + accumulators [2 buffers][2 half stages][NM]
  static constexpr uint32_t kTmemCols = NM == 16 ? 256 : 512;
  static_assert(kDCol + 4 * NM <= static_cast<int>(kTmemCols), "TMEM plan");
};

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory layout of one launch (byte offsets from the 1024-aligned
// base), computed on the host per call.  A stage holds the codes
// [128 rows][128 B] (128B-swizzled), the scales [128 rows][16 B], the bf16
// activations [M rows][256 k] and their f16 MMA operand: four 64-k column
// blocks of [N rows][128 B], 128B-swizzled, N = 16 or 32.
struct SmemLayout {
  int stages;
  int stage_bytes;
  int s_off;        // scales, within a stage
  int x_off;        // bf16 activations, within a stage
  int b_off;        // f16 MMA operand, within a stage
  int exp_off;      // int[2 * stages][32]: activation exponents per stage
  int lut_off;      // 256 f16 scale pairs
  int bar_off;      // mbarriers, abort flag, TMEM base
  int total;        // dynamic shared memory to request (with alignment slack)
};

__host__ __device__ constexpr int num_barriers(int stages) { return 5 * stages + 7; }

__host__ __device__ constexpr SmemLayout make_layout(int n_mma, int m_rows, int stages) {
  SmemLayout l{};
  l.stages = stages;
  l.s_off = kRows * 128;
  l.x_off = align_up(l.s_off + kRows * 16, 128);
  l.b_off = align_up(l.x_off + m_rows * kStageK * 2, 1024);
  l.stage_bytes = align_up(l.b_off + n_mma * kStageK * 2, 1024);
  l.exp_off = stages * l.stage_bytes;
  l.lut_off = l.exp_off + 2 * stages * kMaxRows * 4;
  l.bar_off = l.lut_off + 256 * 4;
  l.total = l.bar_off + num_barriers(stages) * 8 + 16 + 1024;
  return l;
}

// The final cross-warp exchange reuses the ring; it must fit.
__host__ __device__ constexpr bool layout_ok(const SmemLayout& l, int n_mma) {
  return l.stages >= 2 && kRows * n_mma * 4 <= l.stages * l.stage_bytes;
}

struct Params {
  void* y;              // [M, N] (or [M, N/2] with swiglu), bf16 or f32
  void* y_host;         // nullptr, or the same output again in host memory mapped
                        // into the device (the host-buffer entry point)
  int64_t M, N, K;
  float out_scale;      // 1 / global_scale
  float out_scale_up;   // 1 / the up rows' global scale (SwiGLU)
  int stages_total;     // K / 256
  int split;            // CTAs per cluster along k
  int out_f32;          // 1: write f32 (before the bf16 rounding)
  int swiglu;           // 1: rows [0,N/2) gate, [N/2,N) up, y = silu(g)*u
  SmemLayout lay;
  SegScales seg;        // per-segment scales (seg.n == 0: out_scale for every column)
  unsigned int* err;    // device error word
};

__device__ __forceinline__ float pow2f(int a) { return __int_as_float((a + 127) << 23); }

// A wait whose outcome the whole warp shares: the warp-aligned tcgen05 and
// reduction instructions after it need every lane converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

__device__ __forceinline__ int next_slot(int slot, int n, uint32_t& parity) {
  if (++slot == n) {
    parity ^= 1u;
    return 0;
  }
  return slot;
}

template <int NM>
__global__ void __launch_bounds__(Roles<NM>::kThreads, NM == 16 ? 2 : 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_s,
                   const __grid_constant__ CUtensorMap tm_x, const Params p) {
  static_assert(NM == 16 || NM == 32, "MMA N is 16 or 32");
  using R = Roles<NM>;
  constexpr int kThreads = R::kThreads;
  const SmemLayout& L = p.lay;
  const int S = L.stages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base, formed by arithmetic on the shared array itself so
  // that every access through it stays a shared-memory access
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + L.lut_off);
  int* exps = reinterpret_cast<int*>(smem + L.exp_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);   // TMA landed
  // stage consumed: both issuers' MMAs of the stage have completed (their one
  // commit each).  Besides releasing the ring slot, it tells the accumulator
  // warps that the stage's D is ready and the dequantisers that the stage's
  // TMEM weight slots are free: one tcgen05.commit per stage and issuer
  // (a commit costs the issuing thread far more than an MMA).
  uint64_t* empty = full + S;
  uint64_t* b_full = empty + S;        // f16 activations written (converters)
  uint64_t* exp_full = b_full + S;     // [2S] exponents written (converters)
  uint64_t* a_full = exp_full + 2 * S; // [3] TMEM weights written (dequantisers)
  uint64_t* d_empty = a_full + kASlots;    // [2] stage accumulators read (acc warps)
  uint64_t* mma_done = d_empty + 2;        // [2] every MMA of issuer h has completed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(mma_done + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = static_cast<int>(p.M);
  const int split = p.split;
  const int z = blockIdx.y;                                  // k-slice index
  const int st_begin = static_cast<int>((int64_t)p.stages_total * z / split);
  const int st_end = static_cast<int>((int64_t)p.stages_total * (z + 1) / split);
  const int n_stages = st_end - st_begin;

  // Weight rows of this CTA, as two boxes of 64 rows: consecutive rows, or
  // (SwiGLU) 64 gate rows and the 64 matching up rows.
  int row0, row1;
  if (p.swiglu) {
    row0 = blockIdx.x * kHalfRows;
    row1 = static_cast<int>(p.N / 2) + blockIdx.x * kHalfRows;
  } else {
    row0 = blockIdx.x * kRows;
    row1 = row0 + kHalfRows;
  }

  for (int i = threadIdx.x; i < 256; i += kThreads) lut[i] = scale_pair_f16_from_e4m3(i);
  // The f16 operand rows past M stay zero for the whole launch.
  for (int s = 0; s < S; ++s) {
    uint4* b = reinterpret_cast<uint4*>(smem + s * L.stage_bytes + L.b_off);
    for (int i = threadIdx.x; i < NM * kStageK * 2 / 16; i += kThreads)
      b[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
      mbar_init(&b_full[s], R::kConvWarps);
    }
    for (int e = 0; e < 2 * S; ++e) mbar_init(&exp_full[e], R::kConvWarps);
    for (int a = 0; a < kASlots; ++a) mbar_init(&a_full[a], R::kDeqWarps);
    for (int d = 0; d < 2; ++d) {
      mbar_init(&d_empty[d], R::kAccWarps);
      mbar_init(&mma_done[d], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == R::kWarpMma) {
    tmem_alloc(tmem_slot, R::kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();            // the zeroed operand rows, for the MMA
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Let the next kernel in the stream launch now: its CTAs take the SM room
  // this grid leaves free and prefetch their weights while this one runs.
  // (They read this kernel's results only after griddepcontrol.wait, which
  // waits for the whole grid to complete.)
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == R::kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_s);
      prefetch_tensormap(&tm_x);
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      const uint32_t tx = static_cast<uint32_t>(kRows * (kStageK / 2 + kStageK / 16) +
                                                M * kStageK * 2);
      auto issue_weights = [&](int it, int slot) {
        uint8_t* st = smem + slot * L.stage_bytes;
        const int k0 = (st_begin + it) * kStageK;
        tma_load_2d_hint(st, &tm_w, &full[slot], k0 / 2, row0, pol_stream);
        tma_load_2d_hint(st + kHalfRows * 128, &tm_w, &full[slot], k0 / 2, row1, pol_stream);
        tma_load_2d_hint(st + L.s_off, &tm_s, &full[slot], k0 / 16, row0, pol_stream);
        tma_load_2d_hint(st + L.s_off + kHalfRows * 16, &tm_s, &full[slot], k0 / 16, row1,
                         pol_stream);
      };
      auto issue_acts = [&](int it, int slot) {
        uint8_t* st = smem + slot * L.stage_bytes;
        tma_load_2d_hint(st + L.x_off, &tm_x, &full[slot], (st_begin + it) * kStageK, 0,
                         pol_keep);
      };
      // The weights do not depend on the preceding kernel in the stream:
      // fill the ring with them first, then wait for that kernel before
      // touching the activations.
      const int pre = n_stages < S ? n_stages : S;
      for (int it = 0; it < pre; ++it) {
        mbar_arrive_expect_tx(&full[it], tx);
        issue_weights(it, it);
      }
      griddep_wait();
      for (int it = 0; it < pre; ++it) issue_acts(it, it);
      int issued = pre;
      int slot = pre == S ? 0 : pre;
      uint32_t par = pre == S ? 0u : 1u;
      for (int it = pre; it < n_stages; ++it) {
        if (!mbar_wait(&empty[slot], par, abort_flag)) break;
        mbar_arrive_expect_tx(&full[slot], tx);
        issue_weights(it, slot);
        issue_acts(it, slot);
        ++issued;
        slot = next_slot(slot, S, par);
      }
      // Drain: never leave a copy in flight into this CTA's shared memory.
      const int first = issued > S ? issued - S : 0;
      for (int it = first; it < issued; ++it) {
        volatile int no_abort = 0;
        if (!mbar_wait(&full[it % S], (it / S) & 1, &no_abort)) atomicOr(p.err, kErrWaitTimeout);
      }
    }
  } else if (warp == R::kWarpMma || warp == R::kWarpMma + 1) {
    // ------------------------------------------------------------ MMA issue
    // Issuer h takes half stage h (k [128h, 128h + 128)) of every stage:
    // 8 MMAs of K = 16 into accumulator [dbuf][h].
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_f16(kRows, NM);
      const int h = warp - R::kWarpMma;
      int slot = 0;
      uint32_t par = 0;
      int g = h;                                     // half-stage index 2 * it + h
      for (int it = 0; it < n_stages; ++it, g += 2) {
        const int dbuf = it & 1;
        const int aslot = g % kASlots;
        const uint32_t apar = static_cast<uint32_t>(g / kASlots) & 1u;
        if (!mbar_wait(&b_full[slot], par, abort_flag)) break;
        if (!mbar_wait(&d_empty[dbuf], ((it >> 1) & 1) ^ 1u, abort_flag)) break;
        if (!mbar_wait(&a_full[aslot], apar, abort_flag)) break;
        tc_fence_after_sync();
        // Operand column blocks 2h and 2h + 1; 32-byte steps within their
        // 128-byte swizzled rows (the descriptor's address field counts 16 B).
        const uint64_t b_desc0 =
            umma_desc_sw128(smem_addr(smem + slot * L.stage_bytes + L.b_off) + 2 * h * (NM * 128));
        const uint32_t d_tmem = tmem + kDCol + (2 * dbuf + h) * NM;
        const uint32_t a_tmem = tmem + aslot * kAColsPerSlot;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t b_desc =
              b_desc0 + static_cast<uint64_t>(((kk / 4) * (NM * 128) + (kk % 4) * 32) >> 4);
          umma_f16_tmem_a(d_tmem, a_tmem + kk * 8, b_desc, idesc, kk != 0);
        }
        umma_commit(&empty[slot]);
        slot = next_slot(slot, S, par);
      }
      // Every MMA issued must have completed before TMEM is released.
      umma_commit(&mma_done[h]);
      volatile int no_abort = 0;
      if (!mbar_wait(&mma_done[h], 0, &no_abort)) atomicOr(p.err, kErrWaitTimeout);
    }
  } else if (warp < R::kWarpDeq) {
    // ------------------------------------------------------------ converters
    // Converter c takes activation rows c, c+2, ...; lane l the 16-byte
    // chunk l (8 consecutive k) of each.  Row m of stage s is stored as
    // f16(x * 2^a) with a = the largest exponent keeping the row's maximum
    // |x| within this stage below 2^15.
    const int c = warp - R::kWarpConv;
    const int q = lane >> 3, c16 = lane & 7;       // 64-k column block, 16-B unit
    int slot = 0, e = 0;
    uint32_t par = 0, epar = 0;
    for (int it = 0; it < n_stages; ++it) {
      if (!warp_wait(&full[slot], par, abort_flag)) break;
      uint8_t* st = smem + slot * L.stage_bytes;
      // four rows at a time: their load -> max -> scale -> store chains
      // overlap (one row at a time leaves the warp waiting on latencies)
      for (int m0 = c; m0 < M; m0 += 4 * R::kConvWarps) {
        uint4 v[4];
        int e_max[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int m = m0 + u * R::kConvWarps;
          v[u] = m < M ? *reinterpret_cast<const uint4*>(st + L.x_off + m * 512 + lane * 16)
                       : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t mx = max_u16x2(max_u16x2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu),
                                  max_u16x2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu));
          mx = __reduce_max_sync(0xffffffffu, max(mx & 0xFFFFu, mx >> 16));
          e_max[u] = static_cast<int>(mx >> 7);                 // biased bf16 exponent
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int m = m0 + u * R::kConvWarps;
          if (m >= M) break;
          const int a = min(126, max(-126, 141 - e_max[u]));    // max * 2^a < 2^15
          const float f = pow2f(a);
          const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            o[j] = f32x2_to_f16x2(__uint_as_float(w4[j] << 16) * f,
                                  __uint_as_float(w4[j] & 0xFFFF0000u) * f);
          *reinterpret_cast<uint4*>(st + L.b_off + q * (NM * 128) + (m >> 3) * 1024 +
                                    (m & 7) * 128 + ((c16 ^ (m & 7)) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
          if (lane == 0) exps[e * kMaxRows + m] = a;
        }
      }
      fence_proxy_async_smem();      // the operand, for the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&b_full[slot]);
        mbar_arrive(&exp_full[e]);
      }
      slot = next_slot(slot, S, par);
      e = next_slot(e, 2 * S, epar);
    }
  } else if (warp < R::kWarpAcc) {
    // ------------------------------------------------------------ dequantisers
    // Warp (quadrant q, k half kh): lane = weight row 32q + lane = its TMEM
    // lane; per half stage it writes k [64kh, 64kh + 64) of that row.
    const int dw = warp - R::kWarpDeq;
    const int q = warp & 3, kh = dw >> 2;
    const int row = 32 * q + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16) + kh * 32;
    int slot = 0, aslot = 0;
    uint32_t par = 0;
    // Half stage g reuses the TMEM slot of half g - 3, whose stage
    // (g - 3) / 2 must have completed: `done_*` walks those stages.
    int done_slot = 0;
    uint32_t done_par = 0;
    bool ok = true;
    for (int it = 0; it < n_stages && ok; ++it) {
      if (!warp_wait(&full[slot], par, abort_flag)) break;
      const uint8_t* st = smem + slot * L.stage_bytes;
      const uint4 sc = *reinterpret_cast<const uint4*>(st + L.s_off + row * 16);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int g = 2 * it + h;
        if (g >= kASlots) {
          if (!warp_wait(&empty[done_slot], done_par, abort_flag)) {
            ok = false;
            break;
          }
          // g - 3 odd: the next half (g + 1) waits on the same stage
          if ((g - kASlots) & 1) done_slot = next_slot(done_slot, S, done_par);
        }
        // 64 k = two 16-byte code chunks of the row's 128-byte line
        const int c0 = 4 * h + 2 * kh;
        const uint4 w0 = *reinterpret_cast<const uint4*>(st + row * 128 + ((c0 ^ (row & 7)) << 4));
        const uint4 w1 =
            *reinterpret_cast<const uint4*>(st + row * 128 + (((c0 + 1) ^ (row & 7)) << 4));
        // their four 16-k blocks' scales: bytes 8h + 4kh .. +3 of the row
        const uint32_t s4 = h == 0 ? (kh ? sc.y : sc.x) : (kh ? sc.w : sc.z);
        const uint32_t S0 = lut[s4 & 0xFFu], S1 = lut[(s4 >> 8) & 0xFFu];
        const uint32_t S2 = lut[(s4 >> 16) & 0xFFu], S3 = lut[s4 >> 24];
        uint32_t out[32];
        dequant8_f16(w0.x, S0, &out[0]);
        dequant8_f16(w0.y, S0, &out[4]);
        dequant8_f16(w0.z, S1, &out[8]);
        dequant8_f16(w0.w, S1, &out[12]);
        dequant8_f16(w1.x, S2, &out[16]);
        dequant8_f16(w1.y, S2, &out[20]);
        dequant8_f16(w1.z, S3, &out[24]);
        dequant8_f16(w1.w, S3, &out[28]);
        tc_fence_after_sync();
        tmem_st_32cols(t_lane + aslot * kAColsPerSlot, out);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[aslot]);
        aslot = aslot + 1 == kASlots ? 0 : aslot + 1;
      }
      slot = next_slot(slot, S, par);
    }
  }

  // ---------------------------------------------------------------- accumulators
  // Warp (quadrant q): lane = weight row 32q + lane; acc[m] sums
  // D_stage[row][m] * 2^-a(stage, m) over this CTA's stages.
  float acc[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.f;
  if (warp >= R::kWarpAcc) {
    const int q = warp & 3;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16) + kDCol;
    int e = 0, slot = 0;
    uint32_t epar = 0, par = 0;
    for (int it = 0; it < n_stages; ++it) {
      const int dbuf = it & 1;
      // the stage's MMAs have completed: its accumulators are ready
      if (!warp_wait(&empty[slot], par, abort_flag)) break;
      slot = next_slot(slot, S, par);
      if (!warp_wait(&exp_full[e], epar, abort_flag)) break;
      tc_fence_after_sync();
      const int* ex = exps + e * kMaxRows;
#pragma unroll
      for (int half = 0; half < NM / 16; ++half) {
        // the two half-stage accumulators of this stage, columns [16 half, +16)
        uint32_t d0[16], d1[16];
        tmem_ld_16cols(t_lane + (2 * dbuf) * NM + 16 * half, d0);
        tmem_ld_16cols(t_lane + (2 * dbuf + 1) * NM + 16 * half, d1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = 16 * half + j;
          if (m < M)
            acc[m] = fmaf(__uint_as_float(d0[j]) + __uint_as_float(d1[j]), pow2f(-ex[m]), acc[m]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[dbuf]);
      e = next_slot(e, 2 * S, epar);
    }
  }

  if (*abort_flag && threadIdx.x == 0) atomicOr(p.err, kErrWaitTimeout);
  // Every role is done with the ring and TMEM: release TMEM, then reuse the
  // ring for the partial sums [128 rows][NM].
  tc_fence_before_sync();
  __syncthreads();
  if (warp == R::kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, R::kTmemCols);
  }
  float* part = reinterpret_cast<float*>(smem);
  if (warp >= R::kWarpAcc) {
    const int row = 32 * (warp & 3) + lane;
#pragma unroll
    for (int m = 0; m < NM; ++m)
      if (m < M) part[row * NM + m] = acc[m];
  }

  // ---------------------------------------------------------------- epilogue
  // Every CTA of the cluster finishes its partial; CTA z then reduces a
  // 1/split share of the outputs across the cluster's shared memories.
  // (Reconverge each warp first: the cluster barrier is a warp-aligned op.)
  __syncwarp();
  if (split > 1)
    cluster_sync();
  else
    __syncthreads();
  {
    const int R = p.swiglu ? kHalfRows : kRows;            // outputs per activation row
    const int items = R * M;
    const int i0 = static_cast<int>((int64_t)items * z / split);
    const int i1 = static_cast<int>((int64_t)items * (z + 1) / split);
    const uint32_t part_local = smem_addr(part);
    const int64_t n_out = p.swiglu ? p.N / 2 : p.N;
    const int64_t n_base = static_cast<int64_t>(blockIdx.x) * R;
    for (int i = i0 + threadIdx.x; i < i1; i += kThreads) {
      const int m = i / R, j = i % R;
      float v = 0.f, u = 0.f;
      if (split == 1) {
        v = part[j * NM + m];
        if (p.swiglu) u = part[(kHalfRows + j) * NM + m];
      } else {
        v = cluster_sum_f32<kMaxSplit>(part_local, 4u * (j * NM + m), split);
        if (p.swiglu)
          u = cluster_sum_f32<kMaxSplit>(part_local, 4u * ((kHalfRows + j) * NM + m), split);
      }
      float yv = v * (p.seg.n ? seg_scale(p.seg, n_base + j) : p.out_scale);
      if (p.swiglu) yv = silu_mul(yv, u * p.out_scale_up);
      const int64_t off = static_cast<int64_t>(m) * n_out + n_base + j;
      if (p.out_f32) {
        static_cast<float*>(p.y)[off] = yv;
        if (p.y_host) static_cast<float*>(p.y_host)[off] = yv;
      } else {
        const __nv_bfloat16 yb = __float2bfloat16_rn(yv);
        static_cast<__nv_bfloat16*>(p.y)[off] = yb;
        if (p.y_host) static_cast<__nv_bfloat16*>(p.y_host)[off] = yb;
      }
    }
  }
  if (split > 1) {
    __syncwarp();
    cluster_sync();   // keep every partial alive until all readers are done
  }
}

}  // namespace gemvtc
}  // namespace nvfp4
