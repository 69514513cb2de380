// gemv_bf16.cuh -- NVFP4 W4A16 linear for few activation rows (M <= 32) on
// the tcgen05 tensor cores, in bf16: decode (M = 1), speculative verify
// (M = K+1, FlashRT docs section 3) and small continuous batches.
//
// The layer is bound by streaming the packed weights and scales from HBM
// once.  The CUDA cores dequantise, the tensor core does every multiply-add,
// and nothing in the main loop depends on reading results back:
//
//  * One CTA owns 128 weight rows (the MMA's M; SwiGLU: 64 gate rows and
//    the 64 matching up rows) and a contiguous range of k.  A producer warp
//    streams 256-k stages -- packed codes (128B-swizzled), block scales and
//    the activations -- into a shared-memory ring with TMA.  The activation
//    tile is the MMA's B operand: bf16, 128B-swizzled K-major, NM = 16 or
//    32 rows, the rows past M filled with zeros by the copy.
//  * A stage is four 64-k jobs.  Job j goes to lane group j mod NI: four
//    dequantisation warps (one per 32-row TMEM lane quadrant) write the
//    job's weights as bf16 code * scale * 2^-10 (exact) into that group's
//    TMEM ring, with the k of every 8-k block in the order the bit trick
//    yields them, and permute the job's activation tile in place to the same
//    order; the group's own MMA issuer then adds A (TMEM) x B (shared
//    memory) into the group's own fp32 accumulator in TMEM.  NI issuers run
//    side by side: one thread issues at most one tcgen05.mma every
//    ~30-60 ns, far below what the tensor core accepts from several.
//  * The accumulators stay in TMEM for the whole k range; the epilogue reads
//    them once, sums the NI groups and applies 2^10 / global scale.
//  * Split-K: CTAs that share rows but not k form one thread-block cluster;
//    each CTA owns a share of the outputs, pushes its partial values of the
//    others' shares into their shared memory (remote stores) and, after one
//    cluster barrier, sums its own share in rank order.  No global
//    workspace, no atomics.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace gemvbf {

constexpr int kRows = 128;              // weight rows per CTA (the MMA's M)
constexpr int kHalfRows = kRows / 2;    // one TMA box of rows
constexpr int kStageK = 256;            // k per pipeline stage
constexpr int kJobK = 64;               // k per job (one TMEM slot, 32 columns)
constexpr int kJobsPerStage = kStageK / kJobK;
constexpr int kSlotCols = kJobK / 2;    // bf16 pairs per TMEM column
constexpr int kSlotsPerGroup = 3;       // TMEM weight ring depth of one lane group
constexpr int kMaxSplit = 16;           // cluster size limit (non-portable above 8)

// Warp roles for NI lane groups: warp 0 the producer, warps 1..NI the
// issuers, then NI quartets of dequantisation warps.  NI = 4 runs one CTA
// per SM (TMEM 512 columns), NI = 2 two CTAs per SM (256 columns each).
template <int NM, int NI>
struct Roles {
  static constexpr int kWarpProducer = 0;
  static constexpr int kWarpMma = 1;
  static constexpr int kWarpDeq = 1 + NI;
  static constexpr int kDeqWarps = 4 * NI;
  static constexpr int kThreads = (kWarpDeq + kDeqWarps) * 32;
  static constexpr int kCtasPerSm = NI == 4 ? 1 : 2;
  static constexpr int kDCol = NI * kSlotsPerGroup * kSlotCols;   // accumulators' first column
  static constexpr uint32_t kTmemCols = 512 / kCtasPerSm;
  static_assert(NI == 2 || NI == 4, "two or four lane groups");
  static_assert(kDCol + NI * NM <= static_cast<int>(kTmemCols), "TMEM plan");
};

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory layout of one launch (byte offsets from the 1024-aligned
// base), computed on the host per call.  A stage holds the codes
// [128 rows][128 B] (128B-swizzled), the scales [128 rows][16 B] and the
// activations: four 64-k column blocks of [NM rows][128 B], 128B-swizzled.
struct SmemLayout {
  int stages;
  int stage_bytes;
  int s_off;        // scales, within a stage
  int x_off;        // activations, within a stage
  int lut_off;      // 256 bf16 scale pairs
  int bar_off;      // mbarriers, abort flag, TMEM base
  int total;        // dynamic shared memory to request (with alignment slack)
};

__host__ __device__ constexpr int num_barriers(int stages, int ni) {
  return 2 * stages + 2 * ni * kSlotsPerGroup + 1;
}

__host__ __device__ constexpr SmemLayout make_layout(int nm, int ni, int stages) {
  SmemLayout l{};
  l.stages = stages;
  l.s_off = kRows * 128;
  l.x_off = align_up(l.s_off + kRows * 16, 1024);
  l.stage_bytes = align_up(l.x_off + nm * kStageK * 2, 1024);
  l.lut_off = stages * l.stage_bytes;
  l.bar_off = l.lut_off + 256 * 4;
  l.total = l.bar_off + num_barriers(stages, ni) * 8 + 16 + 1024;
  return l;
}

// The CTA's partial [128 rows][NM] lives in the ring with a row pitch of
// NM + 1 floats: a warp's stores (one row per thread) and the epilogue's
// loads (consecutive rows) then fall in distinct banks.
__host__ __device__ constexpr int part_pitch(int nm) { return nm + 1; }

// Receive area of the k-split reduction, after the partial: the partial
// values of this CTA's share of the outputs from every CTA of the cluster,
// [split][1 or 2][share] floats (two with SwiGLU, whose outputs have half
// the rows; shares rounded to even sizes), at most 128 NM + 8 kMaxSplit
// floats.
__host__ __device__ constexpr int recv_floats(int nm) { return kRows * nm + 8 * kMaxSplit; }

// The final exchange reuses the ring; it must fit.
__host__ __device__ constexpr bool layout_ok(const SmemLayout& l, int nm) {
  return l.stages >= 2 &&
         (kRows * part_pitch(nm) + recv_floats(nm)) * 4 <= l.stages * l.stage_bytes;
}

struct Params {
  void* y;              // [M, N] (or [M, N/2] with swiglu), bf16 or f32
  void* y_host;         // nullptr, or the same output again in host memory mapped
                        // into the device (the host-buffer entry point)
  int64_t M, N, K;
  float out_scale;      // fp32(2^10 / global_scale)
  float out_scale_up;   // the same for the up rows of SwiGLU (their own global scale)
  int stages_total;     // K / 256
  int split;            // CTAs per cluster along k
  int out_f32;          // 1: write f32 (before the bf16 rounding)
  int swiglu;           // 1: rows [0,N/2) gate, [N/2,N) up, y = silu(g)*u
  SmemLayout lay;
  SegScales seg;        // per-segment scales (seg.n == 0: out_scale for every column)
  unsigned int* err;    // device error word
};

// A wait whose outcome the whole warp shares: the warp-aligned tcgen05
// instructions after it need every lane converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

// Position of a stage in the ring (slot and barrier parity), walked forward
// stage by stage: the ring depth is a launch parameter, and a division by
// it per job measurably slowed the dequantisers.
struct RingPos {
  int stage = 0, slot = 0;
  uint32_t parity = 0;
  __device__ __forceinline__ void advance_to(int target, int depth) {
    for (; stage < target; ++stage)
      if (++slot == depth) {
        slot = 0;
        parity ^= 1u;
      }
  }
};

template <int NM, int NI>
__global__ void __launch_bounds__(Roles<NM, NI>::kThreads, Roles<NM, NI>::kCtasPerSm)
    gemv_bf16_kernel(const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_s,
                     const __grid_constant__ CUtensorMap tm_x, const Params p) {
  static_assert(NM == 16 || NM == 32, "MMA N is 16 or 32");
  using R = Roles<NM, NI>;
  constexpr int kThreads = R::kThreads;
  constexpr int kPitch = part_pitch(NM);
  const SmemLayout& L = p.lay;
  const int S = L.stages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base, formed by arithmetic on the shared array itself so
  // that every access through it stays a shared-memory access
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + L.lut_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);   // TMA landed
  // Stage consumed: every issuer has committed its last job of the stage
  // (one tcgen05.commit per stage and issuer); releases the ring slot.
  uint64_t* empty = full + S;
  uint64_t* a_full = empty + S;                  // [NI][3] TMEM weights written
  // [NI][3] the slot's MMAs have completed (one commit per job): releases
  // the TMEM slot to its group's dequantisers, so that the groups do not
  // wait for each other (a wait on the stage barrier had them in lockstep).
  uint64_t* a_empty = a_full + NI * kSlotsPerGroup;
  uint64_t* mma_done = a_empty + NI * kSlotsPerGroup;  // every MMA has completed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(mma_done + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = static_cast<int>(p.M);
  const int split = p.split;
  const int z = blockIdx.y;                                  // k-slice index
  const int st_begin = static_cast<int>((int64_t)p.stages_total * z / split);
  const int st_end = static_cast<int>((int64_t)p.stages_total * (z + 1) / split);
  const int n_stages = st_end - st_begin;
  // jobs of lane group i: i, i + NI, ... < 4 * n_stages
  const int n_jobs_total = kJobsPerStage * n_stages;

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

  for (int i = threadIdx.x; i < 256; i += kThreads) lut[i] = scale_pair_from_e4m3(i);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NI);
    }
    for (int a = 0; a < NI * kSlotsPerGroup; ++a) {
      mbar_init(&a_full[a], 4);
      mbar_init(&a_empty[a], 1);
    }
    mbar_init(mma_done, NI);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == R::kWarpMma) {
    tmem_alloc(tmem_slot, R::kTmemCols);
    tmem_relinquish();
  }
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
      const uint32_t tx =
          static_cast<uint32_t>(kRows * (kStageK / 2 + kStageK / 16) + NM * kStageK * 2);
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
        const int k0 = (st_begin + it) * kStageK;
#pragma unroll
        for (int q = 0; q < kJobsPerStage; ++q)
          tma_load_2d_hint(st + L.x_off + q * (NM * 128), &tm_x, &full[slot], k0 + kJobK * q, 0,
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
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
        }
      }
      // Drain: never leave a copy in flight into this CTA's shared memory.
      const int first = issued > S ? issued - S : 0;
      for (int it = first; it < issued; ++it) {
        volatile int no_abort = 0;
        if (!mbar_wait(&full[it % S], (it / S) & 1, &no_abort)) atomicOr(p.err, kErrWaitTimeout);
      }
    }
  } else if (warp < R::kWarpDeq) {
    // ------------------------------------------------------------ MMA issue
    // Issuer i takes jobs i, i + NI, ...: job j is k [64 (j % 4), +64) of
    // stage j / 4, four MMAs of K = 16 into accumulator i.  It commits each
    // job to the job's TMEM slot and, after its last job of a stage, to the
    // stage.
    const int gi = warp - R::kWarpMma;
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kRows, NM);
      const uint32_t d_tmem = tmem + R::kDCol + gi * NM;
      int n = 0, aslot = 0;
      uint32_t apar = 0;
      RingPos pos;
      for (int j = gi; j < n_jobs_total; j += NI, ++n) {
        const int q = j % kJobsPerStage;
        pos.advance_to(j / kJobsPerStage, S);
        const int slot = pos.slot;
        if (!mbar_wait(&full[slot], pos.parity, abort_flag)) break;
        if (!mbar_wait(&a_full[gi * kSlotsPerGroup + aslot], apar, abort_flag)) break;
        tc_fence_after_sync();
        const uint64_t b_desc0 =
            umma_desc_sw128(smem_addr(smem + slot * L.stage_bytes + L.x_off + q * (NM * 128)));
        const uint32_t a_tmem = tmem + (gi * kSlotsPerGroup + aslot) * kSlotCols;
#pragma unroll
        for (int kk = 0; kk < kJobK / 16; ++kk)
          umma_f16_tmem_a(d_tmem, a_tmem + kk * 8, b_desc0 + static_cast<uint64_t>((kk * 32) >> 4),
                          idesc, (n > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&a_empty[gi * kSlotsPerGroup + aslot]);
        if (q + NI >= kJobsPerStage) umma_commit(&empty[slot]);
        if (++aslot == kSlotsPerGroup) {
          aslot = 0;
          apar ^= 1u;
        }
      }
      // The accumulators are final once every MMA issued has completed.
      umma_commit(mma_done);
    }
  } else {
    // ------------------------------------------------------------ dequantisers
    // Warp (lane group gi, quadrant qd): lane = weight row 32 qd + lane = its
    // TMEM lane; for each job of the group it writes the row's 64 k as 32
    // bf16 pairs into the group's next TMEM slot: column 4i + p holds
    // k = 8i + p and 8i + p + 4, the order the bit trick yields (the job's
    // activations are permuted to match).
    const int dw = warp - R::kWarpDeq;
    const int gi = dw >> 2, qd = warp & 3;
    const int row = 32 * qd + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    int n = 0, aslot = 0;
    uint32_t epar = 0;          // parity of the slot's previous use
    RingPos pos;
    for (int j = gi; j < n_jobs_total; j += NI, ++n) {
      const int q = j % kJobsPerStage;
      pos.advance_to(j / kJobsPerStage, S);
      const int slot = pos.slot;
      if (!warp_wait(&full[slot], pos.parity, abort_flag)) break;
      if (n >= kSlotsPerGroup &&
          !warp_wait(&a_empty[gi * kSlotsPerGroup + aslot], epar, abort_flag))
        break;          // the slot's previous job (kSlotsPerGroup jobs back) not done
      uint8_t* st = smem + slot * L.stage_bytes;
      // The job's activations (64 k of NM rows) into the weights' k order:
      // within every 8 k, (k0, k4, k1, k5, k2, k6, k3, k7).  Both MMA
      // operands then list the k of each 8-k block in that same order, which
      // leaves every product and sum of the contraction as it was, and the
      // weights need no re-pairing after the bit trick.  A 16-byte chunk is 8
      // consecutive k of one row (the 128B swizzle moves whole chunks), so
      // the permutation is chunk-local; the job's four warps share it.
      {
        uint8_t* xq = st + L.x_off + q * (NM * 128);
#pragma unroll
        for (int c = 32 * qd + lane; c < NM * 8; c += 128) {
          const uint4 v = *reinterpret_cast<const uint4*>(xq + c * 16);
          *reinterpret_cast<uint4*>(xq + c * 16) =
              make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u),
                         prmt(v.y, v.w, 0x5410u), prmt(v.y, v.w, 0x7632u));
        }
        fence_proxy_async_smem();   // the tensor core reads the tile next
      }
      // 64 k = code chunks 2q, 2q+1 of the row's 128-byte swizzled line
      const uint4 w0 =
          *reinterpret_cast<const uint4*>(st + row * 128 + (((2 * q) ^ (row & 7)) << 4));
      const uint4 w1 =
          *reinterpret_cast<const uint4*>(st + row * 128 + (((2 * q + 1) ^ (row & 7)) << 4));
      // scales of the four 16-k blocks: bytes 4q .. 4q+3 of the row
      const uint32_t s4 = *reinterpret_cast<const uint32_t*>(st + L.s_off + row * 16 + 4 * q);
      const uint32_t S0 = lut[s4 & 0xFFu], S1 = lut[(s4 >> 8) & 0xFFu];
      const uint32_t S2 = lut[(s4 >> 16) & 0xFFu], S3 = lut[s4 >> 24];
      const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const uint32_t sc[4] = {S0, S1, S2, S3};
      uint32_t out[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) dequant8_strided(words[i], sc[i >> 1], &out[4 * i]);
      tc_fence_after_sync();
      tmem_st_32cols(t_lane + (gi * kSlotsPerGroup + aslot) * kSlotCols, out);
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[gi * kSlotsPerGroup + aslot]);
      if (++aslot == kSlotsPerGroup) {
        aslot = 0;
        if (n + 1 > kSlotsPerGroup) epar ^= 1u;   // from the second round on
      }
    }
  }

  // ---------------------------------------------------------------- accumulators
  // The first quartet reads the NI accumulators (lane = weight row) once
  // every MMA has completed, and leaves their sum in the ring as the CTA's
  // partial [128 rows][NM].
  {
    volatile int no_abort = 0;
    const bool first_quartet = warp >= R::kWarpDeq && warp < R::kWarpDeq + 4;
    bool ok = true;
    if (first_quartet) ok = warp_wait(mma_done, 0, &no_abort);
    if (first_quartet && !ok && lane == 0) atomicOr(p.err, kErrWaitTimeout);
    tc_fence_before_sync();
    __syncthreads();            // every role is done with the ring
    if (first_quartet && ok) {
      tc_fence_after_sync();
      const int qd = warp & 3;
      const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * qd) << 16) + R::kDCol;
      float* part = reinterpret_cast<float*>(smem);
      const int row = 32 * qd + lane;
#pragma unroll
      for (int h = 0; h < NM / 16; ++h) {
        float sum[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) sum[c] = 0.f;
#pragma unroll
        for (int gi = 0; gi < NI; ++gi) {
          uint32_t d[16];
          tmem_ld_16cols(t_lane + gi * NM + 16 * h, d);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) sum[c] += __uint_as_float(d[c]);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (16 * h + c < M) part[row * kPitch + 16 * h + c] = sum[c];
      }
    }
  }
  if (*abort_flag && threadIdx.x == 0) atomicOr(p.err, kErrWaitTimeout);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == R::kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, R::kTmemCols);
  }
  float* part = reinterpret_cast<float*>(smem);

  // ---------------------------------------------------------------- epilogue
  // Output item i = (activation row i / Rn, weight row i % Rn of the CTA).
  // Items go in pairs (i even; Rn is even, so both are of one activation
  // row): one word stored per pair.
  const int Rn = p.swiglu ? kHalfRows : kRows;           // outputs per activation row
  const int shift = p.swiglu ? 6 : 7;                    // log2(Rn)
  const int items = Rn * M;
  const int nv = p.swiglu ? 2 : 1;                       // partial values per item
  const int64_t n_base = static_cast<int64_t>(blockIdx.x) * Rn;
  const int64_t n_out = p.swiglu ? p.N / 2 : p.N;
  // value c of item i in this CTA's partial (c = 1: SwiGLU's up row)
  auto local_part = [&](int i, int c) {
    return part[((c ? kHalfRows : 0) + (i & (Rn - 1))) * kPitch + (i >> shift)];
  };
  // outputs i and i + 1 from their sums v (the row, or SwiGLU's gate row)
  // and u (SwiGLU's up row), both before the global scale
  auto emit2 = [&](int i, float v0, float v1, float u0, float u1) {
    const int m = i >> shift, jr = i & (Rn - 1);
    float y0 = v0 * (p.seg.n ? seg_scale(p.seg, n_base + jr) : p.out_scale);
    float y1 = v1 * (p.seg.n ? seg_scale(p.seg, n_base + jr + 1) : p.out_scale);
    if (p.swiglu) {
      y0 = silu_mul(y0, u0 * p.out_scale_up);
      y1 = silu_mul(y1, u1 * p.out_scale_up);
    }
    const int64_t off = static_cast<int64_t>(m) * n_out + n_base + jr;   // even
    if (p.out_f32) {
      *reinterpret_cast<float2*>(static_cast<float*>(p.y) + off) = make_float2(y0, y1);
      if (p.y_host)
        *reinterpret_cast<float2*>(static_cast<float*>(p.y_host) + off) = make_float2(y0, y1);
    } else {
      const uint32_t yb = f32x2_to_bf16x2(y0, y1);
      *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.y) + off) = yb;
      if (p.y_host) *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.y_host) + off) = yb;
    }
  };
  if (split == 1) {
    __syncthreads();
    for (int i = 2 * threadIdx.x; i < items; i += 2 * kThreads)
      emit2(i, local_part(i, 0), local_part(i + 1, 0), p.swiglu ? local_part(i, 1) : 0.f,
            p.swiglu ? local_part(i + 1, 1) : 0.f);
    return;
  }
  // k split: CTA z owns the items [begin(z), begin(z + 1)) (even bounds, so
  // that pairs stay whole).  Each CTA pushes its partial values of the other
  // CTAs' items into their receive areas (remote stores, so no thread waits
  // on a remote round trip), one cluster barrier makes them visible, and
  // each CTA adds its own items' values in rank order, from local shared
  // memory.  (Reconverge each warp before a cluster barrier: it is a
  // warp-aligned op.)
  auto begin = [&](int r) { return static_cast<int>((int64_t)items * r / split) & ~1; };
  const int share_max = ((items + split - 1) / split + 3) & ~1;   // even, >= every share
  float* recv = part + kRows * kPitch;                   // [split][nv][share_max]
  __syncwarp();
  cluster_sync();     // every partial is final and every ring is free
  for (int r = 0; r < split; ++r) {
    if (r == z) continue;
    const int b = begin(r), e = begin(r + 1);
    const uint32_t dst = map_to_rank(smem_addr(recv), static_cast<uint32_t>(r));
    for (int i = b + 2 * threadIdx.x; i < e; i += 2 * kThreads)
      for (int c = 0; c < nv; ++c)
        st_cluster_f32x2(dst + 4u * static_cast<uint32_t>((z * nv + c) * share_max + (i - b)),
                         local_part(i, c), local_part(i + 1, c));
  }
  __syncwarp();
  cluster_sync();     // every push has landed; nothing reads remote memory after this
  const int b = begin(z), e = begin(z + 1);
  for (int i = b + 2 * threadIdx.x; i < e; i += 2 * kThreads) {
    float v0 = 0.f, v1 = 0.f, u0 = 0.f, u1 = 0.f;
    for (int q = 0; q < split; ++q) {
      const float* rv = recv + (q * nv) * share_max + (i - b);
      v0 += q == z ? local_part(i, 0) : rv[0];
      v1 += q == z ? local_part(i + 1, 0) : rv[1];
      if (p.swiglu) {
        u0 += q == z ? local_part(i, 1) : rv[share_max];
        u1 += q == z ? local_part(i + 1, 1) : rv[share_max + 1];
      }
    }
    emit2(i, v0, v1, u0, u1);
  }
}

}  // namespace gemvbf
}  // namespace nvfp4
