// smallm.cuh -- NVFP4 W4A16 linear for few activation rows (M <= 32):
// decode (M = 1), speculative verify (M = K+1, FlashRT docs section 3) and
// small continuous batches.  At these sizes the layer is bound by streaming
// the packed weights and scales from HBM once; every design choice below is
// about keeping that stream at full rate.
//
//  * One CTA owns 64 weight rows and a contiguous range of k.  A producer
//    warp streams 256-k stages (packed weights, block scales, activations)
//    into a shared-memory ring with TMA; an L2 evict-first hint keeps the
//    once-read weights from displacing the activations.
//  * Four consumer warps each take a 64-k quarter of every stage for all 64
//    rows.  The weights are dequantised in registers straight into the A
//    fragments of the register-fed m16n8k16 bf16 warp MMA (weights as the
//    16-row operand, activations as the 8-wide one), so the dequantised
//    weights never touch shared memory.  (The tcgen05 MMA reads both of its
//    operands from shared memory or TMEM; at N = 8..32 that round trip would
//    cost more shared-memory bandwidth than the weight stream itself.)
//  * k is permuted inside each thread's 16-element block so that the cheap
//    (k, k+4) pairing of the dequantiser is used unchanged; the activation
//    fragments are built with the same permutation, so the dot products are
//    unchanged.
//  * Split-K: CTAs that share rows but not k form one thread-block cluster.
//    Partials are reduced warp -> CTA in shared memory and then across the
//    cluster through distributed shared memory.  No global workspace, no
//    atomics, no spin-waits on other CTAs.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace smallm {

constexpr int kRows = 64;             // weight rows per CTA
constexpr int kHalfRows = 32;         // rows per TMA box (two boxes per stage)
constexpr int kStageK = 256;          // k per pipeline stage
constexpr int kConsumerWarps = 4;     // one 64-k quarter of a stage each
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kWBytes = kRows * kStageK / 2;       // 8 KB packed weights
constexpr int kSBytes = kRows * kStageK / 16;      // 1 KB block scales
constexpr int kSOff = kWBytes;
constexpr int kXOff = kWBytes + kSBytes;           // 9 KB, 1024-aligned

template <int MT>
struct Layout {
  static constexpr int kXBoxBytes = MT * 8 * 128;            // 64 k x MT*8 rows
  static constexpr int kStageBytes = kXOff + kConsumerWarps * kXBoxBytes;
  static constexpr int kStages = (MT <= 2) ? 4 : 4;
  static constexpr int kRingBytes = kStageBytes * kStages;
  static constexpr int kRedFloats = kConsumerWarps * kRows * MT * 8;
  static constexpr int kPartOff = kRingBytes;                // CTA partials
  static constexpr int kPartBytes = kRows * MT * 8 * 4;
  static constexpr int kLutOff = kPartOff + kPartBytes;
  static constexpr int kBarOff = kLutOff + 256 * 4;
  static constexpr int kSmemBytes = kBarOff + 2 * kStages * 8 + 16 + 1024;  // + align
  static_assert(kRedFloats * 4 <= kRingBytes, "reduction buffer must fit the ring");
};

struct Params {
  void* y;              // [M, N] (or [M, N/2] with swiglu), bf16 or f32
  int64_t M, N, K;
  float global_scale;
  int stages_total;     // K / 256
  int split;            // CTAs per cluster along k
  int out_f32;          // 1: write f32 (before the bf16 rounding)
  int swiglu;           // 1: rows [0,N/2) gate, [N/2,N) up, y = silu(g)*u
  unsigned int* err;    // device error word
};

template <int MT>
__global__ void __launch_bounds__(kThreads)
    smallm_kernel(const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_x, const Params p) {
  using L = Layout<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + L::kLutOff);
  float* part = reinterpret_cast<float*>(smem + L::kPartOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + L::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + L::kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = p.split;
  const int z = blockIdx.y;                                  // k-slice index
  const int st_begin = static_cast<int>((int64_t)p.stages_total * z / split);
  const int st_end = static_cast<int>((int64_t)p.stages_total * (z + 1) / split);
  const int n_stages = st_end - st_begin;

  // weight rows of this CTA: two 32-row boxes
  int row0, row1;
  if (p.swiglu) {
    row0 = blockIdx.x * kHalfRows;                               // gate
    row1 = static_cast<int>(p.N / 2) + blockIdx.x * kHalfRows;   // up
  } else {
    row0 = blockIdx.x * kRows;
    row1 = row0 + kHalfRows;
  }

  for (int i = threadIdx.x; i < 256; i += kThreads) lut[i] = scale_pair_from_e4m3(i);
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_s);
      prefetch_tensormap(&tm_x);
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      int issued = 0;
      for (int it = 0; it < n_stages; ++it) {
        const int slot = it % L::kStages;
        const uint32_t par = ((it / L::kStages) & 1) ^ 1;
        if (!mbar_wait(&empty[slot], par, abort_flag)) break;
        uint8_t* st = smem + slot * L::kStageBytes;
        mbar_arrive_expect_tx(&full[slot], L::kStageBytes);
        const int k0 = (st_begin + it) * kStageK;
        tma_load_2d_hint(st, &tm_w, &full[slot], k0 / 2, row0, pol_stream);
        tma_load_2d_hint(st + kWBytes / 2, &tm_w, &full[slot], k0 / 2, row1, pol_stream);
        tma_load_2d_hint(st + kSOff, &tm_s, &full[slot], k0 / 16, row0, pol_stream);
        tma_load_2d_hint(st + kSOff + kSBytes / 2, &tm_s, &full[slot], k0 / 16, row1,
                         pol_stream);
#pragma unroll
        for (int q = 0; q < kConsumerWarps; ++q)
          tma_load_2d_hint(st + kXOff + q * L::kXBoxBytes, &tm_x, &full[slot], k0 + 64 * q,
                           0, pol_keep);
        ++issued;
      }
      // Drain: never leave a copy in flight into this CTA's shared memory.
      const int first = issued > L::kStages ? issued - L::kStages : 0;
      for (int it = first; it < issued; ++it) {
        volatile int no_abort = 0;
        if (!mbar_wait(&full[it % L::kStages], (it / L::kStages) & 1, &no_abort))
          atomicOr(p.err, kErrWaitTimeout);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    float acc[4][MT][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][mt][c] = 0.f;

    for (int it = 0; it < n_stages; ++it) {
      const int slot = it % L::kStages;
      const uint32_t par = (it / L::kStages) & 1;
      if (!mbar_wait(&full[slot], par, abort_flag)) break;
      const uint8_t* st = smem + slot * L::kStageBytes;

      // Activation fragments: x row (8*mt + g), elements [16t, 16t+16) of
      // this warp's 64-k box, paired (k, k+4) like the weights.
      uint32_t bx[MT][8];
      const uint8_t* xb = st + kXOff + warp * L::kXBoxBytes;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int m = mt * 8 + g;
        const uint8_t* row = xb + m * 128;
        const uint4 c0 = *reinterpret_cast<const uint4*>(row + (((2 * t) ^ (m & 7)) << 4));
        const uint4 c1 =
            *reinterpret_cast<const uint4*>(row + (((2 * t + 1) ^ (m & 7)) << 4));
        bx[mt][0] = prmt(c0.x, c0.z, 0x5410u);
        bx[mt][1] = prmt(c0.x, c0.z, 0x7632u);
        bx[mt][2] = prmt(c0.y, c0.w, 0x5410u);
        bx[mt][3] = prmt(c0.y, c0.w, 0x7632u);
        bx[mt][4] = prmt(c1.x, c1.z, 0x5410u);
        bx[mt][5] = prmt(c1.x, c1.z, 0x7632u);
        bx[mt][6] = prmt(c1.y, c1.w, 0x5410u);
        bx[mt][7] = prmt(c1.y, c1.w, 0x7632u);
      }

      const int chunk = 2 * warp + (t >> 1);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        // MMA rows g and g+8 are weight rows 16r+2g and 16r+2g+1 (this
        // choice makes the swizzled loads below bank-conflict free).
        const int ra = 16 * r + 2 * g, rb = ra + 1;
        const uint2 wa = *reinterpret_cast<const uint2*>(
            st + ra * 128 + ((chunk ^ (ra & 7)) << 4) + ((t & 1) << 3));
        const uint2 wb = *reinterpret_cast<const uint2*>(
            st + rb * 128 + ((chunk ^ (rb & 7)) << 4) + ((t & 1) << 3));
        const uint32_t sa = lut[st[kSOff + ra * 16 + 4 * warp + t]];
        const uint32_t sb = lut[st[kSOff + rb * 16 + 4 * warp + t]];
        uint32_t pa[8], pb[8];
        dequant8_strided(wa.x, sa, &pa[0]);
        dequant8_strided(wa.y, sa, &pa[4]);
        dequant8_strided(wb.x, sb, &pb[0]);
        dequant8_strided(wb.y, sb, &pb[4]);
#pragma unroll
        for (int s = 0; s < 4; ++s)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            mma_bf16_16816(acc[r][mt], pa[2 * s], pb[2 * s], pa[2 * s + 1], pb[2 * s + 1],
                           bx[mt][2 * s], bx[mt][2 * s + 1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // Warp partials -> ring (free now: every stage has been consumed once
    // all four warps pass the barrier below).
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    float* red = reinterpret_cast<float*>(smem);
    constexpr int C = MT * 8;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int ra = 16 * r + 2 * g, col = mt * 8 + 2 * t;
        float* base = red + warp * kRows * C;
        base[ra * C + col] = acc[r][mt][0];
        base[ra * C + col + 1] = acc[r][mt][1];
        base[(ra + 1) * C + col] = acc[r][mt][2];
        base[(ra + 1) * C + col + 1] = acc[r][mt][3];
      }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    for (int i = threadIdx.x; i < kRows * C; i += kConsumerWarps * 32) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) s += red[w * kRows * C + i];
      part[i] = s;
    }
  }

  if (*abort_flag && threadIdx.x == 0) atomicOr(p.err, kErrWaitTimeout);

  // ---------------------------------------------------------------- epilogue
  // Every CTA of the cluster finishes its partial; CTA z then reduces a
  // 1/split share of the outputs across the cluster's shared memories.
  cluster_sync();
  {
    constexpr int C = MT * 8;
    const int M = static_cast<int>(p.M);
    const int R = p.swiglu ? kHalfRows : kRows;          // outputs per CTA row
    const int items = R * M;
    const int i0 = static_cast<int>((int64_t)items * z / split);
    const int i1 = static_cast<int>((int64_t)items * (z + 1) / split);
    const uint32_t part_local = smem_addr(part);
    const int64_t n_out = p.swiglu ? p.N / 2 : p.N;
    const int64_t n_base = static_cast<int64_t>(blockIdx.x) * R;
    for (int i = i0 + threadIdx.x; i < i1; i += kThreads) {
      const int m = i / R, j = i % R;
      float v = 0.f, u = 0.f;
      for (int q = 0; q < split; ++q) {
        const uint32_t base = map_to_rank(part_local, q);
        v += ld_cluster_f32(base + 4u * (j * C + m));
        if (p.swiglu) u += ld_cluster_f32(base + 4u * ((kHalfRows + j) * C + m));
      }
      float yv = __fdiv_rn(v * kWeightPow2, p.global_scale);
      if (p.swiglu) {
        const float up = __fdiv_rn(u * kWeightPow2, p.global_scale);
        yv = yv / (1.0f + expf(-yv)) * up;
      }
      const int64_t off = static_cast<int64_t>(m) * n_out + n_base + j;
      if (p.out_f32)
        static_cast<float*>(p.y)[off] = yv;
      else
        static_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(yv);
    }
  }
  cluster_sync();   // keep every partial alive until all readers are done
}

}  // namespace smallm
}  // namespace nvfp4
