// tcgemm.cuh -- NVFP4 W4A16 linear for many activation rows (prefill;
// FlashRT docs section 4, chunked prefill and the fused MLP gate/up GEMM).
// Here the layer is a dense contraction and runs on the tcgen05 tensor cores
// with the accumulator in TMEM.
//
// Tile: 128 weight rows x 256 activation rows, 64 k per pipeline stage.  The
// weights are the MMA's 128-row A operand and the activations its 256-wide
// B operand ("swap AB"): each dequantised weight element then serves 256
// activation rows, halving the dequantisation work per flop compared with
// the other orientation.  D = W x^T sits in TMEM as 128 lanes (weight rows)
// x 256 f32 columns (activation rows).
//
// Warp roles (320 threads):
//   warp 0      TMA producer: activation tile (128B-swizzled, the B operand
//               as-is), packed weights (32B-swizzled) and block scales;
//   warp 1      TMEM allocation and the single MMA-issuing thread;
//   warps 2..9  dequantise packed weights to bf16 straight into the A
//               operand's 128B-swizzled K-major layout; after the k loop
//               they drain TMEM (tcgen05.ld), apply 2^10 / global_scale and
//               the optional SwiGLU, and store bf16 (or f32).
// All waits are mbarrier waits with a time limit (see ptx.cuh).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace tcgemm {

constexpr int kTileW = 128;                 // weight rows per tile (MMA M)
constexpr int kTileX = 256;                 // activation rows per tile (MMA N)
constexpr int kStageK = 64;                 // k per stage (one 128 B swizzle row)
constexpr int kUmmaK = 16;
constexpr int kStages = 4;
constexpr int kDequantWarps = 8;
constexpr int kThreads = (2 + kDequantWarps) * 32;
constexpr int kXBytes = kTileX * kStageK * 2;          // 32 KB
constexpr int kABytes = kTileW * kStageK * 2;          // 16 KB
constexpr int kRawBytes = kTileW * kStageK / 2;        // 4 KB
constexpr int kSclBytes = kTileW * 16;                 // 2 KB (16 B per row)
constexpr int kXOff = 0;
constexpr int kAOff = kXBytes;
constexpr int kRawOff = kAOff + kABytes;
constexpr int kSclOff = kRawOff + kRawBytes;
constexpr int kStageBytes = kSclOff + kSclBytes;      // 54 KB, 1024-multiple
constexpr int kTxBytes = kXBytes + kRawBytes + kSclBytes;
constexpr int kLutOff = kStages * kStageBytes;
constexpr int kBarOff = kLutOff + 256 * 4;
constexpr int kNumBars = 3 * kStages + 1;
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
constexpr uint32_t kTmemCols = 256;
static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");

struct Params {
  void* y;
  int64_t M, N, K;
  float out_scale;      // fp32(2^10 / global_scale)
  int out_f32;
  int swiglu;          // tile = 64 gate rows + the 64 matching up rows
  unsigned int* err;
};

__global__ void __launch_bounds__(kThreads, 1)
    tcgemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_s, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + kLutOff);
  uint64_t* tma_full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* a_full = tma_full + kStages;
  uint64_t* empty = a_full + kStages;
  uint64_t* acc_full = empty + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(acc_full + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_stages = static_cast<int>(p.K / kStageK);
  const int m_tile = blockIdx.y * kTileX;
  const int bw = blockIdx.x;
  // weight rows feeding A rows [0,64) and [64,128)
  int wrow0, wrow1;
  if (p.swiglu) {
    wrow0 = bw * 64;                                   // gate rows
    wrow1 = static_cast<int>(p.N / 2) + bw * 64;       // matching up rows
  } else {
    wrow0 = bw * kTileW;
    wrow1 = wrow0 + 64;
  }

  for (int i = threadIdx.x; i < 256; i += kThreads) lut[i] = scale_pair_from_e4m3(i);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tma_full[s], 1);
      mbar_init(&a_full[s], kDequantWarps);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_acc = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_x);
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_s);
      const uint64_t pol_w = policy_evict_last();    // weights: reused by M tiles
      auto issue_weights = [&](int it, int slot) {
        uint8_t* st = smem + slot * kStageBytes;
        const int k0 = it * kStageK;
        tma_load_2d_hint(st + kRawOff, &tm_w, &tma_full[slot], k0 / 2, wrow0, pol_w);
        tma_load_2d_hint(st + kRawOff + kRawBytes / 2, &tm_w, &tma_full[slot], k0 / 2, wrow1,
                         pol_w);
        const int sx = (k0 / 16) & ~15;
        tma_load_2d_hint(st + kSclOff, &tm_s, &tma_full[slot], sx, wrow0, pol_w);
        tma_load_2d_hint(st + kSclOff + kSclBytes / 2, &tm_s, &tma_full[slot], sx, wrow1,
                         pol_w);
      };
      auto issue_acts = [&](int it, int slot) {
        tma_load_2d(smem + slot * kStageBytes + kXOff, &tm_x, &tma_full[slot], it * kStageK,
                    m_tile);
      };
      // Weights first (independent of the preceding kernel in the stream),
      // activations after the programmatic-dependent-launch wait.
      const int pre = n_stages < kStages ? n_stages : kStages;
      for (int it = 0; it < pre; ++it) {
        mbar_arrive_expect_tx(&tma_full[it], kTxBytes);
        issue_weights(it, it);
      }
      griddep_wait();
      for (int it = 0; it < pre; ++it) issue_acts(it, it);
      int issued = pre;
      for (int it = pre; it < n_stages; ++it) {
        const int slot = it % kStages;
        if (!mbar_wait(&empty[slot], ((it / kStages) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&tma_full[slot], kTxBytes);
        issue_weights(it, slot);
        issue_acts(it, slot);
        ++issued;
      }
      const int first = issued > kStages ? issued - kStages : 0;
      for (int it = first; it < issued; ++it) {
        volatile int no_abort = 0;
        if (!mbar_wait(&tma_full[it % kStages], (it / kStages) & 1, &no_abort))
          atomicOr(p.err, kErrWaitTimeout);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kTileW, kTileX);
      bool ok = true;
      for (int it = 0; it < n_stages && ok; ++it) {
        const int slot = it % kStages;
        const uint32_t par = (it / kStages) & 1;
        ok = mbar_wait(&tma_full[slot], par, abort_flag) &&
             mbar_wait(&a_full[slot], par, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t st = smem_addr(smem + slot * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kStageK / kUmmaK; ++kk) {
          const uint64_t a_desc = umma_desc_sw128(st + kAOff + kk * kUmmaK * 2);
          const uint64_t b_desc = umma_desc_sw128(st + kXOff + kk * kUmmaK * 2);
          umma_bf16(tmem_acc, a_desc, b_desc, idesc, (it | kk) != 0);
        }
        umma_commit(&empty[slot]);
      }
      umma_commit(acc_full);
    }
  } else {
    // ---------------------------------------------------------- dequantisers
    const int d = warp - 2;                       // 0..7
    const int r = (d & 3) * 32 + lane;            // raw weight row in the tile
    const int h = d >> 2;                         // k half: [32h, 32h+32)
    // A row: identity, or interleaved gate/up pairs (2j gate, 2j+1 up) so
    // that one warp holds both halves of every SwiGLU output.
    const int arow = p.swiglu ? (r < 64 ? 2 * r : 2 * (r - 64) + 1) : r;
    const uint32_t a_row_off = (arow >> 3) * 1024 + (arow & 7) * 128;
    for (int it = 0; it < n_stages; ++it) {
      const int slot = it % kStages;
      if (!mbar_wait(&tma_full[slot], (it / kStages) & 1, abort_flag)) break;
      uint8_t* st = smem + slot * kStageBytes;
      const uint4 raw = *reinterpret_cast<const uint4*>(
          st + kRawOff + r * 32 + ((h ^ ((r >> 2) & 1)) << 4));
      const int blk = ((it * kStageK) / 16) & 15;  // block index within the 16 B row
      const uint8_t* srow = st + kSclOff + r * 16 + blk + 2 * h;
      const uint32_t s0 = lut[srow[0]], s1 = lut[srow[1]];
      const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        uint32_t pr[4], cons[4];
        dequant8_strided(words[wi], wi < 2 ? s0 : s1, pr);
        pair_consecutive(pr, cons);
        const int chunk = 4 * h + wi;             // 16 B = 8 k of the 128 B row
        *reinterpret_cast<uint4*>(st + kAOff + a_row_off + ((chunk ^ (arow & 7)) << 4)) =
            make_uint4(cons[0], cons[1], cons[2], cons[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[slot]);
    }

    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quarter
    const int colhalf = d >> 2;                   // activation rows [128c, 128c+128)
    if (warp == 2 && lane == 0) griddep_launch_dependents();
    // Warp-uniform (and reconverged) before the warp-aligned tcgen05.ld.
    const bool have_acc = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag));
    tc_fence_after_sync();
    if (have_acc) {
      const int lane_row = 32 * q + lane;         // A row = TMEM lane
      const int64_t n_out = p.swiglu ? p.N / 2 : p.N;
      int64_t ncol;
      if (p.swiglu)
        ncol = static_cast<int64_t>(bw) * 64 + (lane_row >> 1);
      else
        ncol = static_cast<int64_t>(bw) * kTileW + lane_row;
#pragma unroll 1
      for (int c0 = colhalf * 128; c0 < colhalf * 128 + 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32cols(tmem_acc + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int m = m_tile + c0 + i;
          float yv = __uint_as_float(v[i]) * p.out_scale;
          if (p.swiglu) {
            const float up = __shfl_xor_sync(0xffffffffu, yv, 1);
            yv = silu_mul(yv, up);
            if ((lane & 1) || m >= p.M) continue;
          } else if (m >= p.M) {
            continue;
          }
          const int64_t off = static_cast<int64_t>(m) * n_out + ncol;
          if (p.out_f32)
            static_cast<float*>(p.y)[off] = yv;
          else
            static_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(yv);
        }
      }
    }
  }

  if (*abort_flag && threadIdx.x == 0) atomicOr(p.err, kErrWaitTimeout);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_acc, kTmemCols);
  }
}

}  // namespace tcgemm
}  // namespace nvfp4
