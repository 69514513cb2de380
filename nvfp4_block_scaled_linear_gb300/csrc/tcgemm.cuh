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
// Persistent: one CTA per SM, each walking the output tiles with the grid as
// its stride, and the accumulator double-buffered in TMEM (2 x 256 columns)
// so that the epilogue of one tile overlaps the k loop of the next.  Tile
// order: bands of `band` activation tiles (42 MB of a 5120-wide x for 16
// tiles), within a band weight tile by weight tile, the band's activation
// tiles innermost.  The CTAs working at one time then take a few weight
// tiles, each shared by `band` of them, and the whole band's activations,
// which the copies mark evict-last so that they stay in L2 while the band's
// weights stream past once; the results are stored as streaming data.
//
// Warp roles (448 threads):
//   warp 0      TMA producer: activation tile (128B-swizzled, the B operand
//               as-is), packed weights (32B-swizzled) and block scales;
//   warp 1      TMEM allocation and the single MMA-issuing thread;
//   warps 2..9  dequantise packed weights to bf16 straight into the A
//               operand's 128B-swizzled K-major layout;
//   warps 10..13 epilogue: drain a finished accumulator (tcgen05.ld), apply
//               2^10 / global_scale and the optional SwiGLU, store bf16 (or
//               f32), and hand the accumulator back to the MMA issuer.
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
constexpr int kEpiWarps = 4;
constexpr int kWarpDeq = 2;
constexpr int kWarpEpi = kWarpDeq + kDequantWarps;     // 10
constexpr int kThreads = (kWarpEpi + kEpiWarps) * 32;  // 448
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
constexpr int kNumBars = 3 * kStages + 5;
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
constexpr uint32_t kAccCols = 256;          // one accumulator: 256 f32 columns
constexpr uint32_t kTmemCols = 2 * kAccCols;  // double-buffered
static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");

struct Params {
  void* y;
  int64_t M, N, K;
  float out_scale;      // fp32(2^10 / global_scale)
  float out_scale_up;   // the same for the up rows of SwiGLU (their own global scale)
  int out_f32;
  int swiglu;          // tile = 64 gate rows + the 64 matching up rows
  int tiles_w;         // weight tiles (N / 128)
  int tiles_x;         // activation tiles (M / 256, rounded up)
  int tiles_total;     // weight tiles x activation tiles
  int band;            // activation tiles per band of the tile order
  SegScales seg;        // per-segment scales (seg.n == 0: out_scale for every column)
  unsigned int* err;
};

__global__ void __launch_bounds__(kThreads, 1)
    tcgemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_s, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base, formed by arithmetic on the shared array itself so
  // that every access through it stays a shared-memory access
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + kLutOff);
  uint64_t* tma_full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* a_full = tma_full + kStages;
  uint64_t* empty = a_full + kStages;
  uint64_t* acc_full = empty + kStages;      // [2] accumulator b holds a finished tile
  uint64_t* acc_empty = acc_full + 2;        // [2] accumulator b drained by the epilogue
  uint64_t* mma_done = acc_empty + 2;        // every MMA issued has completed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(mma_done + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_stages = static_cast<int>(p.K / kStageK);
  // This CTA's tiles: t = blockIdx.x + i * gridDim.x, i < my_tiles.  Tile t
  // lies in band t / (tiles_w * band); within the band, weight tile by
  // weight tile, activation tiles innermost (the last band may be narrower).
  const int grid = static_cast<int>(gridDim.x);
  const int my_tiles = static_cast<int>(blockIdx.x) < p.tiles_total
                           ? (p.tiles_total - 1 - static_cast<int>(blockIdx.x)) / grid + 1
                           : 0;
  auto tile_of = [&](int i, int& bw, int& m_tile) {
    const int t = static_cast<int>(blockIdx.x) + i * grid;
    const int per_band = p.tiles_w * p.band;
    const int band = t / per_band;
    const int r = t - band * per_band;
    const int a0 = band * p.band;
    const int width = min(p.band, p.tiles_x - a0);
    bw = r / width;
    m_tile = (a0 + (r - bw * width)) * kTileX;
  };
  // weight rows feeding A rows [0,64) and [64,128) of weight tile bw
  auto wrows = [&](int bw, int& wrow0, int& wrow1) {
    if (p.swiglu) {
      wrow0 = bw * 64;                                   // gate rows
      wrow1 = static_cast<int>(p.N / 2) + bw * 64;       // matching up rows
    } else {
      wrow0 = bw * kTileW;
      wrow1 = wrow0 + 64;
    }
  };

  for (int i = threadIdx.x; i < 256; i += kThreads) lut[i] = scale_pair_from_e4m3(i);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tma_full[s], 1);
      mbar_init(&a_full[s], kDequantWarps);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    mbar_init(mma_done, 1);
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
  const uint32_t tmem_base = *tmem_slot;
  // One CTA per SM: a dependent kernel's CTAs only start as these exit.
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int total_stages = my_tiles * n_stages;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_x);
      prefetch_tensormap(&tm_w);
      prefetch_tensormap(&tm_s);
      // activations: reused by every weight tile of their band; weights:
      // read by the band's CTAs at about the same time, then not again
      const uint64_t pol_x = policy_evict_last();
      // Cursor over (tile i, stage it): the single producer thread must not
      // spend its stage budget on divisions, so tile coordinates change only
      // at tile boundaries.
      struct Cursor {
        int i, it, m_tile, wrow0, wrow1;
      };
      auto start_tile = [&](Cursor& c) {
        int bw;
        tile_of(c.i, bw, c.m_tile);
        wrows(bw, c.wrow0, c.wrow1);
      };
      auto advance = [&](Cursor& c) {
        if (++c.it == n_stages) {
          c.it = 0;
          if (++c.i < my_tiles) start_tile(c);
        }
      };
      auto issue_weights = [&](const Cursor& c, int slot) {
        uint8_t* st = smem + slot * kStageBytes;
        const int k0 = c.it * kStageK;
        tma_load_2d(st + kRawOff, &tm_w, &tma_full[slot], k0 / 2, c.wrow0);
        tma_load_2d(st + kRawOff + kRawBytes / 2, &tm_w, &tma_full[slot], k0 / 2, c.wrow1);
        const int sx = (k0 / 16) & ~15;
        tma_load_2d(st + kSclOff, &tm_s, &tma_full[slot], sx, c.wrow0);
        tma_load_2d(st + kSclOff + kSclBytes / 2, &tm_s, &tma_full[slot], sx, c.wrow1);
      };
      auto issue_acts = [&](const Cursor& c, int slot) {
        tma_load_2d_hint(smem + slot * kStageBytes + kXOff, &tm_x, &tma_full[slot],
                         c.it * kStageK, c.m_tile, pol_x);
      };
      Cursor cur{0, 0, 0, 0, 0};
      if (my_tiles > 0) start_tile(cur);
      // Weights first (independent of the preceding kernel in the stream),
      // activations after the programmatic-dependent-launch wait.
      const int pre = total_stages < kStages ? total_stages : kStages;
      const Cursor first_cur = cur;
      for (int g = 0; g < pre; ++g) {
        mbar_arrive_expect_tx(&tma_full[g], kTxBytes);
        issue_weights(cur, g);
        advance(cur);
      }
      griddep_wait();
      Cursor acts_cur = first_cur;
      for (int g = 0; g < pre; ++g) {
        issue_acts(acts_cur, g);
        advance(acts_cur);
      }
      int issued = pre;
      int slot = pre == kStages ? 0 : pre;
      uint32_t par = pre == kStages ? 0u : 1u;
      for (int g = pre; g < total_stages; ++g) {
        if (!mbar_wait(&empty[slot], par, abort_flag)) break;
        mbar_arrive_expect_tx(&tma_full[slot], kTxBytes);
        issue_weights(cur, slot);
        issue_acts(cur, slot);
        advance(cur);
        ++issued;
        if (++slot == kStages) {
          slot = 0;
          par ^= 1u;
        }
      }
      const int first = issued > kStages ? issued - kStages : 0;
      for (int g = first; g < issued; ++g) {
        volatile int no_abort = 0;
        if (!mbar_wait(&tma_full[g % kStages], (g / kStages) & 1, &no_abort))
          atomicOr(p.err, kErrWaitTimeout);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kTileW, kTileX);
      bool ok = true;
      int slot = 0;
      uint32_t par = 0;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int b = i & 1;
        // the epilogue has drained accumulator b (tile i - 2)
        ok = mbar_wait(&acc_empty[b], ((i >> 1) & 1) ^ 1u, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t tmem_acc = tmem_base + b * kAccCols;
        for (int it = 0; it < n_stages; ++it) {
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
          if (++slot == kStages) {
            slot = 0;
            par ^= 1u;
          }
        }
        if (ok) umma_commit(&acc_full[b]);
      }
      // Every MMA issued must have completed before TMEM is released.
      umma_commit(mma_done);
      volatile int no_abort = 0;
      if (!mbar_wait(mma_done, 0, &no_abort)) atomicOr(p.err, kErrWaitTimeout);
    }
  } else if (warp < kWarpEpi) {
    // ---------------------------------------------------------- dequantisers
    const int d = warp - kWarpDeq;                // 0..7
    const int h = d >> 2;                         // k half: [32h, 32h+32)
    // A row (= TMEM lane) written by this thread: consecutive across the
    // warp, so that the swizzled shared-memory stores are conflict free.
    // SwiGLU interleaves gate/up pairs (A row 2j = gate row j, 2j+1 = up
    // row j) so that one warp holds both halves of every output.
    const int arow = (d & 3) * 32 + lane;
    const int r = p.swiglu ? ((arow & 1) ? 64 + (arow >> 1) : (arow >> 1)) : arow;  // raw row
    const uint32_t a_row_off = (arow >> 3) * 1024 + (arow & 7) * 128;
    int slot = 0, it = 0;
    uint32_t par = 0;
    for (int g = 0; g < total_stages; ++g, it = (it + 1 == n_stages) ? 0 : it + 1) {
      if (!mbar_wait(&tma_full[slot], par, abort_flag)) break;
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
      if (++slot == kStages) {
        slot = 0;
        par ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quarter
    const int lane_row = 32 * q + lane;           // A row = TMEM lane
    const int64_t n_out = p.swiglu ? p.N / 2 : p.N;
    for (int i = 0; i < my_tiles; ++i) {
      const int b = i & 1;
      // Warp-uniform (and reconverged) before the warp-aligned tcgen05.ld.
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[b], (i >> 1) & 1, abort_flag))) break;
      tc_fence_after_sync();
      int bw, m_tile;
      tile_of(i, bw, m_tile);
      const int64_t ncol = p.swiglu ? static_cast<int64_t>(bw) * 64 + (lane_row >> 1)
                                    : static_cast<int64_t>(bw) * kTileW + lane_row;
      const uint32_t t_acc = tmem_base + b * kAccCols + (static_cast<uint32_t>(32 * q) << 16);
      // SwiGLU: odd A rows are up rows, with their own global scale
      const float lane_scale = p.seg.n ? seg_scale(p.seg, ncol)
                               : ((p.swiglu && (lane & 1)) ? p.out_scale_up : p.out_scale);
#pragma unroll 1
      for (int c0 = 0; c0 < kTileX; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32cols(t_acc + c0, v);
        tmem_ld_wait();
        if (c0 + 32 == kTileX) {
          // the accumulator is read out: the MMA issuer may reuse it
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
        // Written once, read by the next layer: streaming stores, so that
        // the results do not push the band's activations out of L2.
        auto store = [&](int m, float yv) {
          if (m >= p.M) return;
          const int64_t off = static_cast<int64_t>(m) * n_out + ncol;
          if (p.out_f32)
            st_global_cs(static_cast<float*>(p.y) + off, yv);
          else
            st_global_cs(static_cast<__nv_bfloat16*>(p.y) + off, __float2bfloat16_rn(yv));
        };
        if (p.swiglu) {
          // Lanes 2k (gate) and 2k+1 (up) share output column ncol; the
          // even lane produces the even activation rows of the chunk, the
          // odd lane the odd ones.  Per pair of rows each lane sends the
          // value of the row its partner produces and receives the other
          // half of its own row's pair: one exchange per two rows, every
          // lane busy (no divergent half-warp).
          const int odd = lane & 1;
          const float s_gate = p.seg.n ? lane_scale : p.out_scale;
          const float s_up = p.seg.n ? lane_scale : p.out_scale_up;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float mine = __uint_as_float(odd ? v[2 * i + 1] : v[2 * i]);
            const float send = __uint_as_float(odd ? v[2 * i] : v[2 * i + 1]);
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float g = (odd ? recv : mine) * s_gate;
            const float u = (odd ? mine : recv) * s_up;
            store(m_tile + c0 + 2 * i + odd, silu_mul(g, u));
          }
        } else {
          // Lanes 2k and 2k+1 hold adjacent output columns: per pair of
          // rows each lane sends its partner one value and stores both
          // columns of one row as a single 4-byte (f32: 8-byte) word.
          const int odd = lane & 1;
          const int64_t col0 = ncol - odd;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = __uint_as_float(v[2 * i]) * lane_scale;
            const float a1 = __uint_as_float(v[2 * i + 1]) * lane_scale;
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
            const int m = m_tile + c0 + 2 * i + odd;
            if (m >= p.M) continue;
            const float lo = odd ? recv : a0, hi = odd ? a1 : recv;
            const int64_t off = static_cast<int64_t>(m) * n_out + col0;
            if (p.out_f32)
              st_global_cs(reinterpret_cast<float2*>(static_cast<float*>(p.y) + off),
                           make_float2(lo, hi));
            else
              st_global_cs(reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.y) + off),
                           f32x2_to_bf16x2(lo, hi));
          }
        }
      }
    }
  }

  if (*abort_flag && threadIdx.x == 0) atomicOr(p.err, kErrWaitTimeout);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace tcgemm
}  // namespace nvfp4
