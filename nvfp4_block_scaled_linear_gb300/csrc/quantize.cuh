// quantize.cuh -- bf16 weights -> the NVFP4 checkpoint format this library
// consumes (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", section 1,
// condition 2: weight_packed FP4 e2m1 two per byte, weight_scale e4m3 per
// 16 inputs, weight_global_scale = 448 / amax).
//
// The pages give the stored format and the dequantisation, not the rounding
// steps; this follows the plainest reading consistent with them, every step
// in fp32 with round-to-nearest-even:
//   amax = max |w|;  gs = 448 / amax  (1 if amax = 0)
//   per 16-input block:  s = e4m3((amax_block * gs) / 6), saturating
//   per weight:          code = e2m1((w * gs) / s), saturating, sign kept;
//                        all codes +0 where s rounds to 0
// Both conversions are the hardware's (cvt.rn.satfinite.e4m3x2 / e2m1x2).
//
// Three stream-ordered steps, no workspace: the tensor maximum is gathered
// by atomicMax into the caller's global-scale word (as fp32 bits: the bit
// patterns of non-negative floats order like their values), the quantiser
// reads it, and a last one-thread kernel turns it into 448 / amax.
//
// The per-weight division by the block scale is done without a general fp32
// division, which dominated the quantiser's instruction count: an e4m3 scale
// is s = d * 2^e with d an odd integer <= 15, so RN(v / s) = RN(v / d) * 2^-e
// (exact scaling while the quotient is a normal number; a smaller quotient
// is far below every e2m1 rounding threshold), and RN(v / d) follows from the
// correctly rounded reciprocal r = RN(1/d) by Markstein's refinement,
// q0 = RN(v r), rem = RN(v - q0 d), q1 = RN(q0 + rem r), which is correctly
// rounded for every fp32 v and every such d (checked exhaustively over all
// significands in the tests).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace nvfp4 {
namespace quant {

constexpr int kThreads = 256;

// |w| maximum over n_vec x 8 bf16 values, into *amax_bits (zeroed before).
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint4* __restrict__ w,
                                                        int64_t n_vec,
                                                        unsigned int* amax_bits) {
  uint32_t m = 0;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < n_vec;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const uint4 v = w[i];
    m = max_u16x2(m, max_u16x2(max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               max_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
  }
  m = max(m & 0xFFFFu, m >> 16);
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t red[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kThreads / 32 ? red[lane] : 0u;
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0 && m != 0) atomicMax(amax_bits, m << 16);   // bf16 -> fp32 bits
  }
}

__device__ __forceinline__ float global_scale_of(float amax) {
  return amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f;
}

// e4m3 bits of the nearest e4m3 to v (saturating).
__device__ __forceinline__ uint32_t to_e4m3(float v) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(0.0f), "f"(v));
  return d & 0xFFu;
}
// A block scale (finite, nonzero e4m3 byte b) as d * 2^e, d odd: the
// divisor d, r = RN(1/d) and the factor 2^-e.
struct ScaleDiv {
  float d, r, p2;
};
__device__ __forceinline__ ScaleDiv scale_div(uint32_t b) {
  const int E = static_cast<int>((b >> 3) & 15u), m = static_cast<int>(b & 7u);
  const int sig = E ? 8 + m : m;                 // s = sig * 2^ex
  const int ex = E ? E - 10 : -9;
  const int t = __ffs(sig) - 1;                  // trailing zero bits of sig
  const int e = ex + t;                          // in [-9, 8]
  ScaleDiv sd;
  sd.d = static_cast<float>(sig >> t);
  sd.r = __frcp_rn(sd.d);
  sd.p2 = __int_as_float((127 - e) << 23);
  return sd;
}
// RN(v / s) for the scale split by scale_div (v finite); the sign of a zero
// quotient follows v, as in the division.
__device__ __forceinline__ float div_by_scale(float v, const ScaleDiv& sd) {
  const float q0 = __fmul_rn(v, sd.r);
  const float rem = __fmaf_rn(-q0, sd.d, v);
  const float q1 = __fmaf_rn(rem, sd.r, q0);
  return copysignf(__fmul_rn(q1, sd.p2), v);
}

// Two codes in one byte: lo -> low nibble (even k), hi -> high nibble.
__device__ __forceinline__ uint32_t to_e2m1x2(float lo, float hi) {
  uint32_t d;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\t"
      "cvt.u32.u8 %0, b;\n\t}"
      : "=r"(d)
      : "f"(hi), "f"(lo));
  return d;
}

// One 16-input block: its 16 weights (fp32 values of bf16 numbers) -> the
// block's e4m3 scale byte and 8 code bytes.
__device__ __forceinline__ void quantize_block16(const float (&f)[16], float gs, uint2& codes,
                                                 uint8_t& scale) {
  float amax_b = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(f[i]));
  const uint32_t sbyte = to_e4m3(__fdiv_rn(__fmul_rn(amax_b, gs), 6.0f));
  uint32_t packed[2] = {0u, 0u};
  // zero scale: all codes +0; a NaN scale (only from non-finite weights,
  // which the format does not cover) likewise
  if (sbyte != 0u && sbyte != 0x7Fu) {
    const ScaleDiv sd = scale_div(sbyte);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = to_e2m1x2(div_by_scale(__fmul_rn(f[2 * i], gs), sd),
                                      div_by_scale(__fmul_rn(f[2 * i + 1], gs), sd));
      packed[i >> 2] |= byte << (8 * (i & 3));
    }
  }
  codes = make_uint2(packed[0], packed[1]);
  scale = static_cast<uint8_t>(sbyte);
}

// One thread per 16-input block: n_blocks = N * K / 16 in row-major order.
__global__ void __launch_bounds__(kThreads)
    quantize_kernel(const uint4* __restrict__ w, int64_t n_blocks,
                    const unsigned int* __restrict__ amax_bits, uint2* __restrict__ codes,
                    uint8_t* __restrict__ scales) {
  const float gs = global_scale_of(__uint_as_float(*amax_bits));
  for (int64_t b = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; b < n_blocks;
       b += static_cast<int64_t>(gridDim.x) * kThreads) {
    const uint4 v0 = w[2 * b], v1 = w[2 * b + 1];
    const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = __uint_as_float(words[i] << 16);
      f[2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
    }
    uint2 c;
    uint8_t sc;
    quantize_block16(f, gs, c, sc);
    codes[b] = c;
    scales[b] = sc;
  }
}

// ---------------------------------------------------------------- FP8 source
// A block-scaled FP8 checkpoint tensor (e4m3 codes, one fp32 scale_inv per
// B x B block) goes FP8 -> BF16 -> NVFP4 (FlashRT docs, the MTP-head note:
// FP8 e4m3 in blocks of 128, converted once at load; qwentin README,
// "Convert a model": block-scaled E4M3 tensors are dequantised first).  The
// bf16 image of each weight, RNE_bf16(e4m3 * scale_inv), is formed on the
// fly in both passes, so no bf16 copy of the tensor is stored.
struct Fp8Layout {
  int64_t n_blocks;     // N * K / 16
  int64_t k_blocks;     // K / 16 (16-input blocks per row)
  int64_t kb;           // ceil(K / B): scale_inv row length
  int64_t B;            // scale block edge (a multiple of 16)
  int b_shift;          // log2(B) when B is a power of two, else -1
};

// Position of 16-input block b (row, k-block) and of its scale, walked
// forward by a fixed stride: one division per thread, not per block.
struct Fp8Cursor {
  int64_t b, row, kblk;
  int64_t d_row, d_kblk;    // the stride as (rows, k-blocks)
  __device__ Fp8Cursor(const Fp8Layout& L, int64_t start, int64_t stride)
      : b(start), row(start / L.k_blocks), kblk(start - (start / L.k_blocks) * L.k_blocks),
        d_row(stride / L.k_blocks), d_kblk(stride - (stride / L.k_blocks) * L.k_blocks) {}
  __device__ __forceinline__ void advance(const Fp8Layout& L, int64_t stride) {
    b += stride;
    row += d_row;
    kblk += d_kblk;
    if (kblk >= L.k_blocks) {
      kblk -= L.k_blocks;
      ++row;
    }
  }
  __device__ __forceinline__ int64_t scale_index(const Fp8Layout& L) const {
    if (L.b_shift >= 0)
      return (row >> L.b_shift) * L.kb + ((kblk * 16) >> L.b_shift);
    return (row / L.B) * L.kb + (kblk * 16) / L.B;
  }
};

// Two e4m3 bytes (the low byte -> .x) as fp32, exactly.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two) {
  uint32_t h;
  asm("{\n\t.reg .b16 s;\n\t"
      "cvt.u16.u32 s, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, s;\n\t}"
      : "=r"(h)
      : "r"(two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The bf16 images (as fp32) of the 16 FP8 weights of the cursor's block.
__device__ __forceinline__ void fp8_block16(const uint4* __restrict__ w8,
                                            const float* __restrict__ scale_inv,
                                            const Fp8Layout& L, const Fp8Cursor& c,
                                            float (&f)[16]) {
  const float s = scale_inv[c.scale_index(L)];
  const uint4 v = w8[c.b];
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 lo = e4m3x2_to_f32(words[i] & 0xFFFFu);
    const float2 hi = e4m3x2_to_f32(words[i] >> 16);
    f[4 * i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(lo.x, s)));
    f[4 * i + 1] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(lo.y, s)));
    f[4 * i + 2] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(hi.x, s)));
    f[4 * i + 3] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(hi.y, s)));
  }
}

// |w| maximum of the bf16 images, into *amax_bits (zeroed before).  Both
// roundings are monotone, so a block's largest |bf16 image| is the image of
// its largest e4m3 magnitude: RN_bf16(RN_fp32(max|e4m3| * |scale_inv|)).
// e4m3 magnitudes order like their 7-bit patterns, so the block maximum is
// a byte-wise integer maximum and one conversion per 16 weights.
__global__ void __launch_bounds__(kThreads) amax_fp8_kernel(const uint4* __restrict__ w8,
                                                            const float* __restrict__ scale_inv,
                                                            Fp8Layout L,
                                                            unsigned int* amax_bits) {
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (Fp8Cursor c(L, blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x, stride);
       c.b < L.n_blocks; c.advance(L, stride)) {
    const uint4 v = w8[c.b];
    uint32_t mx = __vmaxu4(__vmaxu4(v.x & 0x7F7F7F7Fu, v.y & 0x7F7F7F7Fu),
                           __vmaxu4(v.z & 0x7F7F7F7Fu, v.w & 0x7F7F7F7Fu));
    mx = max(max(mx & 0xFFu, (mx >> 8) & 0xFFu), max((mx >> 16) & 0xFFu, mx >> 24));
    const float a = e4m3x2_to_f32(mx).x;
    const float sabs = fabsf(scale_inv[c.scale_index(L)]);
    m = fmaxf(m, __bfloat162float(__float2bfloat16_rn(__fmul_rn(a, sabs))));
  }
  // non-negative floats order like their bit patterns
  uint32_t u = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  __shared__ uint32_t red[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = u;
  __syncthreads();
  if (warp == 0) {
    u = lane < kThreads / 32 ? red[lane] : 0u;
    u = __reduce_max_sync(0xffffffffu, u);
    if (lane == 0 && u != 0) atomicMax(amax_bits, u);
  }
}

__global__ void __launch_bounds__(kThreads)
    quantize_fp8_kernel(const uint4* __restrict__ w8, const float* __restrict__ scale_inv,
                        Fp8Layout L, const unsigned int* __restrict__ amax_bits,
                        uint2* __restrict__ codes, uint8_t* __restrict__ scales) {
  const float gs = global_scale_of(__uint_as_float(*amax_bits));
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (Fp8Cursor c(L, blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x, stride);
       c.b < L.n_blocks; c.advance(L, stride)) {
    float f[16];
    fp8_block16(w8, scale_inv, L, c, f);
    uint2 cw;
    uint8_t sc;
    quantize_block16(f, gs, cw, sc);
    codes[c.b] = cw;
    scales[c.b] = sc;
  }
}

// *gs = 448 / amax, in place over the gathered maximum.
__global__ void finalize_kernel(float* gs) {
  if (threadIdx.x == 0) *gs = global_scale_of(*gs);
}

}  // namespace quant
}  // namespace nvfp4
