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

// Packed fp32 pairs: Blackwell's mul / fma .rn.f32x2 round each lane exactly
// as the scalar instruction does (subnormals kept), at one instruction per
// pair.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
  return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// RN(1/d) for the odd divisors d = 2i + 1 <= 15, one shared copy per CTA
// (filled by the first eight threads before the CTA's first block).
struct OddReciprocals {
  float r[8];
};
__device__ __forceinline__ void fill_odd_reciprocals(OddReciprocals& t) {
  if (threadIdx.x < 8) t.r[threadIdx.x] = __frcp_rn(static_cast<float>(2 * threadIdx.x + 1));
  __syncthreads();
}

// A block scale (finite, nonzero e4m3 byte b) as d * 2^e, d odd: the
// divisor d, r = RN(1/d) and the factor 2^-e.
struct ScaleDiv {
  float d, r, p2;
};
__device__ __forceinline__ ScaleDiv scale_div(uint32_t b, const OddReciprocals& rcp) {
  const int E = static_cast<int>((b >> 3) & 15u), m = static_cast<int>(b & 7u);
  const int sig = E ? 8 + m : m;                 // s = sig * 2^ex
  const int ex = E ? E - 10 : -9;
  const int t = __ffs(sig) - 1;                  // trailing zero bits of sig
  const int e = ex + t;                          // in [-9, 8]
  ScaleDiv sd;
  sd.d = static_cast<float>(sig >> t);
  sd.r = rcp.r[sig >> (t + 1)];
  sd.p2 = __int_as_float((127 - e) << 23);
  return sd;
}

// Eight codes, weights 2i (low nibble) and 2i + 1 of byte i, in one word.
__device__ __forceinline__ uint32_t to_e2m1x8(const float (&q)[8]) {
  uint32_t d;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(d)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]),
        "f"(q[7]));
  return d;
}

// One 16-input block: its 16 weights (fp32 values of bf16 numbers) -> the
// block's e4m3 scale byte and 8 code bytes.  Per weight pair: x = RN(w gs),
// then RN(x / s) by the refinement above (q0 = RN(x r), rem = RN(x - q0 d)
// as an fma with -d, q1 = RN(q0 + rem r), times 2^-e), in f32x2; the sign of
// x is put back on the quotient (an exactly cancelled refinement gives +0).
__device__ __forceinline__ void quantize_block16(const float (&f)[16], float gs,
                                                 const OddReciprocals& rcp, uint2& codes,
                                                 uint8_t& scale) {
  float amax_b = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(f[i]));
  const uint32_t sbyte = to_e4m3(__fdiv_rn(__fmul_rn(amax_b, gs), 6.0f));
  uint32_t packed[2] = {0u, 0u};
  // zero scale: all codes +0; a NaN scale (only from non-finite weights,
  // which the format does not cover) likewise
  if (sbyte != 0u && sbyte != 0x7Fu) {
    const ScaleDiv sd = scale_div(sbyte, rcp);
    const uint64_t g2 = f2(gs, gs), r2 = f2(sd.r, sd.r), nd2 = f2(-sd.d, -sd.d),
                   p2 = f2(sd.p2, sd.p2);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float q[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t x = f2_mul(f2(f[8 * h + 2 * i], f[8 * h + 2 * i + 1]), g2);
        const uint64_t q0 = f2_mul(x, r2);
        const uint64_t rem = f2_fma(q0, nd2, x);
        const float2 qv = f2_split(f2_mul(f2_fma(rem, r2, q0), p2));
        const float2 xv = f2_split(x);
        q[2 * i] = copysignf(qv.x, xv.x);
        q[2 * i + 1] = copysignf(qv.y, xv.y);
      }
      packed[h] = to_e2m1x8(q);
    }
  }
  codes = make_uint2(packed[0], packed[1]);
  scale = static_cast<uint8_t>(sbyte);
}

// One thread per 16-input block: n_blocks = N * K / 16 in row-major order.
// The next block's 32 bytes are loaded before the current one is quantised,
// so that each thread keeps two blocks' loads in flight (one alone left the
// pass waiting on memory latency).
__global__ void __launch_bounds__(kThreads)
    quantize_kernel(const uint4* __restrict__ w, int64_t n_blocks,
                    const unsigned int* __restrict__ amax_bits, uint2* __restrict__ codes,
                    uint8_t* __restrict__ scales) {
  __shared__ OddReciprocals rcp;
  fill_odd_reciprocals(rcp);
  const float gs = global_scale_of(__uint_as_float(*amax_bits));
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  int64_t b = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
  uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
  if (b < n_blocks) {
    v0 = w[2 * b];
    v1 = w[2 * b + 1];
  }
  for (; b < n_blocks; b += stride) {
    uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0;
    if (b + stride < n_blocks) {
      n0 = w[2 * (b + stride)];
      n1 = w[2 * (b + stride) + 1];
    }
    const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = __uint_as_float(words[i] << 16);
      f[2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
    }
    uint2 c;
    uint8_t sc;
    quantize_block16(f, gs, rcp, c, sc);
    codes[b] = c;
    scales[b] = sc;
    v0 = n0;
    v1 = n1;
  }
}

// ---------------------------------------------------------------- FP8 source
// A block-scaled FP8 checkpoint tensor (e4m3 codes, one fp32 scale_inv per
// B x B block) goes FP8 -> BF16 -> NVFP4 (FlashRT docs, the MTP-head note:
// FP8 e4m3 in blocks of 128, converted once at load; qwentin README,
// "Convert a model": block-scaled E4M3 tensors are dequantised first).  The
// bf16 image of each weight, RNE_bf16(e4m3 * scale_inv), is formed on the
// fly in both passes, so no bf16 copy of the tensor is stored.
//
// Work unit: U consecutive 16-input blocks of one row.  U = 4 (64 weights)
// when K and B are multiples of 64, so that a unit never crosses a row or a
// scale block: one scale lookup and one cursor step per 64 weights; U = 1
// otherwise.
struct Fp8Layout {
  int64_t n_units;      // N * K / (16 U)
  int64_t units_per_row;// K / (16 U)
  int64_t kb;           // ceil(K / B): scale_inv row length
  int64_t B;            // scale block edge (a multiple of 16)
  int b_shift;          // log2(B) when B is a power of two, else -1
};

// Position of unit u (row, unit in row) and of its scale, walked forward by a
// fixed stride: one division per thread, not per unit.
template <int U>
struct Fp8Cursor {
  int64_t u, row, ku;
  int64_t d_row, d_ku;      // the stride as (rows, units)
  __device__ Fp8Cursor(const Fp8Layout& L, int64_t start, int64_t stride)
      : u(start), row(start / L.units_per_row),
        ku(start - (start / L.units_per_row) * L.units_per_row),
        d_row(stride / L.units_per_row), d_ku(stride - (stride / L.units_per_row) * L.units_per_row) {}
  __device__ __forceinline__ void advance(const Fp8Layout& L, int64_t stride) {
    u += stride;
    row += d_row;
    ku += d_ku;
    if (ku >= L.units_per_row) {
      ku -= L.units_per_row;
      ++row;
    }
  }
  __device__ __forceinline__ int64_t scale_index(const Fp8Layout& L) const {
    if (L.b_shift >= 0)
      return (row >> L.b_shift) * L.kb + ((ku * 16 * U) >> L.b_shift);
    return (row / L.B) * L.kb + (ku * 16 * U) / L.B;
  }
};

// The fp32 values of the four e4m3 bytes of a word, two f16x2 conversions
// (exact), times s and rounded to bf16, as fp32: f[j] = RNE_bf16(RN(e_j s)).
__device__ __forceinline__ void fp8_images4(uint32_t word, uint64_t s2, float* f) {
  uint32_t h[2];
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(h[0]), "=r"(h[1])
      : "r"(word));
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
    const float2 p = f2_split(f2_mul(f2(e.x, e.y), s2));
    uint32_t b;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(p.y), "f"(p.x));
    f[2 * j] = __uint_as_float(b << 16);
    f[2 * j + 1] = __uint_as_float(b & 0xFFFF0000u);
  }
}

// |w| maximum of the bf16 images, into *amax_bits (zeroed before).  Both
// roundings are monotone, so a unit's largest |bf16 image| is the image of
// its largest e4m3 magnitude: RN_bf16(RN_fp32(max|e4m3| * |scale_inv|)).
// e4m3 magnitudes order like their 7-bit patterns, so the unit maximum is an
// integer maximum over bytes (odd bytes as the high byte of 16-bit lanes,
// even bytes alone in them) and one conversion per unit.
template <int U>
__global__ void __launch_bounds__(kThreads) amax_fp8_kernel(const uint4* __restrict__ w8,
                                                            const float* __restrict__ scale_inv,
                                                            Fp8Layout L,
                                                            unsigned int* amax_bits) {
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (Fp8Cursor<U> c(L, blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x, stride);
       c.u < L.n_units; c.advance(L, stride)) {
    uint32_t m_odd = 0u, m_even = 0u;
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint4 v = w8[c.u * U + j];
      const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m_odd = max_u16x2(m_odd, words[i] & 0x7F7F7F7Fu);
        m_even = max_u16x2(m_even, words[i] & 0x007F007Fu);
      }
    }
    const uint32_t mx = max(max((m_odd >> 8) & 0xFFu, m_odd >> 24),
                            max(m_even & 0xFFu, m_even >> 16));
    uint32_t h;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
        : "=r"(h)
        : "r"(mx));
    const float a = __low2float(*reinterpret_cast<const __half2*>(&h));
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

// U = 4 stores the unit's four scale bytes as one word (the host takes this
// path only for a 4-byte aligned w_scale).  As in the bf16 quantiser, the
// next unit's codes and scale are loaded before the current unit is
// quantised.
template <int U>
__global__ void __launch_bounds__(kThreads)
    quantize_fp8_kernel(const uint4* __restrict__ w8, const float* __restrict__ scale_inv,
                        Fp8Layout L, const unsigned int* __restrict__ amax_bits,
                        uint2* __restrict__ codes, uint8_t* __restrict__ scales) {
  __shared__ OddReciprocals rcp;
  fill_odd_reciprocals(rcp);
  const float gs = global_scale_of(__uint_as_float(*amax_bits));
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  Fp8Cursor<U> c(L, blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x, stride);
  uint4 v[U];
  float s = 0.0f;
  if (c.u < L.n_units) {
#pragma unroll
    for (int j = 0; j < U; ++j) v[j] = w8[c.u * U + j];
    s = scale_inv[c.scale_index(L)];
  }
  while (c.u < L.n_units) {
    Fp8Cursor<U> cn = c;
    cn.advance(L, stride);
    uint4 vn[U];
    float sn = 0.0f;
#pragma unroll
    for (int j = 0; j < U; ++j) vn[j] = make_uint4(0u, 0u, 0u, 0u);
    if (cn.u < L.n_units) {
#pragma unroll
      for (int j = 0; j < U; ++j) vn[j] = w8[cn.u * U + j];
      sn = scale_inv[cn.scale_index(L)];
    }
    const uint64_t s2 = f2(s, s);
    uint32_t sc_word = 0u;
#pragma unroll
    for (int j = 0; j < U; ++j) {
      float f[16];
      fp8_images4(v[j].x, s2, f);
      fp8_images4(v[j].y, s2, f + 4);
      fp8_images4(v[j].z, s2, f + 8);
      fp8_images4(v[j].w, s2, f + 12);
      uint2 cw;
      uint8_t sc;
      quantize_block16(f, gs, rcp, cw, sc);
      codes[c.u * U + j] = cw;
      sc_word |= static_cast<uint32_t>(sc) << (8 * j);
    }
    if constexpr (U == 4)
      *reinterpret_cast<uint32_t*>(scales + c.u * 4) = sc_word;
    else
      scales[c.u] = static_cast<uint8_t>(sc_word);
#pragma unroll
    for (int j = 0; j < U; ++j) v[j] = vn[j];
    s = sn;
    c = cn;
  }
}

// *gs = 448 / amax, in place over the gathered maximum.
__global__ void finalize_kernel(float* gs) {
  if (threadIdx.x == 0) *gs = global_scale_of(*gs);
}

}  // namespace quant
}  // namespace nvfp4
