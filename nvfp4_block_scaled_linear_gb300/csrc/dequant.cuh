// dequant.cuh -- e2m1 x e4m3 block dequantisation in registers.
//
// Format (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", section 1, checkpoint
// condition 2): weight_packed u8 (out, in/2) holds FP4 e2m1 codes two per
// byte (low nibble = even k), weight_scale holds one fp8 e4m3 per 16 inputs.
//
// A code times a block scale has at most 2 x 4 significant bits, so the
// product is exact in bf16 and in f16.  The kernels therefore feed exact
// weights to the tensor cores and apply the fp32 global scale once, in the
// epilogue.
//
// bf16 bit trick.  Placing a code's three magnitude bits (e1 e0 m) at bf16
// bits 8..6 and its sign at bit 15 gives the bf16 number code * 2^-126: the
// two exponent bits land in the low end of the bf16 exponent field, the
// mantissa bit at the top of the mantissa, and exponent 0 (the e2m1
// subnormals 0 and 0.5) lands on bf16's own subnormals.  One bf16 multiply by
// S = scale * 2^116 then yields code * scale * 2^-10 exactly (2^-20 at the
// smallest, so never subnormal); the epilogue multiplies by 2^10.
//
// f16 path.  The hardware converts two e2m1 codes to f16x2 in one
// instruction; one f16x2 multiply by the scale gives code * scale exactly
// (between 2^-10 and 2688 in magnitude: normal f16 numbers).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace nvfp4 {

// Exponent offset folded into the bf16 dequantised weights; undone in the
// epilogue, which multiplies the fp32 accumulator by fp32(2^10 / global_scale).
constexpr float kWeightPow2 = 1024.0f;   // 2^10

// Output-column segments with their own global scales (one launch over
// weights stacked from several projections, e.g. q, k and v): output
// column n < end[0] uses scale[0], n < end[1] scale[1], ...  n == 0: one
// scale for all columns (the kernel's out_scale).
constexpr int kMaxSegments = 8;
struct SegScales {
  int n;
  int64_t end[kMaxSegments];
  float scale[kMaxSegments];
};

__device__ __forceinline__ float seg_scale(const SegScales& s, int64_t col) {
  float sc = s.scale[0];
#pragma unroll
  for (int i = 1; i < kMaxSegments; ++i)
    if (i < s.n && col >= s.end[i - 1]) sc = s.scale[i];
  return sc;
}

// SwiGLU epilogue: silu(g) * u = g / (1 + e^-g) * u in fp32, written with
// t = e^-|g| so that nothing overflows: g / (1 + t) for g >= 0, and
// g * t / (1 + t) -- the same number -- for g < 0.  t comes from the CUDA fast
// exponential (a few ulp here) and the division is the fast one, exact to a
// few ulp for a denominator in [1, 2].  The fast exponential flushes results
// below fp32's normal range to zero, so for g < -80 (rare) t is taken from
// the accurate expf, which keeps silu(g) -- a normal fp32 number down to
// about g = -92 -- instead of returning zero.
__device__ __forceinline__ float silu_mul(float g, float u) {
  float t = __expf(-fabsf(g));
  if (g < -80.f) t = expf(g);
  return __fdividef(g >= 0.f ? g : g * t, 1.0f + t) * u;
}

// bf16x2 (S, S) for an e4m3 bit pattern, S = value * 2^116; NaN for S.1111.111.
// Exact: an e4m3 value has at most 4 significant bits.
__device__ __forceinline__ uint32_t scale_pair_from_e4m3(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  uint32_t f32;
  if (e == 15u && m == 7u) {
    f32 = 0x7FC00000u;                                  // NaN
  } else if (e != 0u) {
    // 2^(e-7) * (1 + m/8) * 2^116 : biased exponent e - 7 + 116 + 127
    f32 = ((e + 236u) << 23) | (m << 20);
  } else {
    // subnormal: (m/8) * 2^-6 * 2^116 = m * 2^107
    f32 = __float_as_uint(static_cast<float>(m) * 0x1p107f);
  }
  f32 |= (b & 0x80u) << 24;                             // sign
  const uint32_t h = f32 >> 16;                         // exact bf16
  return h | (h << 16);
}

// f16x2 (S, S) for an e4m3 bit pattern, S = its value (exact in f16); NaN
// for S.1111.111.
__device__ __forceinline__ uint32_t scale_pair_f16_from_e4m3(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  uint32_t h;
  if (e == 15u && m == 7u)
    h = 0x7E00u;                                   // NaN
  else if (e != 0u)
    h = ((e + 8u) << 10) | (m << 7);               // 2^(e-7) (1 + m/8), f16 bias 15
  else
    h = __half_as_ushort(__float2half_rn(static_cast<float>(m) * 0x1p-9f));  // m 2^-9
  h |= (b & 0x80u) << 8;                           // sign
  return h | (h << 16);
}

// Integer shifts by a constant, written as multiplies so that they issue on
// the FMA pipe (IMAD) rather than the integer/logic pipe, which the masks
// below already keep busy.
__device__ __forceinline__ uint32_t shl_fma(uint32_t w, uint32_t pow2) {
  uint32_t d;
  asm("mul.lo.u32 %0, %1, %2;" : "=r"(d) : "r"(w), "r"(pow2));
  return d;
}
__device__ __forceinline__ uint32_t shr_fma(uint32_t w, uint32_t pow2_32_minus_s) {
  uint32_t d;
  asm("mul.hi.u32 %0, %1, %2;" : "=r"(d) : "r"(w), "r"(pow2_32_minus_s));
  return d;
}

// Eight codes (one 32-bit word, k = 0..7 in nibble order) times the bf16
// pair scale S -> four bf16x2 words pairing (k, k+4):
//   out[i] = ( w(k=i), w(k=i+4) ),  i = 0..3,
// each w = code * scale * 2^-10.  Pair i needs its magnitude bits moved by
// 6 - 4i and its sign bits by 12 - 4i.
__device__ __forceinline__ void dequant8_strided(uint32_t w, uint32_t S, uint32_t* out) {
  const uint32_t kMag = 0x01C001C0u, kSign = 0x80008000u;
  const uint32_t r0 = (shl_fma(w, 1u << 6) & kMag) | (shl_fma(w, 1u << 12) & kSign);
  const uint32_t r1 = (shl_fma(w, 1u << 2) & kMag) | (shl_fma(w, 1u << 8) & kSign);
  const uint32_t r2 = (shr_fma(w, 1u << 30) & kMag) | (shl_fma(w, 1u << 4) & kSign);
  const uint32_t r3 = (shr_fma(w, 1u << 26) & kMag) | (w & kSign);
  out[0] = bf16x2_mul(r0, S);
  out[1] = bf16x2_mul(r1, S);
  out[2] = bf16x2_mul(r2, S);
  out[3] = bf16x2_mul(r3, S);
}

// Reorder the (k, k+4) pairs of dequant8_strided into consecutive pairs
// (0,1) (2,3) (4,5) (6,7), the order of a row in memory.
__device__ __forceinline__ void pair_consecutive(const uint32_t* p, uint32_t* out) {
  out[0] = prmt(p[0], p[1], 0x5410u);   // k0 | k1
  out[1] = prmt(p[2], p[3], 0x5410u);   // k2 | k3
  out[2] = prmt(p[0], p[1], 0x7632u);   // k4 | k5
  out[3] = prmt(p[2], p[3], 0x7632u);   // k6 | k7
}

// Eight codes (one 32-bit word, k = 0..7 in order) times the f16 pair scale
// S -> four f16x2 words of consecutive k: out[j] = (w(2j), w(2j+1)), each
// w = code * scale exactly.  The word is split into byte registers, so each
// conversion reads its byte in place (no shifts).
__device__ __forceinline__ void dequant8_f16(uint32_t w, uint32_t S, uint32_t* out) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
      "mul.rn.f16x2 %0, h0, %5;\n\t"
      "mul.rn.f16x2 %1, h1, %5;\n\t"
      "mul.rn.f16x2 %2, h2, %5;\n\t"
      "mul.rn.f16x2 %3, h3, %5;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(w), "r"(S));
}

}  // namespace nvfp4
