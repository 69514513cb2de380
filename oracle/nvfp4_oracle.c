/*
 * nvfp4_oracle.c -- plain, slow, obviously-correct CPU oracle for the NVFP4
 * W4A16 block-scaled linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it and shares no code,
 * header, table or helper with it.
 *
 * What it computes (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", section 1
 * "Model dependencies", subsection "Can I use a different NVFP4 Qwen3.6
 * checkpoint?", condition 2: the compressed-tensors nvfp4-pack-quantized
 * schema):
 *   weight_packed       u8   (out, in/2)   FP4 e2m1, two codes per byte
 *   weight_scale        e4m3 (out, in/16)  one scale per 16-element block
 *   weight_global_scale fp32 scalar
 * and the first table of that section (main model = "NVFP4 W4A16"): weights
 * are 4-bit, activations bf16.
 *
 *   w[n,k]  = e2m1(code[n,k]) * e4m3(scale[n, k/16]) / global_scale
 *   y[m,n]  = sum_k x[m,k] * w[n,k]              (here: exact-ish in fp64)
 *   A[m,n]  = sum_k |x[m,k] * w[n,k]|            (error-bound companion)
 *
 * Readings taken where the pages are silent:
 *   - nibble order: the low nibble of byte j holds k = 2j, the high nibble
 *     k = 2j+1;
 *   - e4m3 is the OCP "E4M3FN" variant (the schema quotes 448 as the e4m3
 *     maximum): bias 7, subnormals, no infinities, S.1111.111 is NaN;
 *   - "dequantised weight = code x block scale / global scale" is evaluated
 *     literally, in fp64;
 *   - the fused gate/up projection (FlashRT docs, section 4 "Long-context
 *     throughput", fused MLP gate/up GEMM; qwen36-fp4 README, SwiGLU in the
 *     baseline kernel list) stores gate rows [0, N/2) then up rows [N/2, N)
 *     and returns silu(gate) * up, in fp64 from the fp64 accumulators.
 *
 * Everything is written for clarity, not speed: one output at a time, every
 * weight decoded from its bits at the point of use.  Parallelism is only a
 * split of the output columns over POSIX threads, which does not change any
 * per-output arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Format decoders, from the bit layouts.                                    */
/* ------------------------------------------------------------------------ */

/* FP4 e2m1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * exponent 0 is subnormal: value = m * 0.5.
 * otherwise value = 2^(e-1) * (1 + m/2).
 * Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u;
    unsigned e = (code >> 1) & 3u;
    unsigned m = code & 1u;
    double mag;
    if (e == 0)
        mag = 0.5 * (double)m;
    else
        mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* FP8 e4m3 (E4M3FN): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.
 * exponent 0 is subnormal: value = (m/8) * 2^-6.
 * S.1111.111 is NaN; there are no infinities, so the largest finite
 * magnitude is S.1111.110 = 448. */
double oracle_e4m3(unsigned bits)
{
    unsigned s = (bits >> 7) & 1u;
    unsigned e = (bits >> 3) & 15u;
    unsigned m = bits & 7u;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* bf16 is the top half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary32 -> bf16, round to nearest, ties to even, done with integers.
 * NaN stays NaN (quiet bit forced), infinities stay infinities, overflow
 * rounds to infinity as IEEE round-to-nearest does. */
uint16_t oracle_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);          /* NaN */
    uint32_t lower = u & 0xffffu;                        /* bits dropped */
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                                     /* carries into exp */
    return (uint16_t)upper;
}

/* Weight element w[n,k] of an NVFP4 matrix with K columns, in fp64. */
static double weight_at(const uint8_t* w_packed, const uint8_t* w_scale,
                        double global_scale, int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = w_packed[n * (K / 2) + k / 2];
    unsigned code = (k % 2 == 0) ? (byte & 0x0fu) : (byte >> 4);
    double scale = oracle_e4m3(w_scale[n * (K / 16) + k / 16]);
    return oracle_e2m1(code) * scale / global_scale;
}

/* One output of the linear layer: y[m,n] and A[m,n] = sum |x w|. */
static void dot_at(const uint16_t* x, const uint8_t* w_packed,
                   const uint8_t* w_scale, double global_scale, int64_t K,
                   int64_t m, int64_t n, double* y, double* a)
{
    double sum = 0.0, abs_sum = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double prod = oracle_bf16_to_f64(x[m * K + k]) *
                      weight_at(w_packed, w_scale, global_scale, K, n, k);
        sum += prod;
        abs_sum += fabs(prod);
    }
    *y = sum;
    *a = abs_sum;
}

/* ------------------------------------------------------------------------ */
/* Whole-matrix evaluation, split over threads by output column n.           */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t* x;
    const uint8_t* w_packed;
    const uint8_t* w_scale;
    double global_scale;
    int64_t M, N, K;
    double* y;      /* [M, N] */
    double* a;      /* [M, N], may be NULL */
    int64_t n_begin, n_end;
} linear_job;

static void* linear_worker(void* arg)
{
    linear_job* j = (linear_job*)arg;
    for (int64_t n = j->n_begin; n < j->n_end; ++n)
        for (int64_t m = 0; m < j->M; ++m) {
            double y, a;
            dot_at(j->x, j->w_packed, j->w_scale, j->global_scale, j->K, m, n,
                   &y, &a);
            j->y[m * j->N + n] = y;
            if (j->a) j->a[m * j->N + n] = a;
        }
    return NULL;
}

/* y64[m,n] = sum_k x[m,k] w[n,k] in fp64, abs64[m,n] = sum_k |x w|.
 * x: bf16 bits [M,K]; w_packed [N,K/2]; w_scale [N,K/16].
 * Returns 0, or -1 on bad arguments. */
int oracle_linear_f64(const uint16_t* x, const uint8_t* w_packed,
                      const uint8_t* w_scale, float global_scale, int64_t M,
                      int64_t N, int64_t K, double* y64, double* abs64,
                      int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 16 != 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = (int)N;
    pthread_t* tid = (pthread_t*)calloc((size_t)nthreads, sizeof *tid);
    linear_job* jobs = (linear_job*)calloc((size_t)nthreads, sizeof *jobs);
    if (!tid || !jobs) { free(tid); free(jobs); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        linear_job* j = &jobs[t];
        j->x = x; j->w_packed = w_packed; j->w_scale = w_scale;
        j->global_scale = (double)global_scale;
        j->M = M; j->N = N; j->K = K; j->y = y64; j->a = abs64;
        j->n_begin = N * t / nthreads;
        j->n_end = N * (t + 1) / nthreads;
    }
    /* job t > 0 runs on its own thread; if a thread cannot be started, its
     * job runs here instead, after job 0. */
    char* on_thread = (char*)calloc((size_t)nthreads, 1);
    for (int t = 1; t < nthreads; ++t)
        on_thread[t] = on_thread &&
                       pthread_create(&tid[t], NULL, linear_worker, &jobs[t]) == 0;
    linear_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (on_thread && on_thread[t])
            pthread_join(tid[t], NULL);
        else
            linear_worker(&jobs[t]);
    }
    free(on_thread);
    free(tid);
    free(jobs);
    return 0;
}

/* Selected outputs only: for i in [0,count): out[i] = y[m_idx[i], n_idx[i]].
 * Used for spot checks of full-size problems. */
int oracle_linear_points_f64(const uint16_t* x, const uint8_t* w_packed,
                             const uint8_t* w_scale, float global_scale,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t* m_idx, const int64_t* n_idx,
                             int64_t count, double* y64, double* abs64)
{
    if (K % 16 != 0) return -1;
    for (int64_t i = 0; i < count; ++i) {
        if (m_idx[i] < 0 || m_idx[i] >= M || n_idx[i] < 0 || n_idx[i] >= N)
            return -1;
        double y, a;
        dot_at(x, w_packed, w_scale, (double)global_scale, K, m_idx[i],
               n_idx[i], &y, &a);
        y64[i] = y;
        if (abs64) abs64[i] = a;
    }
    return 0;
}

/* silu(g) * u = g / (1 + e^-g) * u, in fp64. */
double oracle_swiglu(double gate, double up)
{
    return gate / (1.0 + exp(-gate)) * up;
}

/* Array forms of the scalar routines above, so that a caller does not cross
 * the FFI boundary once per element. */

/* out[i] = bf16 bits of RNE((float)in[i]).  The fp64 -> fp32 step is C's
 * conversion (round to nearest even); the fp32 -> bf16 step is the integer
 * rounding above. */
void oracle_f64_to_bf16_array(const double* in, uint16_t* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = oracle_f32_to_bf16_rne((float)in[i]);
}

/* Fused gate/up: y64 is [M, N] with gate columns [0, N/2) and up columns
 * [N/2, N); out is [M, N/2] with out[m,j] = silu(y[m,j]) * y[m, j + N/2]. */
int oracle_swiglu_rows(const double* y64, int64_t M, int64_t N, double* out)
{
    if (N % 2 != 0) return -1;
    int64_t H = N / 2;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < H; ++j)
            out[m * H + j] = oracle_swiglu(y64[m * N + j], y64[m * N + H + j]);
    return 0;
}

/* Decoder tables, for tests: all 16 e2m1 codes and all 256 e4m3 codes. */
void oracle_decode_tables(double* e2m1_16, double* e4m3_256)
{
    for (unsigned c = 0; c < 16; ++c) e2m1_16[c] = oracle_e2m1(c);
    for (unsigned b = 0; b < 256; ++b) e4m3_256[b] = oracle_e4m3(b);
}

/* ------------------------------------------------------------------------ */
/* Quantiser: bf16 weights -> NVFP4 (codes, e4m3 block scales, fp32 global  */
/* scale).                                                                   */
/* ------------------------------------------------------------------------ */
/*
 * The pages fix the stored format (FlashRT docs, section 1, condition 2:
 * weight_global_scale = 448 / amax; e4m3 block scales per 16 inputs; FP4
 * e2m1 codes) and that dequantisation is code * block scale / global scale,
 * but not the rounding steps.  Reading taken (the plainest one consistent
 * with those facts), every step in fp32 with round-to-nearest-even:
 *
 *   amax = max |w| over the tensor;  gs = 448 / amax   (gs = 1 if amax = 0)
 *   per 16-input block:  s = e4m3((amax_block * gs) / 6)   (saturating)
 *   per weight:          code = e2m1((w * gs) / s)          (saturating;
 *                        the sign kept, so a negative weight that rounds to
 *                        zero gets the code -0; a block whose scale rounds
 *                        to 0 gets all codes +0)
 *
 * so that code * s / gs reproduces w to within half an e2m1 step of the
 * block.  The roundings are written as brute-force nearest searches over the
 * formats' value tables (ties to the even code), not as bit tricks.
 */

/* Nearest e4m3 (E4M3FN) value to v >= 0, ties to the even code; values
 * above the largest finite e4m3 (448) saturate to it; NaN gives the NaN
 * pattern 0x7F. */
static unsigned e4m3_round(float v)
{
    if (v != v) return 0x7Fu;
    if (v >= 448.0f) return 0x7Eu;
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned b = 0; b <= 0x7Eu; ++b) {
        const double d = fabs(oracle_e4m3(b) - (double)v);
        if (d < best_d || (d == best_d && (b & 1u) == 0)) {
            best = b;
            best_d = d;
        }
    }
    return best;
}

/* Nearest e2m1 magnitude code (0..7) to |t|, ties to the even code, values
 * above 6 saturating to 6; the sign bit from t. */
static unsigned e2m1_round(float t)
{
    const double a = fabs((double)t);
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned c = 0; c < 8u; ++c) {
        const double d = fabs(oracle_e2m1(c) - a);
        if (d < best_d || (d == best_d && (c & 1u) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best | (signbit(t) ? 8u : 0u);   /* |t| > 6: nearest is 6 (saturation) */
}

/* Exposed for tests. */
unsigned oracle_e4m3_round(float v) { return e4m3_round(v); }
unsigned oracle_e2m1_round(float t) { return e2m1_round(t); }

/* w_bits: bf16 [N][K] row-major, K % 16 == 0.  Outputs: w_packed [N][K/2]
 * (low nibble = even k), w_scale [N][K/16] (e4m3 bits), *gs_out.  Returns 0,
 * or -1 on a bad shape.  Non-finite weights are outside this reading. */
int oracle_quantize(const uint16_t* w_bits, int64_t N, int64_t K, uint8_t* w_packed,
                    uint8_t* w_scale, float* gs_out)
{
    if (N <= 0 || K <= 0 || K % 16) return -1;
    float amax = 0.0f;
    for (int64_t i = 0; i < N * K; ++i) {
        const float a = fabsf((float)oracle_bf16_to_f64(w_bits[i]));
        if (a > amax) amax = a;
    }
    const float gs = amax > 0.0f ? 448.0f / amax : 1.0f;
    *gs_out = gs;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < K / 16; ++b) {
            const uint16_t* blk = w_bits + n * K + b * 16;
            float amax_b = 0.0f;
            for (int j = 0; j < 16; ++j) {
                const float a = fabsf((float)oracle_bf16_to_f64(blk[j]));
                if (a > amax_b) amax_b = a;
            }
            const float s_f = (amax_b * gs) / 6.0f;
            const unsigned sbyte = e4m3_round(s_f);
            w_scale[n * (K / 16) + b] = (uint8_t)sbyte;
            const float s = (float)oracle_e4m3(sbyte);
            for (int j = 0; j < 16; j += 2) {
                unsigned c[2];
                for (int h = 0; h < 2; ++h) {
                    if (s == 0.0f) {
                        c[h] = 0;
                    } else {
                        const float w = (float)oracle_bf16_to_f64(blk[j + h]);
                        c[h] = e2m1_round((w * gs) / s);
                    }
                }
                w_packed[n * (K / 2) + b * 8 + j / 2] = (uint8_t)(c[0] | (c[1] << 4));
            }
        }
    }
    return 0;
}

/* A block-scaled FP8 checkpoint tensor as bf16: the first step of the
 * FP8 -> BF16 -> NVFP4 conversion the pages describe for FP8-source weights
 * (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", the MTP-head note: FP8
 * e4m3 in blocks of 128 converted once at load; qwentin README, "Convert a
 * model": block-scaled E4M3 tensors with `*_scale_inv` are dequantised
 * first).  w8: e4m3fn bits [N][K]; scale_inv: fp32 [ceil(N/B)][ceil(K/B)];
 * out: bf16 bits [N][K], each RNE_bf16(fp32(e4m3(w8) * scale_inv of its
 * B x B block)).  Returns 0, or -1 on a bad shape. */
int oracle_fp8_to_bf16(const uint8_t* w8, const float* scale_inv, int64_t block, int64_t N,
                       int64_t K, uint16_t* out)
{
    if (N <= 0 || K <= 0 || block <= 0) return -1;
    const int64_t kb = (K + block - 1) / block;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            const float v = (float)oracle_e4m3(w8[n * K + k]);   /* exact in fp32 */
            const float p = v * scale_inv[(n / block) * kb + k / block];
            out[n * K + k] = oracle_f32_to_bf16_rne(p);
        }
    }
    return 0;
}
