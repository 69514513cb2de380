/*
 * nvfp4_linear.h -- C ABI of libnvfp4_linear.so, the GB300 (sm_103a) NVFP4
 * W4A16 block-scaled linear layer.
 *
 * Operation (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", section 1 "Model
 * dependencies", checkpoint condition 2 -- the compressed-tensors
 * nvfp4-pack-quantized schema -- and the section 1 table, "NVFP4 W4A16"):
 *
 *   w[n,k] = e2m1(code[n,k]) * e4m3(w_scale[n, k/16]) / global_scale
 *   y[m,n] = sum_k x[m,k] * w[n,k]          accumulated in fp32
 *
 * Arguments common to the compute entry points
 *   x            device pointer, bf16 [M, K], row-major, contiguous.
 *   w_packed     device pointer, uint8 [N, K/2]: FP4 e2m1 codes, two per
 *                byte, the low nibble holding the even k.
 *   w_scale      device pointer, uint8 [N, K/16]: fp8 e4m3 (E4M3FN) block
 *                scales, one per 16 consecutive k of a row.
 *   global_scale fp32 scalar; the weights are divided by it (it is the
 *                checkpoint's "448 / amax").  Used as given.
 *   y            device pointer, output, row-major, contiguous (shape and
 *                type per entry point).  Must not overlap the inputs.
 *   M, N, K      M >= 0 activation rows (M == 0 is a no-op; x and y may
 *                then be NULL), N > 0 weight
 *                rows with N % 128 == 0, K > 0 with K % 256 == 0.
 *   stream       a cudaStream_t (0 = the legacy default stream).
 *
 * Ownership: every buffer belongs to the caller.  The library allocates no
 * device or host memory per call and keeps no state besides per-device
 * attributes it caches on first use (device properties, kernel attributes,
 * the address of its device error word) and small caches of encoded TMA
 * descriptors, keyed by every input of the encoding (pointer, sizes, box),
 * and of launch plans, keyed by device, M, N, K and flags.
 *
 * Behaviour: calls are asynchronous on `stream`; they validate on the host,
 * launch one kernel, and return without synchronising.  A rejected call
 * launches nothing.  Kernels are launched with programmatic dependent
 * launch: the prologue and the weight/scale prefetch of a call may overlap
 * the tail of the kernel before it in the stream, while the activations are
 * read, and the output written, only after that kernel has completed.  So
 * the weights and scales must not be written by the kernel immediately
 * before the call in the same stream.  Calls may be captured into a CUDA
 * graph; a captured call keeps the pointers it was given.  A device-side failure (a pipeline wait that timed out)
 * does not fault the context: the kernel winds down and sets a bit in the
 * library's device error word, readable with nvfp4_device_status().
 *
 * Status codes (return values): see NVFP4_* below; nvfp4_status_string()
 * gives a message.
 */
#ifndef NVFP4_LINEAR_H
#define NVFP4_LINEAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_ABI_VERSION 1

#define NVFP4_OK 0
#define NVFP4_ERR_INVALID (-1)      /* null pointer, negative/zero size, bad flags */
#define NVFP4_ERR_MISALIGNED (-2)   /* a pointer is not 16-byte aligned */
#define NVFP4_ERR_SHAPE (-3)        /* K % 256 != 0 or N % 128 != 0 */
#define NVFP4_ERR_LAUNCH (-4)       /* the CUDA runtime refused the launch */
#define NVFP4_ERR_DEVICE (-5)       /* no current device, or not an sm_103 GPU */
#define NVFP4_ERR_TOO_LARGE (-6)    /* nvfp4_linear_host_noalloc: the call does not fit its scratch */

/* Flags of nvfp4_linear_ex. */
#define NVFP4_FLAG_SWIGLU 1u        /* fused gate/up: y = silu(gate) * up */
#define NVFP4_FLAG_F32_OUT 2u       /* write fp32 (before bf16 rounding) */
#define NVFP4_FLAG_FORCE_SMALLM 4u  /* force the warp-MMA few-row kernel (needs M <= 32) */
#define NVFP4_FLAG_FORCE_TCGEMM 8u  /* force the tcgen05 tensor-core kernel */
/* Tuning override of both few-row kernels: split k over n CTAs of one
 * thread-block cluster (1 <= n <= 16, at most K/256) instead of the
 * built-in choice; n = 0 means automatic.  Encode with NVFP4_FLAG_SPLIT(n). */
#define NVFP4_FLAG_SPLIT_SHIFT 8
#define NVFP4_FLAG_SPLIT_MASK (0x1Fu << NVFP4_FLAG_SPLIT_SHIFT)
#define NVFP4_FLAG_SPLIT(n) (((unsigned int)(n) & 0x1Fu) << NVFP4_FLAG_SPLIT_SHIFT)
/* Tuning override of the warp-MMA few-row kernel: CTAs of 16 * n weight
 * rows (1 <= n <= 8, at most 4 when M > 16) instead of the built-in
 * choice; n = 0 means automatic.  For the bf16 tcgen05 few-row kernel it
 * pins the lane groups instead (n = 2: two CTAs per SM, n = 4: one).  A
 * combination that does not fit on the device is rejected with
 * NVFP4_ERR_INVALID. */
#define NVFP4_FLAG_GROUPS_SHIFT 13
#define NVFP4_FLAG_GROUPS_MASK (0xFu << NVFP4_FLAG_GROUPS_SHIFT)
#define NVFP4_FLAG_GROUPS(n) (((unsigned int)(n) & 0xFu) << NVFP4_FLAG_GROUPS_SHIFT)
/* Multiply in bf16, the activations as given (M <= 32): at M <= 8 the
 * warp-MMA few-row kernel in bf16 instead of f16; with NVFP4_FLAG_FORCE_GEMV
 * the bf16 tcgen05 few-row kernel.  (Every default for M = 9..32 is already
 * bf16: the bf16 tcgen05 kernel on weight matrices of at least 2^27 weights
 * at M <= 16, 2^26 at M = 17..24 and 3 * 2^23 at M = 25..32, the warp-MMA
 * kernel otherwise.)  Without it, M <= 8 multiplies in f16: code *
 * scale is exact in f16, and each activation row is brought to f16 after
 * scaling by a power of two taken from the row's running maximum |x|, which
 * is exact for every activation within a factor 2^31 of that maximum; a
 * 256-k stage of a row holding a nonzero value below that window is
 * multiplied in bf16 instead, so the default is exact for every finite bf16
 * activation as well.  The f16 tcgen05 few-row kernel (only when forced)
 * scales by the maximum within each 256-k stage and has no such fallback:
 * there an activation more than 2^31 below its stage's maximum rounds like
 * an f16 subnormal. */
#define NVFP4_FLAG_BF16_MMA (1u << 17)
/* Force a tcgen05 few-row kernel (needs M <= 32): the f16 one, or with
 * NVFP4_FLAG_BF16_MMA the bf16 one. */
#define NVFP4_FLAG_FORCE_GEMV (1u << 18)
/* Test hook of the wait limit (see nvfp4_device_status): the warp-MMA
 * few-row kernel never loads its last k stage and gives each pipeline wait a
 * 1 ms limit, so the waits for that stage run out.  The call still returns
 * and its kernel completes, with bit 0 of the device error word set and the
 * output undefined.  Accepted only together with NVFP4_FLAG_FORCE_SMALLM and
 * NVFP4_FLAG_SPLIT(1) (no thread-block cluster, no TMEM); otherwise
 * NVFP4_ERR_INVALID.  Not for production calls. */
#define NVFP4_FLAG_TEST_STALL (1u << 19)

/* Kernel identifiers returned by nvfp4_linear_kernel_for. */
#define NVFP4_KERNEL_NONE 0
#define NVFP4_KERNEL_SMALLM 1       /* few rows, register-fed warp MMA (forced, or bf16) */
#define NVFP4_KERNEL_TCGEMM 2       /* M > 32: tcgen05 / TMEM tensor-core GEMM */
#define NVFP4_KERNEL_GEMV 3         /* M <= 32: weight streaming, dequantised into TMEM, tcgen05, f16 */
#define NVFP4_KERNEL_GEMV_BF16 4    /* the same in bf16, accumulating in TMEM over all of k */

/* Version of this ABI (NVFP4_ABI_VERSION). */
int nvfp4_abi_version(void);

/* Static message for a status code. Never NULL. */
const char* nvfp4_status_string(int status);

/* y[M, N] bf16 = RNE_bf16(fp32 result).  The linear layer of the pages:
 * MLP gate/up/down and full-attention q/k/v/o projections in decode,
 * speculative verify and prefill. */
int nvfp4_linear(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                 float global_scale, void* y, int64_t M, int64_t N, int64_t K,
                 void* stream);

/* y[M, N] fp32: the same result before the bf16 rounding (for checking the
 * accumulator against an error bound). */
int nvfp4_linear_f32(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                     float global_scale, float* y, int64_t M, int64_t N, int64_t K,
                     void* stream);

/* Fused MLP gate/up projection with SwiGLU epilogue (FlashRT docs section 4,
 * fused gate/up GEMM; qwen36-fp4 README, SwiGLU kernel).  The weight holds
 * gate rows [0, N/2) then up rows [N/2, N), one global scale for both;
 * y[M, N/2] bf16 = silu(g) * u with g, u the fp32 results of the two halves
 * and silu(g) = g / (1 + exp(-g)), computed in fp32. */
int nvfp4_linear_swiglu(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                        float global_scale, void* y, int64_t M, int64_t N, int64_t K,
                        void* stream);

/* As nvfp4_linear_swiglu with fp32 output [M, N/2]. */
int nvfp4_linear_swiglu_f32(const void* x, const uint8_t* w_packed,
                            const uint8_t* w_scale, float global_scale, float* y,
                            int64_t M, int64_t N, int64_t K, void* stream);

/* Fused gate/up projection with SwiGLU where the gate rows [0, N/2) and the
 * up rows [N/2, N) carry their own global scales (a checkpoint whose gate
 * and up projections were quantised separately, stored as one weight; the
 * FlashRT docs, section 4, fuse the pair only "when the gate/up scales
 * allow it" -- here they always can).  Gate results use gate_global_scale,
 * up results up_global_scale; otherwise as nvfp4_linear_swiglu.  `flags`
 * may add NVFP4_FLAG_F32_OUT and the kernel and tuning flags below. */
int nvfp4_linear_swiglu_gs(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                           float gate_global_scale, float up_global_scale, void* y, int64_t M,
                           int64_t N, int64_t K, unsigned int flags, void* stream);

/* One launch over a weight stacked from up to 8 projections that share
 * their input, each with its own global scale -- e.g. a layer's q, k and v
 * projections, quantised as separate checkpoint tensors (FlashRT docs,
 * section 1, condition 3: q/k/v/o are NVFP4; one scale per tensor).
 * w_packed / w_scale hold the segments' rows one after another
 * (segment_rows[i] rows each, summing to N); y[M, N] holds their outputs
 * side by side.  global_scales and segment_rows are host arrays of
 * num_segments (1..8) entries.  `flags` as for nvfp4_linear_ex, without
 * NVFP4_FLAG_SWIGLU.  Rejected (NVFP4_ERR_INVALID): a NULL array, a
 * segment of no rows, rows not summing to N, or num_segments out of range. */
int nvfp4_linear_segmented(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                           const float* global_scales, const int64_t* segment_rows,
                           int num_segments, void* y, int64_t M, int64_t N, int64_t K,
                           unsigned int flags, void* stream);

/* Quantise bf16 weights w[N, K] (device, row-major, 16-byte aligned,
 * K % 16 == 0) into the format the calls above consume: w_packed[N, K/2]
 * (device, 8-byte aligned), w_scale[N, K/16] and *global_scale (device
 * fp32).  The pages (FlashRT docs, section 1, condition 2) fix the format and
 * weight_global_scale = 448 / amax, not the rounding; the steps taken, in
 * fp32 with round-to-nearest-even:
 *   gs = 448 / max|w| (1 for an all-zero tensor);
 *   block scale = e4m3((max|w in block| * gs) / 6), saturating at 448;
 *   code = e2m1((w * gs) / block scale), saturating at 6, sign kept (a
 *   negative weight that rounds to zero is -0); all codes +0 where the
 *   block scale rounds to 0.
 * Non-finite weights are outside this contract.  Asynchronous on `stream`
 * (a memset and three kernels); *global_scale holds the tensor maximum
 * until the last of them completes.  Allocates nothing. */
int nvfp4_quantize(const void* w, int64_t N, int64_t K, uint8_t* w_packed, uint8_t* w_scale,
                   float* global_scale, void* stream);

/* nvfp4_quantize for a block-scaled FP8 checkpoint tensor: the FP8 -> BF16
 * -> NVFP4 conversion (FlashRT docs, "Qwen3.6-27B NVFP4 on RTX 5090", the
 * MTP-head note: FP8 e4m3 in blocks of 128, converted FP8 -> BF16 -> NVFP4
 * once at load; qwentin README, "Convert a model": block-scaled E4M3
 * tensors with `*_scale_inv` are dequantised first).
 *   w_fp8      device, uint8 [N, K]: e4m3fn bits, row-major; 16-byte aligned.
 *   scale_inv  device, fp32 [ceil(N/block), ceil(K/block)], row-major: the
 *              factor of every weight of its block x block tile.
 *   block      the tile edge (128 in the checkpoints above), a multiple of 16.
 * Each weight's bf16 image is RNE_bf16(fp32(e4m3 * scale_inv)); the outputs
 * are then exactly those of nvfp4_quantize on that bf16 tensor (which is
 * never stored: both passes form it on the fly).  K % 16 == 0.  NaN codes
 * (S.1111.111) are outside this contract.  Asynchronous on `stream` (a
 * memset and three kernels); allocates nothing.  Errors: NVFP4_ERR_INVALID
 * (NULL, sizes <= 0), NVFP4_ERR_MISALIGNED, NVFP4_ERR_SHAPE (K or block not
 * a multiple of 16), NVFP4_ERR_LAUNCH, NVFP4_ERR_DEVICE. */
int nvfp4_quantize_fp8(const uint8_t* w_fp8, const float* scale_inv, int64_t block, int64_t N,
                       int64_t K, uint8_t* w_packed, uint8_t* w_scale, float* global_scale,
                       void* stream);

/* General form of nvfp4_linear, _f32, _swiglu and _swiglu_f32; `flags` is
 * an OR of NVFP4_FLAG_*.
 * The FORCE flags pick a kernel regardless of M (for A/B measurements and
 * for checking the kernels against each other on the same inputs). */
int nvfp4_linear_ex(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                    float global_scale, void* y, int64_t M, int64_t N, int64_t K,
                    unsigned int flags, void* stream);

/* nvfp4_linear_ex with the activations and the result in host memory:
 * enqueues on `stream` a transfer of x_host into the caller's device buffer
 * x_dev, the layer (y_dev = x_dev . w^T as nvfp4_linear_ex), and a transfer
 * of y_dev into y_host; nothing is allocated.  (A convenience for callers
 * whose activations live in host memory; the operation is that of
 * nvfp4_linear_ex.)
 *   x_host  host, bf16 [M, K] row-major;  x_dev  device, bf16 [M, K].
 *   y_dev   device, the output of nvfp4_linear_ex for `flags` (bf16, or
 *           fp32 with NVFP4_FLAG_F32_OUT; [M, N], or [M, N/2] with SWIGLU).
 *   y_host  host, same shape and type as y_dev.
 * Transfers: when both host buffers are page-locked and mapped into the
 * device's address space (cudaHostAlloc, cudaHostRegister: every
 * page-locked buffer under unified addressing) and all four buffers are
 * 16-byte aligned, they go directly over the host link (zero-copy): a small
 * kernel reads x_host into x_dev, and the layer's kernel writes its result
 * to y_host as well as y_dev from its epilogue (M <= 32; for M > 32 a
 * second small kernel copies y_dev to y_host).  All are launched like the
 * layer's own kernels as programmatic dependents, so that consecutive calls
 * on a stream overlap (the next call's weights stream in while this one
 * finishes).  The input stage reads x_host before the kernel ahead of it in
 * the stream has completed (as the layer does with its weights), so x_host
 * must not be written by that kernel.  Otherwise one cudaMemcpyAsync each
 * way around the launch; pageable buffers then make the copies synchronise
 * with the host.
 * The host buffers must stay valid, and x_host unchanged, until the stream
 * has passed the call.  Validation and errors as nvfp4_linear_ex (x_dev,
 * y_dev in place of x, y; x_host and y_host must not be NULL when M > 0);
 * NVFP4_ERR_LAUNCH also when a transfer cannot be enqueued (an enqueued
 * input transfer is then left to complete). */
int nvfp4_linear_host(const void* x_host, void* x_dev, const uint8_t* w_packed,
                      const uint8_t* w_scale, float global_scale, void* y_dev, void* y_host,
                      int64_t M, int64_t N, int64_t K, unsigned int flags, void* stream);

/* Bytes of device scratch that nvfp4_linear_host_noalloc owns (8 MiB). */
#define NVFP4_NOALLOC_SCRATCH_BYTES (8 * 1024 * 1024)

/* nvfp4_linear_host for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is a convenience of this library.
 *
 * Some callers cannot call cudaMalloc -- a plug-in inside an application
 * that owns every device allocation, a latency-bound loop where an
 * allocation's implicit device synchronisation is not allowed, a process
 * whose device memory is fully reserved -- yet hold the packed weights and
 * scales on the device already and their activations in host memory.  This
 * entry point runs the layer for them with no device buffer of theirs: the
 * activations' device copy and the device result that nvfp4_linear_host
 * stages through live in one array of NVFP4_NOALLOC_SCRATCH_BYTES that the
 * library itself holds on every device that loads it, for the life of the
 * process.  It allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *   x_host, y_host, w_packed, w_scale, global_scale, M, N, K, flags, stream:
 *           as for nvfp4_linear_host (x_host bf16 [M, K] in host memory;
 *           y_host the result in host memory, [M, N] or [M, N/2] with
 *           SWIGLU, bf16 or fp32 with F32_OUT).  Page-locked host buffers
 *           go zero-copy, others through cudaMemcpyAsync (pageable memory
 *           then makes the copies synchronise with the host).
 * Limit: the activations (M * K * 2 bytes, rounded up to 256) and the
 * result (M * N_out * 2 or 4 bytes) must fit in NVFP4_NOALLOC_SCRATCH_BYTES
 * together; otherwise NVFP4_ERR_TOO_LARGE and nothing is launched.  (Decode,
 * verify and the M = 32 layer's linears of a 5120-wide model fit; a prefill
 * chunk does not.)  Other errors as nvfp4_linear_host.
 * Set-up: the first call on a device looks up the array's device address
 * with that device current; make that first call before any stream capture.
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Nothing in it has to start at zero: each call writes
 * the activations' part and the result's part before reading them.  Calls
 * whose work can overlap on the GPU -- calls on different streams, or from
 * host threads that do not order them on one stream -- race on the array;
 * calls enqueued one after another on one stream do not. */
int nvfp4_linear_host_noalloc(const void* x_host, const uint8_t* w_packed,
                              const uint8_t* w_scale, float global_scale, void* y_host,
                              int64_t M, int64_t N, int64_t K, unsigned int flags,
                              void* stream);

/* Which kernel a call with these sizes and flags would launch
 * (NVFP4_KERNEL_*), or NVFP4_KERNEL_NONE if the call would be rejected.
 * Pure host function: touches no device. */
int nvfp4_linear_kernel_for(int64_t M, int64_t N, int64_t K, unsigned int flags);

/* Read the current device's error word (OR of bits set by kernels since it
 * was last cleared: bit 0 = a pipeline wait timed out) into *bits; clear it
 * if `clear` is non-zero.  Synchronises with the whole device (every stream)
 * first; the read and the clear are one atomic step on the device, so a bit
 * set meanwhile is never lost.  Returns a status. */
int nvfp4_device_status(unsigned int* bits, int clear);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_LINEAR_H */
