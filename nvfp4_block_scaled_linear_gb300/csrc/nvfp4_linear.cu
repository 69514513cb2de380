// nvfp4_linear.cu -- the C ABI of include/nvfp4_linear.h: host-side
// validation, kernel choice by M, TMA tensor-map encoding and launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/nvfp4_linear.h"
#include "gemv_bf16.cuh"
#include "gemv_tc.cuh"
#include "host_io.cuh"
#include "quantize.cuh"
#include "smallm.cuh"
#include "tcgemm.cuh"

namespace {

namespace sm = nvfp4::smallm;
namespace gt = nvfp4::gemvtc;
namespace gb = nvfp4::gemvbf;

// Weight and scale bytes one 16-row group brings per 256-k stage, and the
// weight bytes an SM should keep in flight (HBM latency x its bandwidth share).
constexpr double kGroupBytesPerStage = 16.0 * (256 / 2 + 256 / 16);
constexpr double kWantInFlight = 128.0 * 1024;
constexpr double kLoneCtaEfficiency = 0.74;
// Activation tiles per band of the tensor-core kernel's tile order (16
// tiles of 256 rows of a 5120-wide x: 42 MB, kept in L2 while the band's
// weights stream past).
constexpr int kTcgemmBand = 16;
// Wait limit under NVFP4_FLAG_TEST_STALL: long enough for the loads that are
// issued, short enough for a test.
constexpr uint64_t kTestStallWaitNs = 1000000ull;   // 1 ms

// Bits set by kernels when a pipeline wait gives up (see ptx.cuh), and the
// word as nvfp4_device_status last read it.
__device__ unsigned int g_device_error;
__device__ unsigned int g_device_error_read;

// Read (and, if `clear`, reset) the error word in one atomic step, so that a
// bit set by a kernel running meanwhile is either read or kept.
__global__ void read_device_error_kernel(int clear) {
  g_device_error_read =
      clear ? atomicExch(&g_device_error, 0u) : atomicOr(&g_device_error, 0u);
}

constexpr int kMaxDevices = 64;
constexpr int64_t kSmallMMax = 32;

using SmallmFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, sm::Params);

// The few-row kernel instance for (MT, G, CV, W) (CV: 0 bf16, 1, 2 or 4 f16
// with that many activation converters; W: consumer row-group ways, 4 only
// for bf16); combinations the kernel does not support are never
// instantiated.
template <int MT, int G, int CV, int W>
constexpr SmallmFn smallm_instance() {
  if constexpr (G <= sm::max_groups(MT) && (CV == 0 || MT == 1) && (W == sm::kWays || CV == 0))
    return &sm::smallm_kernel<MT, G, CV, W>;
  else
    return nullptr;
}
template <int MT, int CV, int W = sm::kWays>
SmallmFn smallm_fn(int g) {
  switch (g) {
    case 1: return smallm_instance<MT, 1, CV, W>();
    case 2: return smallm_instance<MT, 2, CV, W>();
    case 3: return smallm_instance<MT, 3, CV, W>();
    case 4: return smallm_instance<MT, 4, CV, W>();
    case 5: return smallm_instance<MT, 5, CV, W>();
    case 6: return smallm_instance<MT, 6, CV, W>();
    case 7: return smallm_instance<MT, 7, CV, W>();
    case 8: return smallm_instance<MT, 8, CV, W>();
    default: return nullptr;
  }
}

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  int max_smem = 0;                    // opt-in shared memory per block
  int smem_per_sm = 0, smem_reserved = 0, regs_per_sm = 0, threads_per_sm = 0;
  unsigned int* err = nullptr;         // device address of g_device_error
  // registers per thread of the warp-MMA kernel by (W == 4, CV, MT, G)
  int smallm_regs[2][5][5][sm::kMaxGroups + 1] = {};
  int gemv_regs[2] = {};               // registers per thread of the tcgen05 few-row kernel (N 16, 32)
  int gemv_bf16_regs[2][2] = {};       // the same, bf16 kernel, by (N 16 / 32, lane groups 2 / 4)
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <int MT, int CV, int W = sm::kWays>
cudaError_t prepare_smallm(DeviceInfo& d) {
  for (int g = 1; g <= sm::max_groups(MT); ++g) {
    const SmallmFn kern = smallm_fn<MT, CV, W>(g);
    if (!kern) continue;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    d.smallm_regs[W == 4][CV][MT][g] = fa.numRegs;
  }
  return cudaSuccess;
}

template <int NM>
cudaError_t prepare_gemv(DeviceInfo& d) {
  const auto kern = &gt::gemv_tc_kernel<NM>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  d.gemv_regs[NM == 16 ? 0 : 1] = fa.numRegs;
  return cudaSuccess;
}

template <int NM, int NI>
cudaError_t prepare_gemv_bf16(DeviceInfo& d) {
  const auto kern = &gb::gemv_bf16_kernel<NM, NI>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  d.gemv_bf16_regs[NM == 16 ? 0 : 1][NI == 2 ? 0 : 1] = fa.numRegs;
  return cudaSuccess;
}

// Resident CTAs per SM for a block of `threads` threads using `regs`
// registers each and `smem` bytes of dynamic shared memory.
int resident_ctas(const DeviceInfo& d, int threads, int regs, int smem) {
  const int warps = (threads + 31) / 32;
  const int regs_per_warp = (regs * 32 + 255) / 256 * 256;
  int n = d.smem_per_sm / (smem + d.smem_reserved);
  if (regs_per_warp > 0) n = std::min(n, d.regs_per_sm / (regs_per_warp * warps));
  n = std::min(n, d.threads_per_sm / threads);
  return std::max(0, std::min(n, 32));
}

// Per-device, one-time set-up.  Returns a status.
int device_setup(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return NVFP4_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return NVFP4_ERR_DEVICE;
    }
    d.supported = (prop.major == 10 && prop.minor == 3);
    d.num_sms = prop.multiProcessorCount;
    d.max_smem = static_cast<int>(prop.sharedMemPerBlockOptin);
    d.smem_per_sm = static_cast<int>(prop.sharedMemPerMultiprocessor);
    d.smem_reserved = static_cast<int>(prop.reservedSharedMemPerBlock);
    d.regs_per_sm = prop.regsPerMultiprocessor;
    d.threads_per_sm = prop.maxThreadsPerMultiProcessor;
    if (d.supported) {
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
          cudaGetLastError();
          return NVFP4_ERR_DEVICE;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
      void* err_addr = nullptr;
      if (cudaGetSymbolAddress(&err_addr, g_device_error) != cudaSuccess ||
          prepare_smallm<1, 0>(d) != cudaSuccess ||
          prepare_smallm<3, 0>(d) != cudaSuccess ||
          prepare_smallm<4, 0>(d) != cudaSuccess ||
          prepare_smallm<1, 1>(d) != cudaSuccess ||
          prepare_smallm<1, 2>(d) != cudaSuccess ||
          prepare_smallm<1, 4>(d) != cudaSuccess ||
          prepare_smallm<2, 0, 4>(d) != cudaSuccess ||
          prepare_gemv<16>(d) != cudaSuccess || prepare_gemv<32>(d) != cudaSuccess ||
          prepare_gemv_bf16<16, 2>(d) != cudaSuccess ||
          prepare_gemv_bf16<16, 4>(d) != cudaSuccess ||
          prepare_gemv_bf16<32, 2>(d) != cudaSuccess ||
          prepare_gemv_bf16<32, 4>(d) != cudaSuccess ||
          cudaFuncSetAttribute(nvfp4::tcgemm::tcgemm_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               nvfp4::tcgemm::kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return NVFP4_ERR_DEVICE;
      }
      d.err = static_cast<unsigned int*>(err_addr);
    }
    d.ready = true;
  }
  if (!d.supported) return NVFP4_ERR_DEVICE;
  *out = &d;
  return NVFP4_OK;
}

// Encoding a tensor map costs microseconds of host time, comparable to a
// decode-sized kernel, so encoded maps are kept in a small direct-mapped
// cache.  The key holds every encoding input, so a hit is always valid.
struct MapKey {
  const void* base;
  uint64_t dim0, dim1, row_bytes;
  uint32_t box0, box1;
  int dtype, swizzle;
  bool operator==(const MapKey& o) const {
    return base == o.base && dim0 == o.dim0 && dim1 == o.dim1 && row_bytes == o.row_bytes &&
           box0 == o.box0 && box1 == o.box1 && dtype == o.dtype && swizzle == o.swizzle;
  }
};
struct MapSlot {
  bool valid = false;
  MapKey key{};
  CUtensorMap map{};
};
constexpr int kMapCacheSlots = 256;
MapSlot g_map_cache[kMapCacheSlots];
std::mutex g_map_mutex;

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
               uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
               CUtensorMapSwizzle swizzle) {
  const MapKey key{base, dim0, dim1, row_bytes, box0, box1, static_cast<int>(dtype),
                   static_cast<int>(swizzle)};
  uint64_t h = reinterpret_cast<uintptr_t>(base) >> 4;
  h ^= dim0 * 0x9E3779B97F4A7C15ull ^ dim1 * 0xC2B2AE3D27D4EB4Full ^ (uint64_t(box1) << 20) ^
       (uint64_t(box0) << 7) ^ uint64_t(swizzle) ^ (uint64_t(dtype) << 3);
  h ^= h >> 29;
  MapSlot& slot = g_map_cache[h % kMapCacheSlots];
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    if (slot.valid && slot.key == key) {
      *map = slot.map;
      return true;
    }
  }
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  if (g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  slot.valid = true;
  slot.key = key;
  slot.map = *map;
  return true;
}

// Host form of a segmented call: up to kMaxSegments row segments with their
// global scales (count == 0: an ordinary call).
struct SegSpec {
  int count = 0;
  int64_t end[nvfp4::kMaxSegments] = {};
  float gs[nvfp4::kMaxSegments] = {};
};

// Fill a kernel's segment table, each scale in the kernel's units:
// weight_pow2 / global_scale (2^10 for bf16 operands, 1 for f16).
nvfp4::SegScales seg_table(const SegSpec* spec, double weight_pow2) {
  nvfp4::SegScales t{};
  if (!spec || spec->count == 0) return t;
  t.n = spec->count;
  for (int i = 0; i < spec->count; ++i) {
    t.end[i] = spec->end[i];
    t.scale[i] = static_cast<float>(weight_pow2 / static_cast<double>(spec->gs[i]));
  }
  return t;
}

// The global scale is applied as one fp32 multiply by 2^10 / global_scale
// (2^10 undoes the exponent offset of the bf16 dequantised weights).
float out_scale(float global_scale) {
  return static_cast<float>(static_cast<double>(nvfp4::kWeightPow2) /
                            static_cast<double>(global_scale));
}

int validate(const void* x, const void* wp, const void* ws, const void* y, int64_t M,
             int64_t N, int64_t K, unsigned int flags) {
  if (M < 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID;
  // With M == 0 nothing is read from x or written to y: an empty tensor's
  // null data pointer is fine there.
  if (!wp || !ws || (M > 0 && (!x || !y))) return NVFP4_ERR_INVALID;
  if (flags & ~(NVFP4_FLAG_SWIGLU | NVFP4_FLAG_F32_OUT | NVFP4_FLAG_FORCE_SMALLM |
                NVFP4_FLAG_FORCE_TCGEMM | NVFP4_FLAG_SPLIT_MASK | NVFP4_FLAG_GROUPS_MASK |
                NVFP4_FLAG_BF16_MMA | NVFP4_FLAG_FORCE_GEMV | NVFP4_FLAG_TEST_STALL))
    return NVFP4_ERR_INVALID;
  // the wait-limit test hook: the warp-MMA kernel without a k split only
  // (no cluster barrier and no TMEM for a stalled CTA to hold)
  if ((flags & NVFP4_FLAG_TEST_STALL) &&
      (!(flags & NVFP4_FLAG_FORCE_SMALLM) ||
       (flags & NVFP4_FLAG_SPLIT_MASK) != NVFP4_FLAG_SPLIT(1)))
    return NVFP4_ERR_INVALID;
  if (((flags & NVFP4_FLAG_SPLIT_MASK) >> NVFP4_FLAG_SPLIT_SHIFT) > sm::kMaxSplit ||
      ((flags & NVFP4_FLAG_GROUPS_MASK) >> NVFP4_FLAG_GROUPS_SHIFT) > sm::kMaxGroups)
    return NVFP4_ERR_INVALID;
  const unsigned int force = flags & (NVFP4_FLAG_FORCE_SMALLM | NVFP4_FLAG_FORCE_TCGEMM |
                                      NVFP4_FLAG_FORCE_GEMV);
  if (force & (force - 1)) return NVFP4_ERR_INVALID;        // at most one
  if ((flags & NVFP4_FLAG_BF16_MMA) && (flags & NVFP4_FLAG_FORCE_TCGEMM)) return NVFP4_ERR_INVALID;
  if ((flags & (NVFP4_FLAG_FORCE_SMALLM | NVFP4_FLAG_FORCE_GEMV | NVFP4_FLAG_BF16_MMA)) &&
      M > kSmallMMax)
    return NVFP4_ERR_INVALID;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(wp) |
                        reinterpret_cast<uintptr_t>(ws) | reinterpret_cast<uintptr_t>(y);
  if (mis & 15u) return NVFP4_ERR_MISALIGNED;
  if (K % 256 != 0 || N % 128 != 0) return NVFP4_ERR_SHAPE;
  // tensor-map and grid limits
  if (K > (int64_t(1) << 31) || N > (int64_t(1) << 31) || M > (int64_t(1) << 24))
    return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

// Kernel by M (and, for M = 9..32, the weight size), from graph-timed
// measurements on GB300: M <= 8 the warp-MMA kernel in f16 (decode 18.5 us
// against 29.5-32 us for the tcgen05 few-row kernels); M = 9..32 the bf16
// tcgen05 few-row kernel on weight matrices of at least kBf16GemvMinWeights(M)
// and the warp-MMA kernel in bf16 below.  The crossover falls as M grows,
// the warp MMAs' work growing with M while the tensor core's does not:
//   M = 12/16: 34816 x 5120 40.7 us against 41.0-41.2 (tcgen05 ahead),
//              5120 x 17408 27.4-27.8 against 24.5-25.1 (warp MMA ahead);
//   M = 24:    5120 x 17408 28.2 against 29.2, 12288 x 5120 22.5 against 19.6;
//   M = 32:    5120 x 6144 14.8 against 16.9, 12288 x 5120 22.8 against 28.7,
//              8192 x 5120 16.4 against 15.3, 4096 x 4096 10.9 against 9.6.
// The f16 tcgen05 few-row kernel runs only when forced.  Every default above
// M = 8 multiplies the activations exactly (bf16).
constexpr int64_t kBf16GemvMinWeights(int64_t M) {
  return M <= 16 ? int64_t(1) << 27 : M <= 24 ? int64_t(1) << 26 : int64_t(3) << 23;
}

int kernel_for(int64_t M, int64_t N, int64_t K, unsigned int flags) {
  if (flags & NVFP4_FLAG_FORCE_SMALLM) return NVFP4_KERNEL_SMALLM;
  if (flags & NVFP4_FLAG_FORCE_TCGEMM) return NVFP4_KERNEL_TCGEMM;
  if (flags & NVFP4_FLAG_FORCE_GEMV)
    return (flags & NVFP4_FLAG_BF16_MMA) ? NVFP4_KERNEL_GEMV_BF16 : NVFP4_KERNEL_GEMV;
  if (M > kSmallMMax) return NVFP4_KERNEL_TCGEMM;
  if (M > 8 && N * K >= kBf16GemvMinWeights(M)) return NVFP4_KERNEL_GEMV_BF16;
  return NVFP4_KERNEL_SMALLM;
}

// Plans depend only on the device and (M, N, K, flags), and the search
// over CTA shapes costs microseconds of host time per call -- as much as a
// decode-sized kernel's launch -- so each planner keeps its results in a
// small direct-mapped cache (a miss recomputes; a hit is always valid, the
// key holding every input of the search).
template <typename Plan>
class PlanMemo {
 public:
  template <typename Fn>
  Plan get(const DeviceInfo& d, int64_t M, int64_t N, int64_t K, unsigned int flags, Fn&& make) {
    const Key key{&d, M, N, K, flags};
    uint64_t h = static_cast<uint64_t>(M) * 0x9E3779B97F4A7C15ull ^
                 static_cast<uint64_t>(N) * 0xC2B2AE3D27D4EB4Full ^
                 static_cast<uint64_t>(K) * 0x165667B19E3779F9ull ^ (uint64_t(flags) << 1) ^
                 (reinterpret_cast<uintptr_t>(&d) >> 4);
    h ^= h >> 31;
    Slot& slot = slots_[h % kSlots];
    {
      std::lock_guard<std::mutex> lock(mu_);
      if (slot.valid && slot.key == key) return slot.plan;
    }
    const Plan plan = make();
    std::lock_guard<std::mutex> lock(mu_);
    slot.valid = true;
    slot.key = key;
    slot.plan = plan;
    return plan;
  }

 private:
  struct Key {
    const DeviceInfo* dev;
    int64_t M, N, K;
    unsigned int flags;
    bool operator==(const Key& o) const {
      return dev == o.dev && M == o.M && N == o.N && K == o.K && flags == o.flags;
    }
  };
  struct Slot {
    bool valid = false;
    Key key{};
    Plan plan{};
  };
  static constexpr int kSlots = 64;
  Slot slots_[kSlots];
  std::mutex mu_;
};

struct SmallmPlan {
  int groups = 0;
  int split = 0;
  int stages = 0;
  int64_t row_blocks = 0;
};

// Choose the CTA height (G groups of 16 rows), the k split and the ring
// depth.  Cost model: the work of the busiest SM, ceil(CTAs / SMs) x
// (G x stages per CTA + a fixed per-CTA cost of two stages), inflated when
// the rings of an SM hold less than ~128 KB of weights in flight; grids that
// are resident in one wave win over those that are not; ties go to fewer
// CTAs.  Overrides in `flags` pin G or the split.
template <int MT, int CV, int W>
SmallmPlan plan_smallm(const DeviceInfo& d, int64_t M, int64_t N, int64_t K,
                       unsigned int flags) {
  const bool swiglu = flags & NVFP4_FLAG_SWIGLU;
  const int64_t T = K / sm::kStageK;
  const int want_split = (flags & NVFP4_FLAG_SPLIT_MASK) >> NVFP4_FLAG_SPLIT_SHIFT;
  const int want_groups = (flags & NVFP4_FLAG_GROUPS_MASK) >> NVFP4_FLAG_GROUPS_SHIFT;
  const int64_t unit_rows = swiglu ? N / 2 : N;
  constexpr bool F16 = CV > 0;
  const int threads = sm::threads_for(CV, W);
  static const int kStageChoices[] = {3, 4, 5, 6, 8};
  SmallmPlan best;
  double best_cost = -1.0;
  int64_t best_ctas = 0;
  bool best_one_wave = false;
  for (int g = 1; g <= sm::max_groups(MT); ++g) {
    if (want_groups && g != want_groups) continue;
    const int regs = d.smallm_regs[W == 4][CV][MT][g];
    if (regs <= 0) continue;
    const int64_t rows_per_cta = swiglu ? 8 * g : 16 * g;
    const int64_t row_blocks = (unit_rows + rows_per_cta - 1) / rows_per_cta;
    for (int stages : kStageChoices) {
      const sm::SmemLayout lay = sm::make_layout(MT, g, stages, F16, static_cast<int>(M));
      if (lay.total > d.max_smem || !sm::layout_ok(lay, MT, g)) continue;
      const int occ = resident_ctas(d, threads, regs, lay.total);
      if (occ <= 0) continue;
      const int64_t slots = static_cast<int64_t>(d.num_sms) * occ;
      const int s_max = want_split ? want_split : 8;
      for (int s = 1; s <= s_max && s <= T; ++s) {
        if (want_split && s != want_split) continue;
        const int64_t ctas = row_blocks * s;
        const bool one_wave = ctas <= slots;
        const int64_t per_sm = (ctas + d.num_sms - 1) / d.num_sms;
        // bytes a stage brings: the weights and scales of its g groups and,
        // with four 8-row activation tiles (16 KB a stage, more than most
        // CTAs' weights), the activations: o at M = 32 (5120 x 6144) 19.9 ->
        // 17.9 us, 1024 x 4096 17.7 -> 7.3; counting them at M = 17..24 as
        // well cost 2-9%
        const double stage_bytes = g * kGroupBytesPerStage + (MT == 4 ? lay.x_tx : 0);
        const double in_flight =
            static_cast<double>(std::min<int64_t>(per_sm, occ)) * (stages - 1) * stage_bytes;
        double cost = static_cast<double>(per_sm) * g * ((T + s - 1) / s + 2);
        if (in_flight < kWantInFlight) cost *= kWantInFlight / in_flight;
        // A lone CTA on an SM issues ~26% slower than two sharing it (fewer
        // warps to hide latency; measured on the decode shape).  Not so for
        // three or four 8-row activation tiles (M = 17..32): q/k/v at M = 32
        // (8192 x 5120) takes 18.3 us with 128 lone CTAs against 20.5 us with
        // two CTAs per SM and a split of 2.
        if (MT <= 2 && std::min<int64_t>(per_sm, occ) < 2) cost /= kLoneCtaEfficiency;
        const bool better =
            best_cost < 0 || (one_wave && !best_one_wave) ||
            (one_wave == best_one_wave &&
             (cost < best_cost * 0.999 || (cost <= best_cost * 1.001 && ctas < best_ctas)));
        if (better) {
          best_cost = cost;
          best_ctas = ctas;
          best_one_wave = one_wave;
          best.groups = g;
          best.split = s;
          best.stages = stages;
          best.row_blocks = row_blocks;
        }
      }
    }
  }
  return best;
}

template <int MT, int CV, int W = sm::kWays>
int launch_smallm(const DeviceInfo& d, const void* x, const uint8_t* wp, const uint8_t* ws,
                  float gs, float gs_up, void* y, int64_t M, int64_t N, int64_t K, unsigned int flags,
                  cudaStream_t stream, const SegSpec* segs,
                  void* y_host) {
  constexpr bool F16 = CV > 0;
  const bool swiglu = flags & NVFP4_FLAG_SWIGLU;
  static PlanMemo<SmallmPlan> memo;
  const SmallmPlan plan =
      memo.get(d, M, N, K, flags, [&] { return plan_smallm<MT, CV, W>(d, M, N, K, flags); });
  if (plan.groups == 0) return NVFP4_ERR_INVALID;   // overrides that cannot run
  const int half_rows = 8 * plan.groups;
  CUtensorMap tw, ts, tx;
  const bool x_ok =
      MT == 1 ? encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, K * 2, sm::kStageK,
                          static_cast<uint32_t>(M), CU_TENSOR_MAP_SWIZZLE_NONE)
              : encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, K * 2, 64, MT * 8,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wp, K / 2, N, K / 2, 128, half_rows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws, K / 16, N, K / 16, 16, half_rows,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !x_ok)
    return NVFP4_ERR_LAUNCH;

  sm::Params p;
  p.y = y;
  p.y_host = y_host;
  p.M = M;
  p.N = N;
  p.K = K;
  // f16 weights are exact code * scale; the bf16 ones carry 2^-10
  p.out_scale = F16 ? static_cast<float>(1.0 / static_cast<double>(gs)) : out_scale(gs);
  p.out_scale_up = F16 ? static_cast<float>(1.0 / static_cast<double>(gs_up)) : out_scale(gs_up);
  p.seg = seg_table(segs, F16 ? 1.0 : static_cast<double>(nvfp4::kWeightPow2));
  p.stages_total = static_cast<int>(K / sm::kStageK);
  p.split = plan.split;
  p.lay = sm::make_layout(MT, plan.groups, plan.stages, F16, static_cast<int>(M));
  p.out_f32 = (flags & NVFP4_FLAG_F32_OUT) ? 1 : 0;
  p.swiglu = swiglu ? 1 : 0;
  p.err = d.err;
  p.test_stall = (flags & NVFP4_FLAG_TEST_STALL) ? 1 : 0;
  p.wait_ns = p.test_stall ? kTestStallWaitNs : nvfp4::kWaitTimeoutNs;

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(plan.row_blocks), static_cast<unsigned>(plan.split), 1);
  cfg.blockDim = dim3(sm::threads_for(CV, W), 1, 1);
  cfg.dynamicSmemBytes = p.lay.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(plan.split);
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: the prologue and the weight prefetch may
  // overlap the tail of the preceding kernel in the stream.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, smallm_fn<MT, CV, W>(plan.groups), tw, ts, tx, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

struct GemvPlan {
  int split = 0;
  int stages = 0;
  int64_t row_blocks = 0;
};

// The tcgen05 few-row kernel: 128 weight rows per CTA.  Ring depth: the
// deepest that keeps the most CTAs resident per SM.  Split: the cost is the
// busiest SM's stages (ceil(CTAs / SMs) x (stages per CTA + a fixed
// per-CTA cost)); grids resident in one wave win over those that are not;
// ties go to fewer CTAs.  NVFP4_FLAG_SPLIT pins the split.
template <int NM>
GemvPlan plan_gemv(const DeviceInfo& d, int64_t M, int64_t N, int64_t K, unsigned int flags) {
  GemvPlan best;
  const int64_t T = K / gt::kStageK;
  const int want_split = (flags & NVFP4_FLAG_SPLIT_MASK) >> NVFP4_FLAG_SPLIT_SHIFT;
  const int regs = d.gemv_regs[NM == 16 ? 0 : 1];
  int occ = 0, stages = 0;
  for (int s = 2; s <= 8; ++s) {
    const gt::SmemLayout lay = gt::make_layout(NM, static_cast<int>(M), s);
    if (lay.total > d.max_smem || !gt::layout_ok(lay, NM)) continue;
    const int o = resident_ctas(d, gt::Roles<NM>::kThreads, regs, lay.total);
    if (o > occ || (o == occ && o > 0)) {
      occ = o;
      stages = s;
    }
  }
  if (occ == 0) return best;
  best.stages = stages;
  best.row_blocks = N / gt::kRows;                  // SwiGLU: 64 gate + 64 up rows, same count
  const int64_t slots = static_cast<int64_t>(d.num_sms) * occ;
  double best_cost = -1.0;
  int64_t best_ctas = 0;
  bool best_one_wave = false;
  const int s_max = static_cast<int>(std::min<int64_t>(T, gt::kMaxSplit));
  for (int s = 1; s <= s_max; ++s) {
    if (want_split && s != want_split) continue;
    const int64_t ctas = best.row_blocks * s;
    const bool one_wave = ctas <= slots;
    const int64_t per_sm = (ctas + d.num_sms - 1) / d.num_sms;
    const double cost = static_cast<double>(per_sm) * (static_cast<double>((T + s - 1) / s) + 1.5);
    const bool better =
        best_cost < 0 || (one_wave && !best_one_wave) ||
        (one_wave == best_one_wave &&
         (cost < best_cost * 0.999 || (cost <= best_cost * 1.001 && ctas < best_ctas)));
    if (better) {
      best_cost = cost;
      best_ctas = ctas;
      best_one_wave = one_wave;
      best.split = s;
    }
  }
  if (best.split == 0) best.stages = 0;
  return best;
}

template <int NM>
int launch_gemv(const DeviceInfo& d, const void* x, const uint8_t* wp, const uint8_t* ws,
                float gs, float gs_up, void* y, int64_t M, int64_t N, int64_t K, unsigned int flags,
                cudaStream_t stream, const SegSpec* segs,
                  void* y_host) {
  static PlanMemo<GemvPlan> memo;
  const GemvPlan plan =
      memo.get(d, M, N, K, flags, [&] { return plan_gemv<NM>(d, M, N, K, flags); });
  if (plan.stages == 0) return NVFP4_ERR_INVALID;   // an override that cannot run
  CUtensorMap tw, ts, tx;
  if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wp, K / 2, N, K / 2, 128, gt::kHalfRows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws, K / 16, N, K / 16, 16, gt::kHalfRows,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, K * 2, gt::kStageK,
                 static_cast<uint32_t>(M), CU_TENSOR_MAP_SWIZZLE_NONE))
    return NVFP4_ERR_LAUNCH;
  gt::Params p;
  p.y = y;
  p.y_host = y_host;
  p.M = M;
  p.N = N;
  p.K = K;
  p.out_scale = static_cast<float>(1.0 / static_cast<double>(gs));   // f16 weights are exact
  p.out_scale_up = static_cast<float>(1.0 / static_cast<double>(gs_up));
  p.seg = seg_table(segs, 1.0);
  p.stages_total = static_cast<int>(K / gt::kStageK);
  p.split = plan.split;
  p.lay = gt::make_layout(NM, static_cast<int>(M), plan.stages);
  p.out_f32 = (flags & NVFP4_FLAG_F32_OUT) ? 1 : 0;
  p.swiglu = (flags & NVFP4_FLAG_SWIGLU) ? 1 : 0;
  p.err = d.err;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(plan.row_blocks), static_cast<unsigned>(plan.split), 1);
  cfg.blockDim = dim3(gt::Roles<NM>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.lay.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(plan.split);
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gt::gemv_tc_kernel<NM>, tw, ts, tx, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

struct GemvBfPlan {
  int split = 0;
  int stages = 0;
  int64_t row_blocks = 0;
  double cost = -1.0;
};

// The bf16 tcgen05 few-row kernel with NI lane groups: the deepest ring that
// keeps exactly Roles::kCtasPerSm CTAs resident per SM (TMEM is split
// between them), then the split as for plan_gemv.
template <int NM, int NI>
GemvBfPlan plan_gemv_bf16(const DeviceInfo& d, int64_t N, int64_t K, unsigned int flags) {
  using R = gb::Roles<NM, NI>;
  GemvBfPlan best;
  const int64_t T = K / gb::kStageK;
  const int want_split = (flags & NVFP4_FLAG_SPLIT_MASK) >> NVFP4_FLAG_SPLIT_SHIFT;
  const int regs = d.gemv_bf16_regs[NM == 16 ? 0 : 1][NI == 2 ? 0 : 1];
  int stages = 0;
  for (int s = 2; s <= 12; ++s) {
    const gb::SmemLayout lay = gb::make_layout(NM, NI, s);
    if (lay.total > d.max_smem || !gb::layout_ok(lay, NM)) continue;
    if (resident_ctas(d, R::kThreads, regs, lay.total) == R::kCtasPerSm) stages = s;
  }
  if (stages == 0) return best;
  best.row_blocks = N / gb::kRows;                  // SwiGLU: 64 gate + 64 up rows, same count
  const int64_t slots = static_cast<int64_t>(d.num_sms) * R::kCtasPerSm;
  int64_t best_ctas = 0;
  bool best_one_wave = false;
  const int s_max = static_cast<int>(std::min<int64_t>(T, gb::kMaxSplit));
  for (int s = 1; s <= s_max; ++s) {
    if (want_split && s != want_split) continue;
    const int64_t ctas = best.row_blocks * s;
    const bool one_wave = ctas <= slots;
    const int64_t per_sm = (ctas + d.num_sms - 1) / d.num_sms;
    const double cost = static_cast<double>(per_sm) * (static_cast<double>((T + s - 1) / s) + 1.5);
    const bool better =
        best.cost < 0 || (one_wave && !best_one_wave) ||
        (one_wave == best_one_wave &&
         (cost < best.cost * 0.999 || (cost <= best.cost * 1.001 && ctas < best_ctas)));
    if (better) {
      best.cost = cost;
      best_ctas = ctas;
      best_one_wave = one_wave;
      best.split = s;
    }
  }
  if (best.split > 0) best.stages = stages;
  return best;
}

template <int NM, int NI>
int launch_gemv_bf16(const DeviceInfo& d, const void* x, const uint8_t* wp, const uint8_t* ws,
                     float gs, float gs_up, void* y, int64_t M, int64_t N, int64_t K,
                     unsigned int flags, cudaStream_t stream, const SegSpec* segs,
                  void* y_host) {
  static PlanMemo<GemvBfPlan> memo;
  const GemvBfPlan plan =
      memo.get(d, 0, N, K, flags, [&] { return plan_gemv_bf16<NM, NI>(d, N, K, flags); });
  if (plan.stages == 0) return NVFP4_ERR_INVALID;   // an override that cannot run
  CUtensorMap tw, ts, tx;
  if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wp, K / 2, N, K / 2, 128, gb::kHalfRows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws, K / 16, N, K / 16, 16, gb::kHalfRows,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, K * 2, gb::kJobK, NM,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4_ERR_LAUNCH;
  gb::Params p;
  p.y = y;
  p.y_host = y_host;
  p.M = M;
  p.N = N;
  p.K = K;
  p.out_scale = out_scale(gs);                      // the bf16 weights carry 2^-10
  p.out_scale_up = out_scale(gs_up);
  p.seg = seg_table(segs, static_cast<double>(nvfp4::kWeightPow2));
  p.stages_total = static_cast<int>(K / gb::kStageK);
  p.split = plan.split;
  p.lay = gb::make_layout(NM, NI, plan.stages);
  p.out_f32 = (flags & NVFP4_FLAG_F32_OUT) ? 1 : 0;
  p.swiglu = (flags & NVFP4_FLAG_SWIGLU) ? 1 : 0;
  p.err = d.err;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(plan.row_blocks), static_cast<unsigned>(plan.split), 1);
  cfg.blockDim = dim3(gb::Roles<NM, NI>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.lay.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(plan.split);
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gb::gemv_bf16_kernel<NM, NI>, tw, ts, tx, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

// Lane groups: NVFP4_FLAG_GROUPS(2 | 4) pins them; otherwise two (two CTAs
// per SM) when the row blocks alone fill the SMs, else four (one CTA per SM,
// the larger TMEM share suits the k splits that fill the SMs then).
template <int NM>
int launch_gemv_bf16_any(const DeviceInfo& d, const void* x, const uint8_t* wp,
                         const uint8_t* ws, float gs, float gs_up, void* y, int64_t M, int64_t N,
                         int64_t K, unsigned int flags, cudaStream_t stream, const SegSpec* segs,
                  void* y_host) {
  int want = (flags & NVFP4_FLAG_GROUPS_MASK) >> NVFP4_FLAG_GROUPS_SHIFT;
  if (want != 0 && want != 2 && want != 4) return NVFP4_ERR_INVALID;
  if (want == 0) want = N / gb::kRows >= d.num_sms ? 2 : 4;
  if (want == 2)
    return launch_gemv_bf16<NM, 2>(d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
  return launch_gemv_bf16<NM, 4>(d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
}

int launch_tcgemm(const DeviceInfo& d, const void* x, const uint8_t* wp, const uint8_t* ws,
                  float gs, float gs_up, void* y, int64_t M, int64_t N, int64_t K, unsigned int flags,
                  cudaStream_t stream, const SegSpec* segs) {
  namespace T = nvfp4::tcgemm;
  const bool swiglu = flags & NVFP4_FLAG_SWIGLU;
  CUtensorMap tx, tw, ts;
  if (!encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, K * 2, T::kStageK, T::kTileX,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wp, K / 2, N, K / 2, T::kStageK / 2, 64,
                 CU_TENSOR_MAP_SWIZZLE_32B) ||
      !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws, K / 16, N, K / 16, 16, 64,
                 CU_TENSOR_MAP_SWIZZLE_NONE))
    return NVFP4_ERR_LAUNCH;
  T::Params p;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.out_scale = out_scale(gs);
  p.out_scale_up = out_scale(gs_up);
  p.seg = seg_table(segs, static_cast<double>(nvfp4::kWeightPow2));
  p.out_f32 = (flags & NVFP4_FLAG_F32_OUT) ? 1 : 0;
  p.swiglu = swiglu ? 1 : 0;
  p.err = d.err;
  const int64_t tiles_w = swiglu ? (N / 2) / 64 : N / T::kTileW;
  const int64_t tiles_x = (M + T::kTileX - 1) / T::kTileX;
  if (tiles_w * tiles_x > INT32_MAX) return NVFP4_ERR_SHAPE;
  p.tiles_w = static_cast<int>(tiles_w);
  p.tiles_x = static_cast<int>(tiles_x);
  p.tiles_total = static_cast<int>(tiles_w * tiles_x);
  p.band = static_cast<int>(std::min<int64_t>(tiles_x, kTcgemmBand));
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  // persistent: one CTA per SM (its shared memory and TMEM allow no more)
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(p.tiles_total, d.num_sms)), 1, 1);
  cfg.blockDim = dim3(T::kThreads, 1, 1);
  cfg.dynamicSmemBytes = T::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, T::tcgemm_kernel, tx, tw, ts, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

// y_host (few-row kernels only): a second copy of the output, written by the
// kernel's epilogue into host memory mapped into the device.
int run(const void* x, const uint8_t* wp, const uint8_t* ws, float gs, float gs_up, void* y,
        int64_t M, int64_t N, int64_t K, unsigned int flags, void* stream_ptr,
        const SegSpec* segs = nullptr, void* y_host = nullptr) {
  int st = validate(x, wp, ws, y, M, N, K, flags);
  if (st != NVFP4_OK) return st;
  if (M == 0) return NVFP4_OK;
  DeviceInfo* d = nullptr;
  st = device_setup(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int kernel = kernel_for(M, N, K, flags);
  if (kernel == NVFP4_KERNEL_GEMV_BF16) {
    if (M <= 16)
      return launch_gemv_bf16_any<16>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
    return launch_gemv_bf16_any<32>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
  }
  if (kernel == NVFP4_KERNEL_GEMV) {
    if (M <= 16) return launch_gemv<16>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
    return launch_gemv<32>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
  }
  if (kernel == NVFP4_KERNEL_SMALLM) {
    switch ((M + 7) / 8) {
      case 1:
        // f16 with one activation converter up to M = 3, two at M = 4 and
        // four from M = 5: the converters' per-row work (the exponent and
        // the f16 window check) sets the pace of a stage from M = 3 on
        // (verify, M = 7: 21.3 us with four against 23.5 with two; decode,
        // M = 1: 22.0 us with one)
        if (flags & NVFP4_FLAG_BF16_MMA)
          return launch_smallm<1, 0>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
        if (M <= 3)
          return launch_smallm<1, 1>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
        if (M == 4)
          return launch_smallm<1, 2>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
        return launch_smallm<1, 4>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
      // M = 9..16: sixteen consumer warps (two 8-row activation tiles each
      // leave them half the accumulators of eight): 16.0 us against 16.6
      // on 8192 x 5120 at M = 16 (and no gain at M = 17..32, which keep
      // eight)
      case 2: return launch_smallm<2, 0, 4>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
      case 3: return launch_smallm<3, 0>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
      default: return launch_smallm<4, 0>(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs, y_host);
    }
  }
  // (the tensor-core kernel writes no second output: a large M's result goes
  // to host memory after the kernel, not from its epilogue)
  if (y_host) return NVFP4_ERR_INVALID;
  return launch_tcgemm(*d, x, wp, ws, gs, gs_up, y, M, N, K, flags, stream, segs);
}

// Grid of a quantiser pass: as many CTAs as fit on the device at once (its
// grid-stride loop then runs in one wave), fewer for a small tensor.
template <typename Kernel>
unsigned resident_grid(Kernel kernel, int num_sms, int64_t units) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, nvfp4::quant::kThreads, 0) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int64_t need = (units + nvfp4::quant::kThreads - 1) / nvfp4::quant::kThreads;
  return static_cast<unsigned>(std::max<int64_t>(
      1, std::min<int64_t>(static_cast<int64_t>(num_sms) * per_sm, need)));
}

// The device address of a page-locked host buffer mapped into the current
// device's address space, or nullptr (pageable memory, device memory).
void* device_view(const void* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// One staging kernel of the host-buffer entry point, launched as a
// programmatic dependent of the preceding kernel in the stream.
int launch_staging(void (*kernel)(const uint4*, uint4*, int64_t), const uint4* src, uint4* dst,
                   int64_t n, int num_sms, cudaStream_t stream) {
  const int64_t need = (n + nvfp4::hostio::kThreads - 1) / nvfp4::hostio::kThreads;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(
      std::max<int64_t>(1, std::min<int64_t>(need, static_cast<int64_t>(num_sms) * 4))));
  cfg.blockDim = dim3(nvfp4::hostio::kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, src, dst, n) != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

}  // namespace

extern "C" {

int nvfp4_abi_version(void) { return NVFP4_ABI_VERSION; }

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID: return "invalid argument (null pointer, size or flags)";
    case NVFP4_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case NVFP4_ERR_SHAPE: return "unsupported shape (need K % 256 == 0 and N % 128 == 0)";
    case NVFP4_ERR_LAUNCH: return "CUDA launch failed";
    case NVFP4_ERR_DEVICE: return "no usable sm_103 device";
    case NVFP4_ERR_TOO_LARGE:
      return "activations plus result exceed the fixed scratch of nvfp4_linear_host_noalloc";
    default: return "unknown status";
  }
}

int nvfp4_linear(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                 float global_scale, void* y, int64_t M, int64_t N, int64_t K, void* stream) {
  return run(x, w_packed, w_scale, global_scale, global_scale, y, M, N, K, 0u, stream);
}

int nvfp4_linear_f32(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                     float global_scale, float* y, int64_t M, int64_t N, int64_t K,
                     void* stream) {
  return run(x, w_packed, w_scale, global_scale, global_scale, y, M, N, K, NVFP4_FLAG_F32_OUT, stream);
}

int nvfp4_linear_swiglu(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                        float global_scale, void* y, int64_t M, int64_t N, int64_t K,
                        void* stream) {
  return run(x, w_packed, w_scale, global_scale, global_scale, y, M, N, K, NVFP4_FLAG_SWIGLU, stream);
}

int nvfp4_linear_swiglu_f32(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                            float global_scale, float* y, int64_t M, int64_t N, int64_t K,
                            void* stream) {
  return run(x, w_packed, w_scale, global_scale, global_scale, y, M, N, K,
             NVFP4_FLAG_SWIGLU | NVFP4_FLAG_F32_OUT, stream);
}

int nvfp4_linear_ex(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                    float global_scale, void* y, int64_t M, int64_t N, int64_t K,
                    unsigned int flags, void* stream) {
  return run(x, w_packed, w_scale, global_scale, global_scale, y, M, N, K, flags, stream);
}

int nvfp4_linear_host(const void* x_host, void* x_dev, const uint8_t* w_packed,
                      const uint8_t* w_scale, float global_scale, void* y_dev, void* y_host,
                      int64_t M, int64_t N, int64_t K, unsigned int flags, void* stream_ptr) {
  int st = validate(x_dev, w_packed, w_scale, y_dev, M, N, K, flags);
  if (st != NVFP4_OK) return st;
  if (M == 0) return NVFP4_OK;
  if (!x_host || !y_host) return NVFP4_ERR_INVALID;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const size_t x_bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * 2;
  const int64_t n_out = (flags & NVFP4_FLAG_SWIGLU) ? N / 2 : N;
  const size_t y_bytes = static_cast<size_t>(M) * static_cast<size_t>(n_out) *
                         ((flags & NVFP4_FLAG_F32_OUT) ? 4 : 2);
  // Page-locked host buffers mapped into the device's address space, all
  // four buffers and both sizes 16-byte aligned: the transfers are kernels
  // chained with the layer (zero-copy, see host_io.cuh); otherwise one
  // cudaMemcpyAsync each way.
  const void* xh = device_view(x_host);
  void* yh = device_view(y_host);
  const bool zero_copy = xh && yh &&
                         ((reinterpret_cast<uintptr_t>(xh) | reinterpret_cast<uintptr_t>(yh) |
                           reinterpret_cast<uintptr_t>(x_dev) |
                           reinterpret_cast<uintptr_t>(y_dev) | x_bytes | y_bytes) &
                          15u) == 0;
  DeviceInfo* d = nullptr;
  if (zero_copy) {
    st = device_setup(&d);
    if (st != NVFP4_OK) return st;
    st = launch_staging(nvfp4::hostio::stage_in_kernel, static_cast<const uint4*>(xh),
                        static_cast<uint4*>(x_dev), static_cast<int64_t>(x_bytes / 16),
                        d->num_sms, stream);
    if (st != NVFP4_OK) return st;
  } else if (cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, stream) !=
             cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  // The few-row kernels (M <= 32) also write the result straight into the
  // mapped host buffer from their epilogue; the tensor-core kernel's output
  // is moved by the output staging kernel.
  const bool mirror = zero_copy && kernel_for(M, N, K, flags) != NVFP4_KERNEL_TCGEMM;
  st = run(x_dev, w_packed, w_scale, global_scale, global_scale, y_dev, M, N, K, flags,
           stream_ptr, nullptr, mirror ? yh : nullptr);
  if (st != NVFP4_OK) return st;
  if (mirror) return NVFP4_OK;
  if (zero_copy)
    return launch_staging(nvfp4::hostio::stage_out_kernel, static_cast<const uint4*>(y_dev),
                          static_cast<uint4*>(yh), static_cast<int64_t>(y_bytes / 16),
                          d->num_sms, stream);
  if (cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

int nvfp4_linear_swiglu_gs(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                           float gate_global_scale, float up_global_scale, void* y, int64_t M,
                           int64_t N, int64_t K, unsigned int flags, void* stream) {
  return run(x, w_packed, w_scale, gate_global_scale, up_global_scale, y, M, N, K,
             flags | NVFP4_FLAG_SWIGLU, stream);
}

int nvfp4_linear_segmented(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                           const float* global_scales, const int64_t* segment_rows,
                           int num_segments, void* y, int64_t M, int64_t N, int64_t K,
                           unsigned int flags, void* stream) {
  if (!global_scales || !segment_rows || num_segments < 1 ||
      num_segments > nvfp4::kMaxSegments || (flags & NVFP4_FLAG_SWIGLU))
    return NVFP4_ERR_INVALID;
  SegSpec spec;
  spec.count = num_segments;
  int64_t end = 0;
  for (int i = 0; i < num_segments; ++i) {
    if (segment_rows[i] <= 0) return NVFP4_ERR_INVALID;
    end += segment_rows[i];
    spec.end[i] = end;
    spec.gs[i] = global_scales[i];
  }
  if (end != N) return NVFP4_ERR_INVALID;
  return run(x, w_packed, w_scale, global_scales[0], global_scales[0], y, M, N, K, flags, stream,
             &spec);
}

int nvfp4_quantize(const void* w, int64_t N, int64_t K, uint8_t* w_packed, uint8_t* w_scale,
                   float* global_scale, void* stream_ptr) {
  namespace Q = nvfp4::quant;
  if (!w || !w_packed || !w_scale || !global_scale || N <= 0 || K <= 0)
    return NVFP4_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(w_packed) & 7u) ||
      (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return NVFP4_ERR_MISALIGNED;
  if (K % 16 != 0 || N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return NVFP4_ERR_SHAPE;
  DeviceInfo* d = nullptr;
  const int st = device_setup(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int64_t n_blocks = N * (K / 16);
  const unsigned g_amax = resident_grid(Q::amax_kernel, d->num_sms, 2 * n_blocks);
  const unsigned g_quant = resident_grid(Q::quantize_kernel, d->num_sms, n_blocks);
  unsigned int* amax_bits = reinterpret_cast<unsigned int*>(global_scale);
  if (cudaMemsetAsync(global_scale, 0, sizeof(float), stream) != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  Q::amax_kernel<<<g_amax, Q::kThreads, 0, stream>>>(static_cast<const uint4*>(w), 2 * n_blocks,
                                                     amax_bits);
  Q::quantize_kernel<<<g_quant, Q::kThreads, 0, stream>>>(
      static_cast<const uint4*>(w), n_blocks, amax_bits, reinterpret_cast<uint2*>(w_packed),
      w_scale);
  Q::finalize_kernel<<<1, 32, 0, stream>>>(global_scale);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_LAUNCH;
  return NVFP4_OK;
}

int nvfp4_quantize_fp8(const uint8_t* w_fp8, const float* scale_inv, int64_t block, int64_t N,
                       int64_t K, uint8_t* w_packed, uint8_t* w_scale, float* global_scale,
                       void* stream_ptr) {
  namespace Q = nvfp4::quant;
  if (!w_fp8 || !scale_inv || !w_packed || !w_scale || !global_scale || N <= 0 || K <= 0 ||
      block <= 0)
    return NVFP4_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(w_fp8) & 15u) || (reinterpret_cast<uintptr_t>(w_packed) & 7u) ||
      (reinterpret_cast<uintptr_t>(scale_inv) & 3u) ||
      (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return NVFP4_ERR_MISALIGNED;
  if (K % 16 != 0 || block % 16 != 0 || N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
    return NVFP4_ERR_SHAPE;
  DeviceInfo* d = nullptr;
  const int st = device_setup(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  // units of four 16-input blocks when they never cross a row or a scale
  // block (and, for the quantiser's word-wide scale store, w_scale is 4-byte
  // aligned); single blocks otherwise
  const bool quad_amax = K % 64 == 0 && block % 64 == 0;
  const bool quad_quant = quad_amax && (reinterpret_cast<uintptr_t>(w_scale) & 3u) == 0;
  auto layout = [&](int U) {
    Q::Fp8Layout L;
    L.units_per_row = K / (16 * U);
    L.n_units = N * L.units_per_row;
    L.kb = (K + block - 1) / block;
    L.B = block;
    L.b_shift = -1;
    for (int sh = 4; sh < 31; ++sh)
      if ((int64_t(1) << sh) == block) L.b_shift = sh;
    return L;
  };
  unsigned int* amax_bits = reinterpret_cast<unsigned int*>(global_scale);
  if (cudaMemsetAsync(global_scale, 0, sizeof(float), stream) != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  const uint4* w = reinterpret_cast<const uint4*>(w_fp8);
  uint2* codes = reinterpret_cast<uint2*>(w_packed);
  const Q::Fp8Layout La = layout(quad_amax ? 4 : 1), Lq = layout(quad_quant ? 4 : 1);
  const int sms = d->num_sms;
  if (quad_amax)
    Q::amax_fp8_kernel<4><<<resident_grid(Q::amax_fp8_kernel<4>, sms, La.n_units), Q::kThreads, 0,
                            stream>>>(w, scale_inv, La, amax_bits);
  else
    Q::amax_fp8_kernel<1><<<resident_grid(Q::amax_fp8_kernel<1>, sms, La.n_units), Q::kThreads, 0,
                            stream>>>(w, scale_inv, La, amax_bits);
  if (quad_quant)
    Q::quantize_fp8_kernel<4><<<resident_grid(Q::quantize_fp8_kernel<4>, sms, Lq.n_units),
                                Q::kThreads, 0, stream>>>(w, scale_inv, Lq, amax_bits, codes,
                                                          w_scale);
  else
    Q::quantize_fp8_kernel<1><<<resident_grid(Q::quantize_fp8_kernel<1>, sms, Lq.n_units),
                                Q::kThreads, 0, stream>>>(w, scale_inv, Lq, amax_bits, codes,
                                                          w_scale);
  Q::finalize_kernel<<<1, 32, 0, stream>>>(global_scale);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_LAUNCH;
  return NVFP4_OK;
}

int nvfp4_linear_kernel_for(int64_t M, int64_t N, int64_t K, unsigned int flags) {
  static const uint8_t dummy[16] __attribute__((aligned(16))) = {0};
  if (validate(dummy, dummy, dummy, dummy, M, N, K, flags) != NVFP4_OK || M == 0)
    return NVFP4_KERNEL_NONE;
  return kernel_for(M, N, K, flags);
}

}  // extern "C"

// ------------------------------------------------------------------------
// nvfp4_linear_host_noalloc: nvfp4_linear_host with its two device staging
// buffers (the activations' copy on the device and the result before it
// goes back to the host) carved from one fixed array of this library, so
// that the caller allocates no device memory at all.  The array is a
// file-scope __device__ object: every device that loads the library holds
// it for the life of the process.  Its name, in host code, is only a host
// stand-in for the symbol, so its device address is looked up once per
// device (cudaGetSymbolAddress, that device current) and cached.
namespace {

__device__ __align__(256) unsigned char g_host_scratch[NVFP4_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_host_scratch on the current device (set up on the
// first call there); nullptr and a status on failure.
void* host_scratch(int* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = NVFP4_ERR_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_host_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      *status = NVFP4_ERR_DEVICE;
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  *status = NVFP4_OK;
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

int nvfp4_linear_host_noalloc(const void* x_host, const uint8_t* w_packed,
                              const uint8_t* w_scale, float global_scale, void* y_host,
                              int64_t M, int64_t N, int64_t K, unsigned int flags,
                              void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID;
  if (M == 0) return NVFP4_OK;
  if (!x_host || !y_host) return NVFP4_ERR_INVALID;
  // sizes first, with no overflow: M, N, K are bounded before they multiply
  if (M > (int64_t(1) << 24) || N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
    return NVFP4_ERR_TOO_LARGE;
  const int64_t n_out = (flags & NVFP4_FLAG_SWIGLU) ? N / 2 : N;
  const int64_t x_bytes = M * K * 2;
  const int64_t x_span = (x_bytes + 255) / 256 * 256;       // y starts 256-aligned
  const int64_t y_bytes = M * n_out * ((flags & NVFP4_FLAG_F32_OUT) ? 4 : 2);
  if (x_bytes > NVFP4_NOALLOC_SCRATCH_BYTES ||
      y_bytes > NVFP4_NOALLOC_SCRATCH_BYTES - x_span)
    return NVFP4_ERR_TOO_LARGE;
  int st = NVFP4_OK;
  unsigned char* scratch = static_cast<unsigned char*>(host_scratch(&st));
  if (!scratch) return st;
  return nvfp4_linear_host(x_host, scratch, w_packed, w_scale, global_scale, scratch + x_span,
                           y_host, M, N, K, flags, stream);
}

int nvfp4_device_status(unsigned int* bits, int clear) {
  if (!bits) return NVFP4_ERR_INVALID;
  DeviceInfo* d = nullptr;
  const int st = device_setup(&d);
  if (st != NVFP4_OK) return st;
  // Every stream of the device first (the copy below orders only against
  // the legacy default stream, not against non-blocking streams), then the
  // atomic read-and-clear, then its result.
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  read_device_error_kernel<<<1, 1, 0, 0>>>(clear ? 1 : 0);
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemcpyFromSymbol(bits, g_device_error_read, sizeof(unsigned int)) != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

}  // extern "C"
