// nvfp4_linear.cu -- the C ABI of include/nvfp4_linear.h: host-side
// validation, kernel choice by M, TMA tensor-map encoding and launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/nvfp4_linear.h"
#include "smallm.cuh"
#include "tcgemm.cuh"

namespace {

using nvfp4::smallm::Layout;

// Bits set by kernels when a pipeline wait gives up (see ptx.cuh).
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
constexpr int64_t kSmallMMax = 32;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  unsigned int* err = nullptr;         // device address of g_device_error
  int smallm_ctas_per_sm[5] = {0, 0, 0, 0, 0};   // by MT
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <int MT>
cudaError_t prepare_smallm(DeviceInfo& d) {
  auto kern = nvfp4::smallm::smallm_kernel<MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Layout<MT>::kSmemBytes);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, nvfp4::smallm::kThreads,
                                                    Layout<MT>::kSmemBytes);
  d.smallm_ctas_per_sm[MT] = n > 0 ? n : 1;
  return e;
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
          prepare_smallm<1>(d) != cudaSuccess || prepare_smallm<2>(d) != cudaSuccess ||
          prepare_smallm<3>(d) != cudaSuccess || prepare_smallm<4>(d) != cudaSuccess ||
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

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0,
               uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
               CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int validate(const void* x, const void* wp, const void* ws, const void* y, int64_t M,
             int64_t N, int64_t K, unsigned int flags) {
  if (M < 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID;
  // With M == 0 nothing is read from x or written to y: an empty tensor's
  // null data pointer is fine there.
  if (!wp || !ws || (M > 0 && (!x || !y))) return NVFP4_ERR_INVALID;
  if (flags & ~(NVFP4_FLAG_SWIGLU | NVFP4_FLAG_F32_OUT | NVFP4_FLAG_FORCE_SMALLM |
                NVFP4_FLAG_FORCE_TCGEMM))
    return NVFP4_ERR_INVALID;
  if ((flags & NVFP4_FLAG_FORCE_SMALLM) && (flags & NVFP4_FLAG_FORCE_TCGEMM))
    return NVFP4_ERR_INVALID;
  if ((flags & NVFP4_FLAG_FORCE_SMALLM) && M > kSmallMMax) return NVFP4_ERR_INVALID;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(wp) |
                        reinterpret_cast<uintptr_t>(ws) | reinterpret_cast<uintptr_t>(y);
  if (mis & 15u) return NVFP4_ERR_MISALIGNED;
  if (K % 256 != 0 || N % 128 != 0) return NVFP4_ERR_SHAPE;
  // tensor-map and grid limits
  if (K > (int64_t(1) << 31) || N > (int64_t(1) << 31) || M > (int64_t(1) << 24))
    return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

int kernel_for(int64_t M, unsigned int flags) {
  if (flags & NVFP4_FLAG_FORCE_SMALLM) return NVFP4_KERNEL_SMALLM;
  if (flags & NVFP4_FLAG_FORCE_TCGEMM) return NVFP4_KERNEL_TCGEMM;
  return M <= kSmallMMax ? NVFP4_KERNEL_SMALLM : NVFP4_KERNEL_TCGEMM;
}

template <int MT>
int launch_smallm(const DeviceInfo& d, const void* x, const uint8_t* wp, const uint8_t* ws,
                  float gs, void* y, int64_t M, int64_t N, int64_t K, unsigned int flags,
                  cudaStream_t stream) {
  using L = Layout<MT>;
  const bool swiglu = flags & NVFP4_FLAG_SWIGLU;
  CUtensorMap tw, ts, tx;
  if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wp, K / 2, N, K / 2, 128,
                 nvfp4::smallm::kHalfRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, ws, K / 16, N, K / 16, 16,
                 nvfp4::smallm::kHalfRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, K * 2, 64, MT * 8,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4_ERR_LAUNCH;

  nvfp4::smallm::Params p;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.global_scale = gs;
  p.stages_total = static_cast<int>(K / nvfp4::smallm::kStageK);
  p.out_f32 = (flags & NVFP4_FLAG_F32_OUT) ? 1 : 0;
  p.swiglu = swiglu ? 1 : 0;
  p.err = d.err;

  const int64_t row_blocks =
      swiglu ? (N / 2) / nvfp4::smallm::kHalfRows : N / nvfp4::smallm::kRows;
  // Split k across a cluster when the row blocks alone cannot fill the GPU.
  const int64_t slots = static_cast<int64_t>(d.num_sms) * d.smallm_ctas_per_sm[MT];
  int64_t split = row_blocks >= slots ? 1 : slots / row_blocks;
  if (split > 8) split = 8;
  if (split > p.stages_total) split = p.stages_total;
  if (split < 1) split = 1;
  p.split = static_cast<int>(split);

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(static_cast<unsigned>(row_blocks), static_cast<unsigned>(split), 1);
  cfg.blockDim = dim3(nvfp4::smallm::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(split);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, nvfp4::smallm::smallm_kernel<MT>, tw, ts, tx, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  return NVFP4_OK;
}

int launch_tcgemm(const DeviceInfo& d, const void* x, const uint8_t* wp, const uint8_t* ws,
                  float gs, void* y, int64_t M, int64_t N, int64_t K, unsigned int flags,
                  cudaStream_t stream) {
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
  p.global_scale = gs;
  p.out_f32 = (flags & NVFP4_FLAG_F32_OUT) ? 1 : 0;
  p.swiglu = swiglu ? 1 : 0;
  p.err = d.err;
  const unsigned gx = static_cast<unsigned>(swiglu ? (N / 2) / 64 : N / T::kTileW);
  const unsigned gy = static_cast<unsigned>((M + T::kTileX - 1) / T::kTileX);
  T::tcgemm_kernel<<<dim3(gx, gy, 1), T::kThreads, T::kSmemBytes, stream>>>(tx, tw, ts, p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_LAUNCH;
  (void)d;
}

int run(const void* x, const uint8_t* wp, const uint8_t* ws, float gs, void* y, int64_t M,
        int64_t N, int64_t K, unsigned int flags, void* stream_ptr) {
  int st = validate(x, wp, ws, y, M, N, K, flags);
  if (st != NVFP4_OK) return st;
  if (M == 0) return NVFP4_OK;
  DeviceInfo* d = nullptr;
  st = device_setup(&d);
  if (st != NVFP4_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (kernel_for(M, flags) == NVFP4_KERNEL_SMALLM) {
    switch ((M + 7) / 8) {
      case 1: return launch_smallm<1>(*d, x, wp, ws, gs, y, M, N, K, flags, stream);
      case 2: return launch_smallm<2>(*d, x, wp, ws, gs, y, M, N, K, flags, stream);
      case 3: return launch_smallm<3>(*d, x, wp, ws, gs, y, M, N, K, flags, stream);
      default: return launch_smallm<4>(*d, x, wp, ws, gs, y, M, N, K, flags, stream);
    }
  }
  return launch_tcgemm(*d, x, wp, ws, gs, y, M, N, K, flags, stream);
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
    default: return "unknown status";
  }
}

int nvfp4_linear(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                 float global_scale, void* y, int64_t M, int64_t N, int64_t K, void* stream) {
  return run(x, w_packed, w_scale, global_scale, y, M, N, K, 0u, stream);
}

int nvfp4_linear_f32(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                     float global_scale, float* y, int64_t M, int64_t N, int64_t K,
                     void* stream) {
  return run(x, w_packed, w_scale, global_scale, y, M, N, K, NVFP4_FLAG_F32_OUT, stream);
}

int nvfp4_linear_swiglu(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                        float global_scale, void* y, int64_t M, int64_t N, int64_t K,
                        void* stream) {
  return run(x, w_packed, w_scale, global_scale, y, M, N, K, NVFP4_FLAG_SWIGLU, stream);
}

int nvfp4_linear_swiglu_f32(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                            float global_scale, float* y, int64_t M, int64_t N, int64_t K,
                            void* stream) {
  return run(x, w_packed, w_scale, global_scale, y, M, N, K,
             NVFP4_FLAG_SWIGLU | NVFP4_FLAG_F32_OUT, stream);
}

int nvfp4_linear_ex(const void* x, const uint8_t* w_packed, const uint8_t* w_scale,
                    float global_scale, void* y, int64_t M, int64_t N, int64_t K,
                    unsigned int flags, void* stream) {
  return run(x, w_packed, w_scale, global_scale, y, M, N, K, flags, stream);
}

int nvfp4_linear_kernel_for(int64_t M, int64_t N, int64_t K, unsigned int flags) {
  static const uint8_t dummy[16] __attribute__((aligned(16))) = {0};
  if (validate(dummy, dummy, dummy, dummy, M, N, K, flags) != NVFP4_OK || M == 0)
    return NVFP4_KERNEL_NONE;
  return kernel_for(M, flags);
}

int nvfp4_device_status(unsigned int* bits, int clear) {
  if (!bits) return NVFP4_ERR_INVALID;
  DeviceInfo* d = nullptr;
  const int st = device_setup(&d);
  if (st != NVFP4_OK) return st;
  if (cudaMemcpyFromSymbol(bits, g_device_error, sizeof(unsigned int)) != cudaSuccess) {
    cudaGetLastError();
    return NVFP4_ERR_LAUNCH;
  }
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) {
      cudaGetLastError();
      return NVFP4_ERR_LAUNCH;
    }
  }
  return NVFP4_OK;
}

}  // extern "C"
