// host_io.cuh -- the host-buffer entry point's transfers as kernels.
//
// On GB300 page-locked host memory sits in the GPU's address space over the
// coherent NVLink-C2C link, so a kernel can read the activations from, and
// write the result to, the caller's host buffers directly (zero-copy).  As
// kernels (or, for a few-row kernel's result, as part of its epilogue), the
// transfers join the chain of programmatic dependent launches the layer's
// kernels already form: consecutive calls on a stream then overlap the next
// call's weight prefetch with the current call, which a copy-engine transfer
// between two kernels prevents.
//
// Ordering (every launch of the chain carries programmatic stream
// serialisation; griddepcontrol.wait waits for the whole preceding grid,
// which itself completed only after its own wait):
//   stage_in   reads the host activations before its wait (nothing on the
//              device writes them), writes x_dev after it (the preceding
//              call may still read x_dev);
//   the layer  reads x_dev after its wait; the few-row kernels (M <= 32)
//              write the result to y_dev and, from the same epilogue, to
//              the host buffer;
//   stage_out  (M > 32 only) reads y_dev and writes the host result after
//              its wait.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace nvfp4 {
namespace hostio {

constexpr int kThreads = 256;

// dst[i] = src[i] for n 16-byte words; src is host memory mapped into the
// device's address space (plain loads: the read-only cache path is not
// used for it).
__global__ void __launch_bounds__(kThreads) stage_in_kernel(const uint4* src, uint4* dst,
                                                            int64_t n) {
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (i < n) v = src[i];
  griddep_wait();
  for (; i < n; i += stride) {
    dst[i] = v;
    if (i + stride < n) v = src[i + stride];
  }
}

// dst[i] = src[i] for n 16-byte words; dst is host memory mapped into the
// device's address space.
__global__ void __launch_bounds__(kThreads) stage_out_kernel(const uint4* src, uint4* dst,
                                                             int64_t n) {
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < n;
       i += stride)
    dst[i] = src[i];
}

}  // namespace hostio
}  // namespace nvfp4
