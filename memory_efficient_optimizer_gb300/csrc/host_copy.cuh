// Upload of a step's descriptor table from pinned host memory by a kernel
// (the device reads the host buffer through its mapping) instead of a
// cudaMemcpyAsync.
//
// A host-to-device cudaMemcpyAsync runs on a copy engine, behind whatever
// copies were queued there before it, from any stream: a training loop that
// uploads the next step's gradients (gigabytes) on a side stream would hold
// the step's few-kilobyte descriptor copy, and with it the whole step, until
// that upload is done.  A kernel that reads the table straight from host
// memory takes no copy engine, so the step runs beside the upload.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace meo {
namespace {

// dst[i] = src[i] for i < n16 (16-byte words); src is host memory, read with
// cache-volatile loads (fetched again on every use: a ring slot is refilled
// by the host between calls).
__global__ void __launch_bounds__(256) k_copy_from_host(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                        int64_t n16) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = __ldcv(src + i);
}

// Enqueues the copy of `bytes` (a multiple of 16) from the pinned, mapped
// host buffer `host` (16-byte aligned) to `dst` (16-byte aligned) on s.
inline cudaError_t copy_from_host(void* dst, const void* host, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  void* src = nullptr;
  cudaError_t e = cudaHostGetDevicePointer(&src, const_cast<void*>(host), 0);
  if (e != cudaSuccess) return e;
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  const int64_t blocks = (n16 + 255) / 256;
  k_copy_from_host<<<static_cast<int>(blocks < 64 ? blocks : 64), 256, 0, s>>>(
      static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
  return cudaGetLastError();
}

}  // namespace
}  // namespace meo
