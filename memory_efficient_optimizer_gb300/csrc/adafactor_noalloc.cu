// adafactor_step_noalloc(): the Adafactor step with a fixed scratch area
// compiled into the library, for callers that cannot allocate device memory.
//
// adafactor_step() needs a caller-provided workspace.  Some callers cannot
// make one: code that runs while a memory pool owns all of the device memory
// and forbids cudaMalloc, code whose allocations would synchronise the device
// at a point where that is not allowed, or hosts that link this library
// without any allocator of their own.  For them, the scratch lives in a
// file-scope __device__ array of kNoAllocScratchBytes that every GPU that
// loads the library holds until the process exits.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "adafactor.h"
#include "adafactor_internal.h"

namespace {

// 64 MiB: enough for the scratch of about 2.1e9 parameters in 2D tensors of
// Llama-like shapes (the workspace is ~1/32 byte per parameter plus a small
// per-tensor part).
constexpr size_t kNoAllocScratchBytes = ADAF_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// g_noalloc_scratch names a host-side stand-in, never the device memory, so
// the address is looked up once per device with that device current.
adaf_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "adafactor_step_noalloc: no usable current device (%s)", cudaGetErrorString(e));
    return meo::set_last_error(ADAF_ERR_CUDA, msg);
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[160];
      std::snprintf(msg, sizeof(msg), "adafactor_step_noalloc: cudaGetSymbolAddress failed (%s)",
                    cudaGetErrorString(e));
      return meo::set_last_error(ADAF_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ADAF_OK;
}

}  // namespace

namespace meo {
void noalloc_forget_addresses() {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  for (void*& a : g_scratch_addr) a = nullptr;
}
}  // namespace meo

extern "C" {

adaf_status adafactor_step_noalloc(const adaf_tensor* tensors, const adaf_state* states, int32_t n,
                                   int64_t step, const adaf_hparams* hp, void* stream) {
  // Host-only checks first: a rejected call touches neither CUDA nor memory.
  adaf_status st = adafactor_validate(hp);
  if (st != ADAF_OK) return st;
  size_t need = 0;
  st = adafactor_workspace_size(tensors, n, &need);
  if (st != ADAF_OK) return st;
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "adafactor_step_noalloc: this tensor list needs %zu bytes of scratch, more than the fixed "
                  "%zu-byte area; call adafactor_step() with a workspace instead",
                  need, kNoAllocScratchBytes);
    return meo::set_last_error(ADAF_ERR_WORKSPACE_TOO_SMALL, msg);
  }
  // The header upload below copies from a host buffer that lives only for
  // this call; recorded into a graph, the copy would read freed memory on
  // every replay.  So a capturing stream is turned away before any work.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
  if (e != cudaSuccess) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "adafactor_step_noalloc: cudaStreamIsCapturing failed (%s)",
                  cudaGetErrorString(e));
    return meo::set_last_error(ADAF_ERR_CUDA, msg);
  }
  if (cap != cudaStreamCaptureStatusNone)
    return meo::set_last_error(ADAF_ERR_UNSUPPORTED,
                               "adafactor_step_noalloc: the stream is capturing; this entry point uploads its "
                               "descriptor table from a host buffer that lives only for the call");
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != ADAF_OK) return st;
  // The header upload (which also resets the status word at offset 0) comes
  // from a pageable host buffer, so no pinned staging is allocated either.
  return meo::step_impl(tensors, states, n, step, hp, scratch, kNoAllocScratchBytes, stream,
                        meo::kStagePageable);
}

adaf_status adafactor_noalloc_device_status(void* stream, int32_t* status) {
  if (status == nullptr) return meo::set_last_error(ADAF_ERR_INVALID_ARGUMENT, "status is NULL");
  void* scratch = nullptr;
  adaf_status st = scratch_address(&scratch);
  if (st != ADAF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "adafactor_noalloc_device_status: reading the status word failed (%s)",
                  cudaGetErrorString(e));
    return meo::set_last_error(ADAF_ERR_CUDA, msg);
  }
  *status = v;
  return ADAF_OK;
}

}  // extern "C"
