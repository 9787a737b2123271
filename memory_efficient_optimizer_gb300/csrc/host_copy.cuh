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
#include <cstring>
#include <utility>
#include <vector>

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

// Device copies of a step's descriptor table, one per distinct content.  A
// step whose table bytes equal a kept copy's reads that copy and uploads
// nothing: the upload kernel's host reads share the host link with the
// caller's own host-to-device copies, and a 16 GB gradient upload on a side
// stream (the next step's) was measured to hold a step back for most of its
// 76 ms on some boxes.
struct TableCache {
  struct Entry {
    std::vector<unsigned char> bytes;  // the table as uploaded
    unsigned char* dev = nullptr;      // its device copy
    cudaEvent_t ready = nullptr;       // recorded after the upload
    cudaEvent_t used = nullptr;        // recorded after the last step that read it
    uint64_t stamp = 0;                // last use, for eviction
  };
  static constexpr size_t kMax = 8;  // copies kept per device
  std::vector<Entry> entries;
  uint64_t clock = 0;

  static void release(Entry& e) {
    if (e.used) cudaEventSynchronize(e.used);  // no step still reads it
    if (e.dev) cudaFree(e.dev);
    if (e.ready) cudaEventDestroy(e.ready);
    if (e.used) cudaEventDestroy(e.used);
    e = Entry();
  }
  void clear() {
    for (Entry& e : entries) release(e);
    entries.clear();
  }
  // The device copy of bytes[0, n): a kept one (s waits for its upload), or
  // a new one that upload(dev) fills on s (the least recently used copy is
  // dropped when kMax are kept).  *used is the event to record on s after the
  // step's last launch.
  template <class Upload>
  cudaError_t lookup(const unsigned char* bytes, size_t n, cudaStream_t s, Upload&& upload, unsigned char** dev,
                     cudaEvent_t* used) {
    Entry* hit = nullptr;
    for (Entry& e : entries) {
      if (e.bytes.size() == n && std::memcmp(e.bytes.data(), bytes, n) == 0) {
        hit = &e;
        break;
      }
    }
    cudaError_t err = cudaSuccess;
    if (hit != nullptr) {
      err = cudaStreamWaitEvent(s, hit->ready, 0);  // the copy may have been made on another stream
      if (err != cudaSuccess) return err;
    } else {
      if (entries.size() >= kMax) {
        size_t lru = 0;
        for (size_t k = 1; k < entries.size(); ++k)
          if (entries[k].stamp < entries[lru].stamp) lru = k;
        release(entries[lru]);
        entries.erase(entries.begin() + static_cast<std::ptrdiff_t>(lru));
      }
      Entry ne;
      err = cudaMalloc(reinterpret_cast<void**>(&ne.dev), (n + 255) & ~size_t{255});  // whole 16-byte words
      if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ne.ready, cudaEventDisableTiming);
      if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ne.used, cudaEventDisableTiming);
      if (err == cudaSuccess) err = upload(ne.dev);
      if (err == cudaSuccess) err = cudaEventRecord(ne.ready, s);
      if (err != cudaSuccess) {
        release(ne);
        return err;
      }
      ne.bytes.assign(bytes, bytes + n);
      entries.push_back(std::move(ne));
      hit = &entries.back();
    }
    hit->stamp = ++clock;
    *dev = hit->dev;
    *used = hit->used;
    return cudaSuccess;
  }
};

// Records `ev` on `s` when a step's launch sequence is left, on every path.
struct RecordOnExit {
  cudaEvent_t ev = nullptr;
  cudaStream_t s = nullptr;
  ~RecordOnExit() {
    if (ev) cudaEventRecord(ev, s);
  }
};

__global__ void k_zero_word(int32_t* p) { *p = 0; }

// Enqueues *p = 0 on s (a one-thread kernel: no copy engine either).
inline cudaError_t zero_word(int32_t* p, cudaStream_t s) {
  k_zero_word<<<1, 1, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace meo
