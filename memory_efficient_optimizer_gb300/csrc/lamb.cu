// Multi-tensor LAMB step for sm_103a: the C ABI of include/lamb.h.
//
// LAMB (the Colossal-AI distributed-optimizer article, overview table and
// "其余优化器的关键参数速查" / DistributedLAMB; the rule is the LAMB algorithm of
// arXiv:1904.00962) scales each tensor's Adam-style direction
// r = mh / (sqrt(vh) + eps) + wd p by the trust ratio ||p|| / ||r||.  The
// ratio needs the norm of r over the whole tensor before any element moves,
// so a step is two streaming passes around a per-tensor reduction:
//
//   k_lamb_moments  g, m, v, p -> m, v; per work unit sum r^2 and sum p^2
//                   (read 14 or 16 B, write 8 B per value)
//   k_lamb_trust    one CTA per tensor: sums its unit partials in a fixed
//                   order, trust = ||p|| / ||r|| (1 where a norm is 0)
//   k_lamb_update   m, v, p -> p - lr trust r  (read 12 B, write 4 B)
//
// Every tensor is a flat range cut into work units of kUnit values, numbered
// with the bf16-gradient tensors first, so that each gradient dtype has its
// own moments launch (and its own register budget).  A persistent grid walks
// a launch's units round-robin, and each CTA finds its tensor by advancing a
// cursor over the unit prefix (units rise with the loop, so the cursor only
// moves forward).  r is computed by the same correctly
// rounded intrinsics in both passes, so the update applies exactly the r
// whose norm set the trust ratio.  All sums are deterministic (fixed-order
// trees, no atomics).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "adafactor_internal.h"
#include "host_copy.cuh"
#include "lamb.h"

namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 8;                               // 4-value vectors per thread per unit
constexpr int64_t kUnit = int64_t{kThreads} * 4 * kVecPerThread;  // 8192 values
// 4-value vectors per stream in flight per thread, moments pass (4 streams):
// 4 with bf16 gradients (2 registers each), 3 with fp32 ones
template <typename GT> struct BatchM { static constexpr int value = 3; };
template <> struct BatchM<__nv_bfloat16> { static constexpr int value = 4; };
constexpr int kBatchU = 4;  // the same, update pass (3 streams)
constexpr int64_t kMaxNumel = int64_t{1} << 40;

// Device descriptor of one tensor (64 bytes).
struct LDev {
  float* p;
  const void* g;
  float* m;
  float* v;
  int64_t numel;
  int64_t unit0;   // first work unit
  int32_t gdt;     // ADAF_FLOAT32 / ADAF_BFLOAT16
  int32_t vec;     // 4-value loads allowed (aligned pointers)
  int64_t nunits;  // work units
};
static_assert(sizeof(LDev) == 64, "descriptor layout");

struct LArgs {
  const LDev* dev;
  const int64_t* pf;       // [n + 1]: first unit of each tensor in unit order, then the total
  const int32_t* ord;      // [n]: the tensor at each position of that order
  double* part;            // [units][2]: sum r^2, sum p^2
  double* trust;           // [n]
  double* coef;            // [n]: lr * trust
  int64_t units;
  int32_t n;
  float b1, omb1, b2, omb2, inv_bc1, inv_bc2, eps, wd;
  double lr;
};

// ---- element arithmetic (shared by both passes) ---------------------------
struct Moments {
  float m, v;
};
__device__ __forceinline__ Moments lamb_moments(float g, float m, float v, const LArgs& a) {
  Moments o;
  o.m = __fmaf_rn(a.b1, m, __fmul_rn(a.omb1, g));
  o.v = __fmaf_rn(a.b2, v, __fmul_rn(a.omb2, __fmul_rn(g, g)));
  return o;
}
// r = mh / (sqrt(vh) + eps) + wd p, every operation correctly rounded.
__device__ __forceinline__ float lamb_dir(float m, float v, float p, const LArgs& a) {
  const float mh = __fmul_rn(m, a.inv_bc1);
  const float vh = __fmul_rn(v, a.inv_bc2);
  return __fmaf_rn(a.wd, p, __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), a.eps)));
}

template <typename GT> struct G4;
template <> struct G4<float> { float4 v; };
template <> struct G4<__nv_bfloat16> { uint2 v; };
__device__ __forceinline__ void load_g4(G4<float>& r, const void* g, int64_t e) {
  r.v = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(g) + e));
}
__device__ __forceinline__ void load_g4(G4<__nv_bfloat16>& r, const void* g, int64_t e) {
  r.v = __ldcs(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(g) + e));
}
__device__ __forceinline__ void widen_g4(const G4<float>& r, float (&x)[4]) {
  x[0] = r.v.x; x[1] = r.v.y; x[2] = r.v.z; x[3] = r.v.w;
}
// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits.
__device__ __forceinline__ void widen_g4(const G4<__nv_bfloat16>& r, float (&x)[4]) {
  x[0] = __uint_as_float(r.v.x << 16); x[1] = __uint_as_float(r.v.x & 0xffff0000u);
  x[2] = __uint_as_float(r.v.y << 16); x[3] = __uint_as_float(r.v.y & 0xffff0000u);
}
__device__ __forceinline__ float load_g1(const void* g, int gdt, int64_t e) {
  if (gdt == ADAF_BFLOAT16)
    return __uint_as_float(static_cast<uint32_t>(__ldcs(static_cast<const unsigned short*>(g) + e)) << 16);
  return __ldcs(static_cast<const float*>(g) + e);
}
__device__ __forceinline__ float4 ld4(const float* p, int64_t e) { return __ldcs(reinterpret_cast<const float4*>(p + e)); }
__device__ __forceinline__ void st4(float* p, int64_t e, float4 x) { __stcs(reinterpret_cast<float4*>(p + e), x); }
__device__ __forceinline__ float get(const float4& x, int q) { return q == 0 ? x.x : q == 1 ? x.y : q == 2 ? x.z : x.w; }

// Deterministic CTA sum of two values (fixed xor trees, warp order).
__device__ __forceinline__ void block_sum2(double& x, double& y, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // red of the previous use is read
  if (lane == 0) {
    red[warp] = x;
    red[32 + warp] = y;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double sx = 0.0, sy = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) {
      sx += red[w];
      sy += red[32 + w];
    }
    x = sx;
    y = sy;
  }
}

// ---- pass 1: moments and the unit's partial norms -------------------------
template <typename GT>
__device__ __forceinline__ void moments_vec(const LDev& d, const LArgs& a, int64_t e0, int64_t nv, float& rs,
                                            float& ps) {
  for (int64_t v0 = threadIdx.x; v0 < nv; v0 += BatchM<GT>::value * kThreads) {
    G4<GT> g[BatchM<GT>::value];
    float4 m[BatchM<GT>::value], v[BatchM<GT>::value], p[BatchM<GT>::value];
#pragma unroll
    for (int k = 0; k < BatchM<GT>::value; ++k) {
      const int64_t e = e0 + 4 * (v0 + k * kThreads);
      if (v0 + k * kThreads < nv) {
        load_g4(g[k], d.g, e);
        m[k] = ld4(d.m, e);
        v[k] = ld4(d.v, e);
        p[k] = ld4(d.p, e);
      }
    }
#pragma unroll
    for (int k = 0; k < BatchM<GT>::value; ++k) {
      if (v0 + k * kThreads < nv) {
        const int64_t e = e0 + 4 * (v0 + k * kThreads);
        float x[4], mo[4], vo[4];
        widen_g4(g[k], x);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const Moments n = lamb_moments(x[q], get(m[k], q), get(v[k], q), a);
          mo[q] = n.m;
          vo[q] = n.v;
          const float pq = get(p[k], q);
          const float r = lamb_dir(n.m, n.v, pq, a);
          rs = fmaf(r, r, rs);
          ps = fmaf(pq, pq, ps);
        }
        st4(d.m, e, make_float4(mo[0], mo[1], mo[2], mo[3]));
        st4(d.v, e, make_float4(vo[0], vo[1], vo[2], vo[3]));
      }
    }
  }
}

__device__ __forceinline__ void moments_scalar(const LDev& d, const LArgs& a, int64_t e0, int64_t e1, float& rs,
                                               float& ps) {
  for (int64_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
    const float x = load_g1(d.g, d.gdt, e);
    const float pq = __ldcs(d.p + e);
    const Moments n = lamb_moments(x, __ldcs(d.m + e), __ldcs(d.v + e), a);
    __stcs(d.m + e, n.m);
    __stcs(d.v + e, n.v);
    const float r = lamb_dir(n.m, n.v, pq, a);
    rs = fmaf(r, r, rs);
    ps = fmaf(pq, pq, ps);
  }
}

// Position (in unit order) of the tensor that holds unit u.
__device__ __forceinline__ int unit_owner(const LArgs& a, int64_t u) {
  int lo = 0, hi = a.n;  // largest lo with pf[lo] <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.pf[mid] <= u) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Units [u_begin, u_end): the tensors of one gradient dtype.
template <typename GT>
__global__ void __launch_bounds__(kThreads, 2) k_lamb_moments(const __grid_constant__ LArgs a, int64_t u_begin,
                                                              int64_t u_end) {
  __shared__ double red[64];
  int k = unit_owner(a, u_begin + blockIdx.x);
  for (int64_t u = u_begin + blockIdx.x; u < u_end; u += gridDim.x) {
    while (a.pf[k + 1] <= u) ++k;
    const LDev d = a.dev[a.ord[k]];
    const int64_t e0 = (u - d.unit0) * kUnit;
    const int64_t e1 = min(d.numel, e0 + kUnit);
    float rs = 0.f, ps = 0.f;
    int64_t es = e0;  // first value left to the scalar loop
    if (d.vec) {
      const int64_t nv = (e1 - e0) >> 2;
      moments_vec<GT>(d, a, e0, nv, rs, ps);
      es = e0 + 4 * nv;
    }
    moments_scalar(d, a, es, e1, rs, ps);
    double x = rs, y = ps;
    block_sum2(x, y, red);
    if (threadIdx.x == 0) {
      a.part[2 * u] = x;
      a.part[2 * u + 1] = y;
    }
  }
}

// ---- per-tensor trust ratio -----------------------------------------------
__global__ void __launch_bounds__(kThreads) k_lamb_trust(const __grid_constant__ LArgs a) {
  __shared__ double red[64];
  const int t = blockIdx.x;
  const LDev d = a.dev[t];
  const int64_t u0 = d.unit0, u1 = d.unit0 + d.nunits;
  double x = 0.0, y = 0.0;
  for (int64_t u = u0 + threadIdx.x; u < u1; u += kThreads) {
    x += a.part[2 * u];
    y += a.part[2 * u + 1];
  }
  block_sum2(x, y, red);
  if (threadIdx.x == 0) {
    const double rn = sqrt(x), pn = sqrt(y);
    const double tr = (pn > 0.0 && rn > 0.0) ? pn / rn : 1.0;
    a.trust[t] = tr;
    a.coef[t] = a.lr * tr;
  }
}

// ---- pass 2: update --------------------------------------------------------
__device__ __forceinline__ void update_vec(const LDev& d, const LArgs& a, float c, int64_t e0, int64_t nv) {
  for (int64_t v0 = threadIdx.x; v0 < nv; v0 += kBatchU * kThreads) {
    float4 m[kBatchU], v[kBatchU], p[kBatchU];
#pragma unroll
    for (int k = 0; k < kBatchU; ++k) {
      const int64_t e = e0 + 4 * (v0 + k * kThreads);
      if (v0 + k * kThreads < nv) {
        m[k] = ld4(d.m, e);
        v[k] = ld4(d.v, e);
        p[k] = ld4(d.p, e);
      }
    }
#pragma unroll
    for (int k = 0; k < kBatchU; ++k) {
      if (v0 + k * kThreads < nv) {
        const int64_t e = e0 + 4 * (v0 + k * kThreads);
        float po[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float pq = get(p[k], q);
          po[q] = __fmaf_rn(-c, lamb_dir(get(m[k], q), get(v[k], q), pq, a), pq);
        }
        st4(d.p, e, make_float4(po[0], po[1], po[2], po[3]));
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) k_lamb_update(const __grid_constant__ LArgs a) {
  int k = unit_owner(a, blockIdx.x);
  for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
    while (a.pf[k + 1] <= u) ++k;
    const int t = a.ord[k];
    const LDev d = a.dev[t];
    const float c = static_cast<float>(a.coef[t]);
    const int64_t e0 = (u - d.unit0) * kUnit;
    const int64_t e1 = min(d.numel, e0 + kUnit);
    int64_t es = e0;
    if (d.vec) {
      const int64_t nv = (e1 - e0) >> 2;
      update_vec(d, a, c, e0, nv);
      es = e0 + 4 * nv;
    }
    for (int64_t e = es + threadIdx.x; e < e1; e += kThreads) {
      const float pq = __ldcs(d.p + e);
      __stcs(d.p + e, __fmaf_rn(-c, lamb_dir(__ldcs(d.m + e), __ldcs(d.v + e), pq, a), pq));
    }
  }
}

// ---- host side --------------------------------------------------------------
adaf_status fail(adaf_status st, const std::string& msg) { return meo::set_last_error(st, msg.c_str()); }
adaf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ADAF_ERR_CUDA, std::string("lamb: ") + what + ": " + cudaGetErrorString(e));
}
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Layout {
  int64_t units = 0;
  size_t off_trust = 0, off_coef = 0, off_dev = 0, off_pf = 0, off_ord = 0, off_part = 0, bytes = 0;
};

adaf_status check_list(const lamb_tensor* tensors, int32_t n, Layout* L) {
  if (n < 0) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: n < 0");
  if (n > 0 && tensors == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: tensors is NULL");
  int64_t units = 0;
  for (int32_t i = 0; i < n; ++i) {
    const lamb_tensor& x = tensors[i];
    if (x.numel < 0) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: tensor " + std::to_string(i) + ": numel < 0");
    if (x.grad_dtype != ADAF_FLOAT32 && x.grad_dtype != ADAF_BFLOAT16)
      return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: tensor " + std::to_string(i) + ": unknown grad_dtype");
    if (x.numel > kMaxNumel)
      return fail(ADAF_ERR_UNSUPPORTED, "lamb: tensor " + std::to_string(i) + " has more than 2^40 values");
    units += (x.numel + kUnit - 1) / kUnit;
  }
  if (units > INT32_MAX) return fail(ADAF_ERR_UNSUPPORTED, "lamb: more than 2^31 work units");
  L->units = units;
  size_t o = 0;
  L->off_trust = o; o = round_up(o + sizeof(double) * n, 256);
  L->off_coef = o;  o = round_up(o + sizeof(double) * n, 256);
  L->off_dev = o;   o += sizeof(LDev) * n;
  L->off_pf = o;    o += sizeof(int64_t) * (n + 1);
  L->off_ord = o;   o = round_up(o + sizeof(int32_t) * n, 256);
  L->off_part = o;  o = round_up(o + sizeof(double) * 2 * units, 256);
  L->bytes = o;
  return ADAF_OK;
}

adaf_status check_hp(const lamb_hparams* hp) {
  if (hp == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: hparams is NULL");
  if (!std::isfinite(hp->lr) || hp->lr < 0.0) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: invalid learning rate");
  if (!std::isfinite(hp->eps) || hp->eps < 0.0) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: invalid eps");
  if (!std::isfinite(hp->beta1) || hp->beta1 < 0.0 || hp->beta1 >= 1.0)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: invalid beta1 (needs 0 <= beta1 < 1)");
  if (!std::isfinite(hp->beta2) || hp->beta2 < 0.0 || hp->beta2 >= 1.0)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: invalid beta2 (needs 0 <= beta2 < 1)");
  if (!std::isfinite(hp->weight_decay) || hp->weight_decay < 0.0)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: invalid weight_decay");
  return ADAF_OK;
}

// Pinned upload ring (per device): a slot is rewritten only after the copy
// that last read it has executed.
constexpr int kRing = 4;
struct Slot {
  void* host = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;
  bool used = false;
};
struct DeviceState {
  Slot ring[kRing];
  int next = 0;
  int grid = 0;  // persistent CTAs for the streaming passes
  std::vector<cudaEvent_t> free_events;
  meo::TableCache tables;  // device copies of the descriptor table (host_copy.cuh)
};

const char* const kKernelNames[] = {"k_lamb_moments", "k_lamb_trust", "k_lamb_update"};
constexpr int kNumKernels = 3;
struct ProfRecord {
  int slot;
  int device;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;
bool g_profile = false;
std::vector<ProfRecord> g_prof;

cudaError_t get_event(DeviceState& ds, cudaEvent_t* ev) {
  if (!ds.free_events.empty()) {
    *ev = ds.free_events.back();
    ds.free_events.pop_back();
    return cudaSuccess;
  }
  return cudaEventCreate(ev);
}

}  // namespace

extern "C" {

adaf_status lamb_validate(const lamb_hparams* hp) { return check_hp(hp); }

adaf_status lamb_workspace_size(const lamb_tensor* tensors, int32_t n, size_t* bytes) {
  if (bytes == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: bytes is NULL");
  Layout L;
  adaf_status st = check_list(tensors, n, &L);
  if (st != ADAF_OK) return st;
  *bytes = n == 0 ? 0 : L.bytes;  // an empty list launches nothing
  return ADAF_OK;
}

adaf_status lamb_step(const lamb_tensor* tensors, int32_t n, int64_t step, const lamb_hparams* hp,
                      void* workspace, size_t workspace_bytes, void* stream) {
  adaf_status st = check_hp(hp);
  if (st != ADAF_OK) return st;
  if (step < 1) return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: step must be >= 1");
  Layout L;
  st = check_list(tensors, n, &L);
  if (st != ADAF_OK) return st;
  for (int32_t i = 0; i < n; ++i) {
    const lamb_tensor& x = tensors[i];
    if (x.numel > 0 && (x.p == nullptr || x.g == nullptr || x.exp_avg == nullptr || x.exp_avg_sq == nullptr))
      return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: tensor " + std::to_string(i) + " has a NULL pointer");
    const size_t ge = x.grad_dtype == ADAF_BFLOAT16 ? 2 : 4;
    if (!aligned(x.p, 4) || !aligned(x.exp_avg, 4) || !aligned(x.exp_avg_sq, 4) || !aligned(x.g, ge))
      return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: tensor " + std::to_string(i) + " is not element-aligned");
  }
  if (n == 0) return ADAF_OK;
  if (workspace == nullptr || !aligned(workspace, 256))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: workspace is NULL or not 256-byte aligned");
  if (workspace_bytes < L.bytes)
    return fail(ADAF_ERR_WORKSPACE_TOO_SMALL, "lamb: workspace needs " + std::to_string(L.bytes) + " bytes");

  // Host copy of the descriptors, the unit prefix in unit order (tensors
  // with bf16 gradients first) and the tensor at each position.
  const size_t hdr = L.off_ord + sizeof(int32_t) * n - L.off_dev;
  std::vector<unsigned char> h(hdr);
  LDev* dv = reinterpret_cast<LDev*>(h.data());
  int64_t* pf = reinterpret_cast<int64_t*>(h.data() + (L.off_pf - L.off_dev));
  int32_t* ord = reinterpret_cast<int32_t*>(h.data() + (L.off_ord - L.off_dev));
  int64_t u = 0, u_bf16 = 0;
  int32_t pos = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int32_t i = 0; i < n; ++i) {
      const lamb_tensor& x = tensors[i];
      if ((x.grad_dtype == ADAF_BFLOAT16) != (pass == 0)) continue;
      LDev d{};
      d.p = x.p;
      d.g = x.g;
      d.m = x.exp_avg;
      d.v = x.exp_avg_sq;
      d.numel = x.numel;
      d.unit0 = u;
      d.nunits = (x.numel + kUnit - 1) / kUnit;
      d.gdt = x.grad_dtype;
      const size_t ga = x.grad_dtype == ADAF_BFLOAT16 ? 8 : 16;
      d.vec = aligned(x.p, 16) && aligned(x.exp_avg, 16) && aligned(x.exp_avg_sq, 16) && aligned(x.g, ga);
      dv[i] = d;
      pf[pos] = u;
      ord[pos] = i;
      ++pos;
      u += d.nunits;
    }
    if (pass == 0) u_bf16 = u;
  }
  pf[n] = u;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  LArgs a{};
  a.dev = reinterpret_cast<const LDev*>(ws + L.off_dev);
  a.pf = reinterpret_cast<const int64_t*>(ws + L.off_pf);
  a.ord = reinterpret_cast<const int32_t*>(ws + L.off_ord);
  a.part = reinterpret_cast<double*>(ws + L.off_part);
  a.trust = reinterpret_cast<double*>(ws + L.off_trust);
  a.coef = reinterpret_cast<double*>(ws + L.off_coef);
  a.units = L.units;
  a.n = n;
  a.b1 = static_cast<float>(hp->beta1);
  a.omb1 = static_cast<float>(1.0 - hp->beta1);
  a.b2 = static_cast<float>(hp->beta2);
  a.omb2 = static_cast<float>(1.0 - hp->beta2);
  const double bc1 = hp->bias_correction ? 1.0 - std::pow(hp->beta1, static_cast<double>(step)) : 1.0;
  const double bc2 = hp->bias_correction ? 1.0 - std::pow(hp->beta2, static_cast<double>(step)) : 1.0;
  if (!(bc1 > 0.0) || !(bc2 > 0.0))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb: 1 - beta^t rounds to 0");
  a.inv_bc1 = static_cast<float>(1.0 / bc1);
  a.inv_bc2 = static_cast<float>(1.0 / bc2);
  a.eps = static_cast<float>(hp->eps);
  a.wd = static_cast<float>(hp->weight_decay);
  a.lr = hp->lr;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  DeviceState& ds = g_dev[device];
  if (ds.grid == 0) {
    int sms = 0, occ = 0;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
      return cuda_fail(err, "cudaDeviceGetAttribute");
    int occ2 = 0, occ3 = 0;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_lamb_moments<__nv_bfloat16>, kThreads, 0)) !=
        cudaSuccess)
      return cuda_fail(err, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, k_lamb_moments<float>, kThreads, 0)) != cudaSuccess)
      return cuda_fail(err, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ3, k_lamb_update, kThreads, 0)) != cudaSuccess)
      return cuda_fail(err, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    ds.grid = sms * std::max(1, std::min(occ, std::min(occ2, occ3)));
  }
  // The descriptor table comes from a kept device copy when one holds the
  // same bytes (TableCache); otherwise it is staged in a pinned ring slot and
  // a kernel reads it from host memory (no copy engine, host_copy.cuh).
  auto upload = [&](unsigned char* dst) -> cudaError_t {
    Slot& sl = ds.ring[ds.next];
    ds.next = (ds.next + 1) % kRing;
    cudaError_t e = cudaSuccess;
    if (sl.used && (e = cudaEventSynchronize(sl.done)) != cudaSuccess) return e;
    const size_t up = round_up(hdr, 16);  // the upload moves whole 16-byte words
    if (sl.cap < up) {
      if (sl.host) cudaFreeHost(sl.host);
      sl.host = nullptr;
      sl.cap = 0;
      if ((e = cudaHostAlloc(&sl.host, up, cudaHostAllocPortable | cudaHostAllocMapped)) != cudaSuccess) return e;
      sl.cap = up;
    }
    if (sl.done == nullptr && (e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming)) != cudaSuccess)
      return e;
    std::memcpy(sl.host, h.data(), hdr);
    if ((e = meo::copy_from_host(dst, sl.host, up, s)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(sl.done, s)) != cudaSuccess) return e;
    sl.used = true;
    return cudaSuccess;
  };
  unsigned char* tab = nullptr;
  meo::RecordOnExit used_guard;
  if ((err = ds.tables.lookup(h.data(), hdr, s, upload, &tab, &used_guard.ev)) != cudaSuccess)
    return cuda_fail(err, "descriptor table upload");
  used_guard.s = s;
  a.dev = reinterpret_cast<const LDev*>(tab);
  a.pf = reinterpret_cast<const int64_t*>(tab + (L.off_pf - L.off_dev));
  a.ord = reinterpret_cast<const int32_t*>(tab + (L.off_ord - L.off_dev));

  auto grid_for = [&](int64_t units) { return static_cast<int>(std::min<int64_t>(ds.grid, std::max<int64_t>(1, units))); };
  for (int k = 0; k < kNumKernels; ++k) {
    ProfRecord rec{k, device, nullptr, nullptr};
    if (g_profile) {
      if ((err = get_event(ds, &rec.start)) != cudaSuccess) return cuda_fail(err, "cudaEventCreate (profile)");
      if ((err = get_event(ds, &rec.stop)) != cudaSuccess) return cuda_fail(err, "cudaEventCreate (profile)");
      if ((err = cudaEventRecord(rec.start, s)) != cudaSuccess) return cuda_fail(err, "cudaEventRecord (profile)");
    }
    if (k == 0) {
      if (u_bf16 > 0) k_lamb_moments<__nv_bfloat16><<<grid_for(u_bf16), kThreads, 0, s>>>(a, 0, u_bf16);
      if (L.units > u_bf16) k_lamb_moments<float><<<grid_for(L.units - u_bf16), kThreads, 0, s>>>(a, u_bf16, L.units);
    } else if (k == 1) {
      k_lamb_trust<<<n, kThreads, 0, s>>>(a);
    } else if (L.units > 0) {
      k_lamb_update<<<grid_for(L.units), kThreads, 0, s>>>(a);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err, kKernelNames[k]);
    if (g_profile) {
      if ((err = cudaEventRecord(rec.stop, s)) != cudaSuccess) return cuda_fail(err, "cudaEventRecord (profile)");
      g_prof.push_back(rec);
    }
  }
  return ADAF_OK;
}

}  // extern "C"

namespace meo {
void lamb_forget_tables() {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  const bool have_dev = cudaGetDevice(&cur) == cudaSuccess;
  for (auto& kv : g_dev) {
    if (cudaSetDevice(kv.first) == cudaSuccess) kv.second.tables.clear();
  }
  if (have_dev) cudaSetDevice(cur);
}
}  // namespace meo

extern "C" {

adaf_status lamb_trust_ratios(const void* workspace, int32_t n, double* out, void* stream) {
  if (n < 0 || (n > 0 && (workspace == nullptr || out == nullptr)))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "lamb_trust_ratios: NULL pointer or n < 0");
  if (n == 0) return ADAF_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(out, workspace, sizeof(double) * n, cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  return err == cudaSuccess ? ADAF_OK : cuda_fail(err, "trust ratio read-back");
}

adaf_status lamb_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profile = on != 0;
  return ADAF_OK;
}

adaf_status lamb_profile_read(double* ms, int64_t* launches, int32_t nk) {
  std::lock_guard<std::mutex> lock(g_mu);
  adaf_status st = ADAF_OK;
  for (ProfRecord& r : g_prof) {
    float el = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&el, r.start, r.stop);
    if (e != cudaSuccess && st == ADAF_OK) st = cuda_fail(e, "profile event");
    if (r.slot < nk) {
      if (ms) ms[r.slot] += el;
      if (launches) launches[r.slot] += 1;
    }
    DeviceState& ds = g_dev[r.device];
    ds.free_events.push_back(r.start);
    ds.free_events.push_back(r.stop);
  }
  g_prof.clear();
  return st;
}

int32_t lamb_num_kernels(void) { return kNumKernels; }

const char* lamb_kernel_name(int32_t k) { return (k >= 0 && k < kNumKernels) ? kKernelNames[k] : ""; }

}  // extern "C"
