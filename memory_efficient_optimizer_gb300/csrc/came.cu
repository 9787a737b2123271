// Multi-tensor CAME step for sm_103a: the C ABI of include/came.h.
//
// CAME (the Colossal-AI distributed-optimizer article, overview table and
// "其余优化器的关键参数速查" / DistributedCAME; the rule is the CAME algorithm of
// arXiv:2307.02047) keeps Adafactor's factored second moment and adds a
// momentum m of the clipped update and a factored "instability" statistic
// of (uh - m)^2 that scales the final step.  Three results are needed over
// whole slices or tensors before an element can move on (the second-moment
// factors, RMS(u), the instability factors), so a step is four streaming
// passes with small reductions between them:
//
//   k_came_pass_a   g -> per-tile row and column sums of g^2        (read g)
//   k_came_panel    (bf16 matrices with 2048 <= W <= 14336, instead of
//                   passes a and b) g -> the row EMA, per-chunk column sums
//                   of g^2 and of g^2 / r_i: sum(u^2) without a second read
//                   of g (the shared row-panel pass, row_panel.cuh)
//   k_came_stats    row/col EMAs of the means (+ eps1), row-chunk sums;
//                   panel tensors: the column EMA and sum_j D_j / c_j
//   k_came_means    mean(r) per slice
//   k_came_pass_b   per-tile sum(u^2), u = g (r_i/mean r)^-1/2 c_j^-1/2 (read g)
//   k_came_clip     coef = 1 / max(1, RMS(u) / d) per tensor
//   k_came_pass_c   uh = coef u; m <- b1 m + (1-b1) uh; per-tile row/column
//                   sums of U = (uh - m)^2, formed as (b1 (uh - m_old))^2
//                   (equal, without the rounding of m)   (read g, m; write m)
//   k_came_stats    R/C EMAs of the means (+ eps2), row-chunk sums
//   k_came_means    mean(R) per slice
//   k_came_pass_d   p <- p - wd lr p - lr m (R_i/mean R)^-1/2 C_j^-1/2
//                                                     (read m, p; write p)
//
// Tensors with ndim < 2 are one row (full per-element v and S); their units
// run inside pass a (v and sum(u^2)) and pass c (m, S and p) and need no
// factored statistics.  Factored tensors are cut into tiles of 256 rows x
// 1024 columns of one slice.  A CTA of 8 warps streams a tile: warp w takes
// rows w, w + 8, ...; each lane owns 8 consecutive columns per 256-column
// chunk (16-byte loads; "vec" class) or one column per 32-column chunk
// ("scalar" class: odd widths, unaligned views), keeps their column sums in
// registers, and the warp reduces each row with a xor tree.  All sums are
// deterministic (fixed orders, no atomics).
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
#include "came.h"
#include "row_panel.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTR = 256;          // tile rows
constexpr int kTC = 1024;         // tile columns
constexpr int64_t kUnit1D = 8192; // values per 1D work unit
constexpr int kRowItem = 1024;    // rows per statistics item
constexpr int kColItem = 256;     // columns per statistics item
constexpr int kClasses = 4;
// vector path with bf16 / fp32 gradients, one column per lane, 1D
enum Cls : int32_t { kVecBF = 0, kVecF = 1, kScalar = 2, k1D = 3 };

struct CDev {
  float* p;
  const void* g;
  float* m;
  float* row;   // second moment factors [B*H], [B*W]
  float* col;
  float* rrow;  // instability factors
  float* rcol;
  float* v;     // 1D: full second moment, full instability
  float* res;
  int64_t B, H, W, n;
  int64_t cb, rb;      // column / row tiles per slice
  int64_t rowpart;     // float offset of [cb][B*H] row partials
  int64_t colpart;     // float offset of [rb][B*W] column partials
  int64_t sp0, nsp;    // sum(u^2) partial slots
  int64_t slice0;      // per-slice mean slots
  int64_t rc0, nrc;    // row-chunk sum slots: B * nrc
  int64_t ncc;         // column items per slice
  int32_t gdt, cls;
  // Row-panel tensors (panel = 1: 8 warps x 2 groups, W <= 4096; 2: 16 x 4,
  // W <= 14336; 0: none): chunks of pr rows, prb per slice.
  int32_t panel, pr;
  int64_t prb;
  int64_t pcol;        // float offset of the panel column partials [B][prb][W] (g^2 and g^2 / r)
  int64_t prc0;        // double offset of the panel row-chunk sums [B][prb]
  int64_t dsum0;       // double offset of sum_j D_j / c_j per column item [B][ncc]
};

constexpr int kPanelCfgs = 2;  // row-panel configurations (CDev::panel - 1)
// Work lists: pass a and pass b walk the tiles of the tensors outside the
// row panels (kListAB), passes c and d those of every tensor (kListCD).
enum List : int32_t { kListAB = 0, kListCD = 1 };

struct CArgs {
  const CDev* dev;
  const int64_t* pf[2][kClasses];   // per list and class: first tile of each member, then the total
  const int32_t* idx[2][kClasses];  // per list and class: tensor index of each member
  int32_t nmem[2][kClasses];
  const int64_t* ppf[kPanelCfgs];   // per panel configuration: first chunk of each member, then the total
  const int32_t* pidx[kPanelCfgs];
  int32_t pnmem[kPanelCfgs];
  float* pcolpart;
  float* pdpart;
  double* prchunk;
  double* dsum;
  const int64_t* item_pf;        // statistics items of factored tensors
  const int32_t* item_idx;
  int32_t nfact;
  float* rowpart;
  float* colpart;
  double* uspart;
  double* rchunk;
  double* mean;   // per slice: mean(r) or mean(R) of the current phase
  double* coef;   // per tensor
  int32_t n;
  int32_t phase;  // statistics kernels: 0 = second moment, 1 = instability
  float b1, omb1, b2, omb2, b3, omb3, eps1, eps2, lr, wdl, clip;
};

// ---- loads -----------------------------------------------------------------
template <int VEC> struct GRaw;
template <> struct GRaw<8> { uint4 a, b; };
template <> struct GRaw<1> { float f; };

// 8 (or 1) gradient values at e, of either dtype, widened to fp32 (exact).
__device__ __forceinline__ void load_g(GRaw<8>& r, const void* g, int gdt, int64_t e) {
  if (gdt == ADAF_BFLOAT16) {
    r.a = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(g) + e));
  } else {
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const float*>(g) + e);
    r.a = __ldcs(q);
    r.b = __ldcs(q + 1);
  }
}
__device__ __forceinline__ void load_g(GRaw<1>& r, const void* g, int gdt, int64_t e) {
  r.f = gdt == ADAF_BFLOAT16
            ? __uint_as_float(static_cast<uint32_t>(__ldcs(static_cast<const unsigned short*>(g) + e)) << 16)
            : __ldcs(static_cast<const float*>(g) + e);
}
__device__ __forceinline__ void widen(const GRaw<8>& r, int gdt, float (&x)[8]) {
  if (gdt == ADAF_BFLOAT16) {
    const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  } else {
    const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = __uint_as_float(w[k]);
  }
}
__device__ __forceinline__ void widen(const GRaw<1>& r, int, float (&x)[1]) { x[0] = r.f; }

template <int VEC> __device__ __forceinline__ void load_f(float (&y)[VEC], const float* p);
template <> __device__ __forceinline__ void load_f<8>(float (&y)[8], const float* p) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w; y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
}
template <> __device__ __forceinline__ void load_f<1>(float (&y)[1], const float* p) { y[0] = __ldcs(p); }
template <int VEC> __device__ __forceinline__ void store_f(float* p, const float (&y)[VEC]);
template <> __device__ __forceinline__ void store_f<8>(float* p, const float (&y)[8]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(y[0], y[1], y[2], y[3]));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(y[4], y[5], y[6], y[7]));
}
template <> __device__ __forceinline__ void store_f<1>(float* p, const float (&y)[1]) { __stcs(p, y[0]); }

// Gradient loads of the tile passes.  GK = 0: the dtype is read at run time
// (fp32 vectors take two 16-byte loads); GK = 1: bf16 on the vector path,
// one 16-byte load into 4 registers, which leaves room for more rows in
// flight in the read-only passes.
struct GRawB8 { uint4 a; };
template <int VEC, int GK> struct GSel {
  using Raw = GRaw<VEC>;
  static constexpr int RPI_A = 2, RPI_B = 2;  // rows per iteration, passes a and b
  static __device__ __forceinline__ void load(Raw& r, const void* g, int gdt, int64_t e) { load_g(r, g, gdt, e); }
  static __device__ __forceinline__ void unpack(const Raw& r, int gdt, float (&x)[VEC]) { widen(r, gdt, x); }
};
template <> struct GSel<8, 1> {
  using Raw = GRawB8;
  static constexpr int RPI_A = 3, RPI_B = 4;
  static __device__ __forceinline__ void load(Raw& r, const void* g, int, int64_t e) {
    r.a = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(g) + e));
  }
  static __device__ __forceinline__ void unpack(const Raw& r, int, float (&x)[8]) {
    const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
};

// ---- reductions --------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Deterministic CTA sum; the result is valid in thread 0.
__device__ __forceinline__ double block_sum(double v, double* red) {
  v = warp_sum_d(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // red of the previous use is read
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kWarps; ++w) s += red[w];
  return s;
}

// ---- tile geometry -------------------------------------------------------------
template <int VEC> struct Lay {
  static constexpr int CH = kTC / (32 * VEC);  // chunks per tile row
  static constexpr int CG = VEC == 8 ? CH : 8;  // chunks loaded together (registers)
  // lane's first column of chunk k inside the tile
  static __device__ __forceinline__ int col(int k, int lane) { return k * 32 * VEC + lane * VEC; }
};

struct Tile {
  int64_t b, r, c;  // slice, row tile, column tile
  int64_t i0, i1, j0;
};
// Unit indices and their divisors fit 32 bits (int32 prefix arrays); a
// 32-bit unsigned division avoids the FP64 pipe that 64-bit division uses.
__device__ __forceinline__ void udivmod32(int64_t n, int64_t d, int64_t& q, int64_t& r) {
  const uint32_t nn = static_cast<uint32_t>(n), dd = static_cast<uint32_t>(d);
  const uint32_t qq = nn / dd;
  q = qq;
  r = nn - qq * dd;
}
__device__ __forceinline__ Tile tile_of(const CDev& d, int64_t local) {
  Tile t;
  int64_t q;
  udivmod32(local, d.cb, q, t.c);
  udivmod32(q, d.rb, t.b, t.r);
  t.i0 = t.r * kTR;
  t.i1 = min(d.H, t.i0 + kTR);
  t.j0 = t.c * kTC;
  return t;
}

// Column sums of the tile's rows, held per lane, added across the warps in
// warp order through shared memory and stored to the column partials.
template <int VEC>
__device__ __forceinline__ void store_col_sums(const CDev& d, const CArgs& a, const Tile& tl,
                                               const float (&cacc)[Lay<VEC>::CH * VEC], float* colbuf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* mine = colbuf + warp * kTC;
#pragma unroll
  for (int k = 0; k < Lay<VEC>::CH; ++k)
#pragma unroll
    for (int v = 0; v < VEC; ++v) mine[Lay<VEC>::col(k, lane) + v] = cacc[k * VEC + v];
  __syncthreads();
  const int ncl = static_cast<int>(min(static_cast<int64_t>(kTC), d.W - tl.j0));
  float* cp = a.colpart + d.colpart + tl.r * (d.B * d.W) + tl.b * d.W + tl.j0;
  for (int cl = threadIdx.x; cl < ncl; cl += kThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += colbuf[w * kTC + cl];
    cp[cl] = s;
  }
  __syncthreads();  // colbuf is reused by the next tile
}

// Walks the units of one member list: calls body(d, t, local) for each.
template <typename Body>
__device__ __forceinline__ void walk_list(const CArgs& a, const int64_t* pf, const int32_t* idx, int nm, Body&& body) {
  int k = 0;
  for (int64_t u = blockIdx.x; u < pf[nm]; u += gridDim.x) {
    while (pf[k + 1] <= u) ++k;
    const int t = idx[k];
    body(a.dev[t], t, u - pf[k]);
  }
}
// Walks the tiles of one class in one list (kListAB, kListCD).
template <typename Body>
__device__ __forceinline__ void walk(const CArgs& a, int list, int cls, Body&& body) {
  walk_list(a, a.pf[list][cls], a.idx[list][cls], a.nmem[list][cls], body);
}

// ---- pass a: row / column sums of g^2 (factored), v and sum(u^2) (1D) -------
template <int VEC, int GK>
__device__ __forceinline__ void pass_a_tile(const CDev& d, const CArgs& a, int64_t local, float* colbuf) {
  constexpr int CH = Lay<VEC>::CH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Tile tl = tile_of(d, local);
  const int64_t base = tl.b * d.H * d.W;
  float cacc[CH * VEC];
#pragma unroll
  for (int k = 0; k < CH * VEC; ++k) cacc[k] = 0.f;
  float* rp = a.rowpart + d.rowpart + tl.c * (d.B * d.H) + tl.b * d.H;
  constexpr int CG = Lay<VEC>::CG;
  using G = GSel<VEC, GK>;
  constexpr int RPI = G::RPI_A;  // rows per iteration (rows i, i + kWarps, ...): more loads in flight
  for (int64_t i = tl.i0 + warp; i < tl.i1; i += RPI * kWarps) {
    float rs[RPI];
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr) rs[rr] = 0.f;
#pragma unroll
    for (int kg = 0; kg < CH; kg += CG) {
      if (tl.j0 + Lay<VEC>::col(kg, 0) >= d.W) break;  // past the row's end (warp-uniform)
      typename G::Raw raw[RPI][CG];
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr)
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int64_t j = tl.j0 + Lay<VEC>::col(kg + k, lane);
          if (i + rr * kWarps < tl.i1 && j < d.W) G::load(raw[rr][k], d.g, d.gdt, base + (i + rr * kWarps) * d.W + j);
        }
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr)
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int64_t j = tl.j0 + Lay<VEC>::col(kg + k, lane);
          if (i + rr * kWarps < tl.i1 && j < d.W) {
            float x[VEC];
            G::unpack(raw[rr][k], d.gdt, x);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              const float q = x[v] * x[v];
              cacc[(kg + k) * VEC + v] += q;
              rs[rr] += q;
            }
          }
        }
    }
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr) {
      const float t = warp_sum(rs[rr]);
      if (lane == 0 && i + rr * kWarps < tl.i1) rp[i + rr * kWarps] = t;
    }
  }
  store_col_sums<VEC>(d, a, tl, cacc, colbuf);
}

__device__ __forceinline__ void pass_a_1d(const CDev& d, const CArgs& a, int64_t local, double* red) {
  const int64_t e0 = local * kUnit1D, e1 = min(d.n, e0 + kUnit1D);
  float acc = 0.f;
  for (int64_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
    GRaw<1> r;
    load_g(r, d.g, d.gdt, e);
    const float x = r.f;
    const float vn = fmaf(a.b2, d.v[e], a.omb2 * fmaf(x, x, a.eps1));
    d.v[e] = vn;
    const float u = x * rsqrtf(vn);
    acc = fmaf(u, u, acc);
  }
  const double s = block_sum(static_cast<double>(acc), red);
  if (threadIdx.x == 0) a.uspart[d.sp0 + local] = s;
}

template <int VEC, int GK>
__global__ void __launch_bounds__(kThreads, 2) k_came_pass_a(const __grid_constant__ CArgs a, int cls) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* colbuf = reinterpret_cast<float*>(smem);
  double* red = reinterpret_cast<double*>(smem + sizeof(float) * kWarps * kTC);
  walk(a, kListAB, cls, [&](const CDev& d, int, int64_t local) {
    if (cls == k1D) pass_a_1d(d, a, local, red);
    else pass_a_tile<VEC, GK>(d, a, local, colbuf);
  });
}

// ---- row-panel pass: statistics and sum(u^2) in one read of g ----------------
// The shared row-panel pass (row_panel.cuh) over chunks of d.pr full rows of
// bf16 matrices: r_i updated in place (beta2, eps1), the chunk's column sums
// C_j of g^2 and D_j of g^2 / r_i, and the chunk's sum of the new r_i.  Then
// sum(u^2) = sum_ij g^2 mean(r) / (r_i c_j) = mean(r) sum_j D_j / c_j
// (k_came_stats, k_came_clip): pass b does not run for these tensors.
template <int NW, int G, int S, int MINB>
__global__ void __launch_bounds__(NW * 32, MINB) k_came_panel(const __grid_constant__ CArgs a, int q) {
  using C = meo::panel::Cfg<__nv_bfloat16, NW, G, S>;
  extern __shared__ __align__(16) unsigned char smem[];
  double* red = reinterpret_cast<double*>(smem + C::kBytes);
  walk_list(a, a.ppf[q], a.pidx[q], a.pnmem[q], [&](const CDev& d, int, int64_t local) {
    int64_t b, chunk;
    udivmod32(local, d.prb, b, chunk);
    const int32_t H = static_cast<int32_t>(d.H), W = static_cast<int32_t>(d.W);
    const int32_t c0 = static_cast<int32_t>(chunk) * d.pr, c1 = min(H, c0 + d.pr);
    const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(d.g) + b * d.H * d.W;
    auto where = [&]() {
      const int64_t off = d.pcol + (b * d.prb + chunk) * d.W;
      return meo::panel::Partials{a.pcolpart + off, a.pdpart + off};
    };
    float rsum = 0.f, psq = 0.f;
    meo::panel::run_chunk<__nv_bfloat16, NW, G, S, false>(smem, gb, nullptr, d.row + b * d.H, W, c0, c1, a.b2,
                                                          a.omb2, a.eps1, where, rsum, psq);
    // (its barriers also order this chunk's last reads of the ring before
    // the next chunk's first copies)
    const double tot = meo::panel::block_sum<NW>(static_cast<double>(rsum), red);
    if (threadIdx.x == 0) a.prchunk[d.prc0 + b * d.prb + chunk] = tot;
  });
  meo::panel::cp_async_wait_all();  // only empty groups can be pending here
}

// ---- statistics: EMAs of the row / column means, row-chunk sums ------------
// phase 0: r, c from the g^2 partials (beta2, eps1); phase 1: R, C from the
// U partials (beta3, eps2).  Items: B * nrc row chunks, then B * ncc column
// chunks of each factored tensor.
// Compensated (Kahan) fp32 addition: this GPU's FP64 rate is a small
// fraction of its FP32 rate, and the partial sums below have up to a few
// hundred terms.
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = x - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// Column sums of one column item: for the kColItem columns [j0, j0 + 256)
// (j0 a multiple of 256, W % 8 == 0 when VEC), sums over nr partial rows
// r of src[r * stride + j] (and of src2 with TWO), compensated fp32.  Warp w
// adds the rows w, w + 8, ...; lane l the 8 consecutive columns 8 l .. 8 l + 7
// (VEC) or the columns l + 32 m; then the 8 warp sums of each column are
// added in warp order through shared memory (part: 2 x kWarps x kColItem
// floats).  Thread t gets the sums of column j0 + t.  Deterministic: fixed
// orders throughout.
template <bool VEC, bool TWO>
__device__ __forceinline__ void col_item_sums(const float* src, const float* src2, int64_t stride, int64_t nr,
                                              int64_t j0, int64_t W, float* part, double& s1, double& s2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float a1[8], c1[8], a2[8], c2[8];
#pragma unroll
  for (int v = 0; v < 8; ++v) a1[v] = c1[v] = a2[v] = c2[v] = 0.f;
  auto col = [&](int v) -> int64_t { return VEC ? j0 + lane * 8 + v : j0 + lane + 32 * v; };
  for (int64_t r = warp; r < nr; r += kWarps) {
    const float* row1 = src + r * stride;
    const float* row2 = TWO ? src2 + r * stride : nullptr;
    if (VEC) {
      if (col(0) < W) {
        const float4 x0 = *reinterpret_cast<const float4*>(row1 + col(0));
        const float4 x1 = *reinterpret_cast<const float4*>(row1 + col(0) + 4);
        const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int v = 0; v < 8; ++v) kahan_add(a1[v], c1[v], x[v]);
        if (TWO) {
          const float4 y0 = *reinterpret_cast<const float4*>(row2 + col(0));
          const float4 y1 = *reinterpret_cast<const float4*>(row2 + col(0) + 4);
          const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
          for (int v = 0; v < 8; ++v) kahan_add(a2[v], c2[v], y[v]);
        }
      }
    } else {
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        if (col(v) < W) {
          kahan_add(a1[v], c1[v], row1[col(v)]);
          if (TWO) kahan_add(a2[v], c2[v], row2[col(v)]);
        }
      }
    }
  }
  __syncthreads();  // part of the previous item is read
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const int cl = static_cast<int>(col(v) - j0);
    part[warp * kColItem + cl] = a1[v];
    if (TWO) part[(kWarps + warp) * kColItem + cl] = a2[v];
  }
  __syncthreads();
  float t1 = 0.f, k1 = 0.f, t2 = 0.f, k2 = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    kahan_add(t1, k1, part[w * kColItem + threadIdx.x]);
    if (TWO) kahan_add(t2, k2, part[(kWarps + w) * kColItem + threadIdx.x]);
  }
  s1 = t1;
  s2 = t2;
}

__global__ void __launch_bounds__(kThreads) k_came_stats(const __grid_constant__ CArgs a) {
  __shared__ double red[kWarps];
  __shared__ float part[2 * kWarps * kColItem];
  static_assert(kColItem == kThreads && kColItem == 32 * 8, "a column item is one column per thread");
  const float beta = a.phase ? a.b3 : a.b2;
  const float omb = a.phase ? a.omb3 : a.omb2;
  const double eps = a.phase ? a.eps2 : a.eps1;
  int k = 0;
  for (int64_t it = blockIdx.x; it < a.item_pf[a.nfact]; it += gridDim.x) {
    while (a.item_pf[k + 1] <= it) ++k;
    const CDev d = a.dev[a.item_idx[k]];
    float* rowst = a.phase ? d.rrow : d.row;
    float* colst = a.phase ? d.rcol : d.col;
    const int64_t local = it - a.item_pf[k];
    const bool panel0 = a.phase == 0 && d.panel != 0;  // rows done by the row-panel pass
    if (local < d.B * d.nrc) {
      if (panel0) continue;
      int64_t b, q;
      udivmod32(local, d.nrc, b, q);
      const int64_t i0 = q * kRowItem, i1 = min(d.H, i0 + kRowItem);
      double acc = 0.0;
      for (int64_t i = i0 + threadIdx.x; i < i1; i += kThreads) {
        double s = 0.0;
        for (int64_t c = 0; c < d.cb; ++c) s += a.rowpart[d.rowpart + c * (d.B * d.H) + b * d.H + i];
        const float mean = static_cast<float>(s / static_cast<double>(d.W) + eps);
        const float rn = fmaf(beta, rowst[b * d.H + i], omb * mean);
        rowst[b * d.H + i] = rn;
        acc += rn;
      }
      const double tot = block_sum(acc, red);
      if (threadIdx.x == 0) a.rchunk[d.rc0 + local] = tot;
    } else if (panel0) {
      // column EMA from the chunks' sums of g^2, and this item's share of
      // sum_j D_j / c_j from the chunks' sums of g^2 / r_i
      const int64_t l2 = local - d.B * d.nrc;
      int64_t b, q;
      udivmod32(l2, d.ncc, b, q);
      const int64_t j = q * kColItem + threadIdx.x;
      const int64_t o = d.pcol + b * d.prb * d.W;  // panel tensors: W % 8 == 0
      double sc, sd;
      col_item_sums<true, true>(a.pcolpart + o, a.pdpart + o, d.W, d.prb, q * kColItem, d.W, part, sc, sd);
      double term = 0.0;
      if (j < d.W) {
        const float mean = static_cast<float>(sc / static_cast<double>(d.H) + eps);
        const float cn = fmaf(beta, colst[b * d.W + j], omb * mean);
        colst[b * d.W + j] = cn;
        term = sd / static_cast<double>(cn);
      }
      const double tot = block_sum(term, red);
      if (threadIdx.x == 0) a.dsum[d.dsum0 + b * d.ncc + q] = tot;
    } else {
      const int64_t l2 = local - d.B * d.nrc;
      int64_t b, q;
      udivmod32(l2, d.ncc, b, q);
      const int64_t j = q * kColItem + threadIdx.x;
      const float* src = a.colpart + d.colpart + b * d.W;
      const bool vec = d.W % 8 == 0 && (d.colpart + b * d.W) % 4 == 0 && (d.B * d.W) % 4 == 0;
      double s, unused;
      if (vec) col_item_sums<true, false>(src, nullptr, d.B * d.W, d.rb, q * kColItem, d.W, part, s, unused);
      else col_item_sums<false, false>(src, nullptr, d.B * d.W, d.rb, q * kColItem, d.W, part, s, unused);
      if (j < d.W) {
        const float mean = static_cast<float>(s / static_cast<double>(d.H) + eps);
        colst[b * d.W + j] = fmaf(beta, colst[b * d.W + j], omb * mean);
      }
    }
  }
}

// mean(r) (phase 0) or mean(R) (phase 1) of every slice: one CTA per factored tensor.
__global__ void __launch_bounds__(kThreads) k_came_means(const __grid_constant__ CArgs a) {
  __shared__ double red[kWarps];
  const CDev d = a.dev[a.item_idx[blockIdx.x]];
  const bool panel0 = a.phase == 0 && d.panel != 0;  // row sums from the row-panel pass
  for (int64_t b = 0; b < d.B; ++b) {
    double s = 0.0;
    if (panel0)
      for (int64_t q = threadIdx.x; q < d.prb; q += kThreads) s += a.prchunk[d.prc0 + b * d.prb + q];
    else
      for (int64_t q = threadIdx.x; q < d.nrc; q += kThreads) s += a.rchunk[d.rc0 + b * d.nrc + q];
    const double tot = block_sum(s, red);
    if (threadIdx.x == 0) a.mean[d.slice0 + b] = tot / static_cast<double>(d.H);
  }
}

// ---- pass b: sum(u^2) per tile ------------------------------------------------
// sum_ij u^2 = sum_i (mean r / r_i) sum_j g^2 / c_j.
template <int VEC, int GK>
__device__ __forceinline__ void pass_b_tile(const CDev& d, const CArgs& a, int64_t local, float* cinv, double* red) {
  constexpr int CH = Lay<VEC>::CH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Tile tl = tile_of(d, local);
  const int64_t base = tl.b * d.H * d.W;
  const float mr = static_cast<float>(a.mean[d.slice0 + tl.b]);
  __syncthreads();  // cinv of the previous tile is read
  for (int cl = threadIdx.x; cl < kTC; cl += kThreads) {
    const int64_t j = tl.j0 + cl;
    cinv[cl] = j < d.W ? 1.0f / d.col[tl.b * d.W + j] : 0.f;
  }
  __syncthreads();
  constexpr int CG = Lay<VEC>::CG;
  float acc = 0.f;
  using G = GSel<VEC, GK>;
  constexpr int RPI = G::RPI_B;  // rows per iteration (rows i, i + kWarps, ...): more loads in flight
  for (int64_t i = tl.i0 + warp; i < tl.i1; i += RPI * kWarps) {
    float ts[RPI];
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr) ts[rr] = 0.f;
#pragma unroll
    for (int kg = 0; kg < CH; kg += CG) {
      if (tl.j0 + Lay<VEC>::col(kg, 0) >= d.W) break;
      typename G::Raw raw[RPI][CG];
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr)
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int64_t j = tl.j0 + Lay<VEC>::col(kg + k, lane);
          if (i + rr * kWarps < tl.i1 && j < d.W) G::load(raw[rr][k], d.g, d.gdt, base + (i + rr * kWarps) * d.W + j);
        }
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr)
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int cl = Lay<VEC>::col(kg + k, lane);
          if (i + rr * kWarps < tl.i1 && tl.j0 + cl < d.W) {
            float x[VEC];
            G::unpack(raw[rr][k], d.gdt, x);
#pragma unroll
            for (int v = 0; v < VEC; ++v) ts[rr] = fmaf(x[v] * x[v], cinv[cl + v], ts[rr]);
          }
        }
    }
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr)
      if (i + rr * kWarps < tl.i1) acc = fmaf(mr / d.row[tl.b * d.H + i + rr * kWarps], ts[rr], acc);
  }
  const double s = block_sum(static_cast<double>(acc), red);
  if (threadIdx.x == 0) a.uspart[d.sp0 + local] = s;
}

template <int VEC, int GK>
__global__ void __launch_bounds__(kThreads, 2) k_came_pass_b(const __grid_constant__ CArgs a, int cls) {
  __shared__ __align__(16) float cinv[kTC];
  __shared__ double red[kWarps];
  walk(a, kListAB, cls, [&](const CDev& d, int, int64_t local) { pass_b_tile<VEC, GK>(d, a, local, cinv, red); });
}

// ---- clip: coef = 1 / max(1, RMS(u) / d), one CTA per tensor ---------------
__global__ void __launch_bounds__(kThreads) k_came_clip(const __grid_constant__ CArgs a) {
  __shared__ double red[kWarps];
  const CDev d = a.dev[blockIdx.x];
  double tot = 0.0;
  if (d.panel) {
    // sum(u^2) = sum_b mean(r)_b sum_j D_bj / c_bj (a.mean: mean(r) of phase 0)
    for (int64_t b = 0; b < d.B; ++b) {
      double s = 0.0;
      for (int64_t q = threadIdx.x; q < d.ncc; q += kThreads) s += a.dsum[d.dsum0 + b * d.ncc + q];
      const double sb = block_sum(s, red);
      if (threadIdx.x == 0) tot += a.mean[d.slice0 + b] * sb;
    }
  } else {
    double s = 0.0;
    for (int64_t k = threadIdx.x; k < d.nsp; k += kThreads) s += a.uspart[d.sp0 + k];
    tot = block_sum(s, red);
  }
  if (threadIdx.x == 0) {
    const double r = d.n > 0 ? sqrt(tot / static_cast<double>(d.n)) / static_cast<double>(a.clip) : 0.0;
    a.coef[blockIdx.x] = 1.0 / (r > 1.0 ? r : 1.0);
  }
}

// ---- pass c: momentum and the instability sums (factored); the whole
// remaining step of 1D tensors ---------------------------------------------------
template <int VEC, int GK>
__device__ __forceinline__ void pass_c_tile(const CDev& d, const CArgs& a, int t, int64_t local, float* colbuf,
                                            float* colf) {
  constexpr int CH = Lay<VEC>::CH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Tile tl = tile_of(d, local);
  const int64_t base = tl.b * d.H * d.W;
  const float mr = static_cast<float>(a.mean[d.slice0 + tl.b]);
  const float coef = static_cast<float>(a.coef[t]);
  __syncthreads();  // colf of the previous tile is read
  for (int cl = threadIdx.x; cl < kTC; cl += kThreads) {
    const int64_t j = tl.j0 + cl;
    colf[cl] = j < d.W ? coef * rsqrtf(d.col[tl.b * d.W + j]) : 0.f;
  }
  __syncthreads();
  float cacc[CH * VEC];
#pragma unroll
  for (int k = 0; k < CH * VEC; ++k) cacc[k] = 0.f;
  float* rp = a.rowpart + d.rowpart + tl.c * (d.B * d.H) + tl.b * d.H;
  constexpr int CG = Lay<VEC>::CG;
  for (int64_t i = tl.i0 + warp; i < tl.i1; i += kWarps) {
    const float rf = rsqrtf(d.row[tl.b * d.H + i] / mr);
    float rs = 0.f;
#pragma unroll
    for (int kg = 0; kg < CH; kg += CG) {
      if (tl.j0 + Lay<VEC>::col(kg, 0) >= d.W) break;
      typename GSel<VEC, GK>::Raw raw[CG];
      float mv[CG][VEC];
#pragma unroll
      for (int k = 0; k < CG; ++k) {
        const int64_t j = tl.j0 + Lay<VEC>::col(kg + k, lane);
        if (j < d.W) {
          GSel<VEC, GK>::load(raw[k], d.g, d.gdt, base + i * d.W + j);
          load_f<VEC>(mv[k], d.m + base + i * d.W + j);
        }
      }
#pragma unroll
      for (int k = 0; k < CG; ++k) {
        const int cl = Lay<VEC>::col(kg + k, lane);
        if (tl.j0 + cl < d.W) {
          float x[VEC];
          GSel<VEC, GK>::unpack(raw[k], d.gdt, x);
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const float uh = (x[v] * rf) * colf[cl + v];
            const float dl = a.b1 * (uh - mv[k][v]);  // = uh - m_new, without rounding m_new first
            const float mn = fmaf(a.b1, mv[k][v], a.omb1 * uh);
            mv[k][v] = mn;
            const float q = dl * dl;
            cacc[(kg + k) * VEC + v] += q;
            rs += q;
          }
          store_f<VEC>(d.m + base + i * d.W + tl.j0 + cl, mv[k]);
        }
      }
    }
    rs = warp_sum(rs);
    if (lane == 0) rp[i] = rs;
  }
  store_col_sums<VEC>(d, a, tl, cacc, colbuf);
}

__device__ __forceinline__ void pass_c_1d(const CDev& d, const CArgs& a, int t, int64_t local) {
  const int64_t e0 = local * kUnit1D, e1 = min(d.n, e0 + kUnit1D);
  const float coef = static_cast<float>(a.coef[t]);
  for (int64_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
    GRaw<1> r;
    load_g(r, d.g, d.gdt, e);
    const float uh = (r.f * rsqrtf(d.v[e])) * coef;
    const float mo = d.m[e];
    const float dl = a.b1 * (uh - mo);  // = uh - m_new, without rounding m_new first
    const float mn = fmaf(a.b1, mo, a.omb1 * uh);
    d.m[e] = mn;
    const float sn = fmaf(a.b3, d.res[e], a.omb3 * (dl * dl + a.eps2));
    d.res[e] = sn;
    const float p = d.p[e];
    d.p[e] = fmaf(-a.wdl, p, p - a.lr * (mn * rsqrtf(sn)));
  }
}

template <int VEC, int GK>
__global__ void __launch_bounds__(kThreads, 2) k_came_pass_c(const __grid_constant__ CArgs a, int cls) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* colbuf = reinterpret_cast<float*>(smem);
  float* colf = colbuf + kWarps * kTC;
  walk(a, kListCD, cls, [&](const CDev& d, int t, int64_t local) {
    if (cls == k1D) pass_c_1d(d, a, t, local);
    else pass_c_tile<VEC, GK>(d, a, t, local, colbuf, colf);
  });
}

// ---- pass d: p <- p - wd lr p - lr m (R_i / mean R)^-1/2 C_j^-1/2 ------------
template <int VEC>
__device__ __forceinline__ void pass_d_tile(const CDev& d, const CArgs& a, int64_t local, float* cf) {
  constexpr int CH = Lay<VEC>::CH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Tile tl = tile_of(d, local);
  const int64_t base = tl.b * d.H * d.W;
  const float mR = static_cast<float>(a.mean[d.slice0 + tl.b]);
  __syncthreads();
  for (int cl = threadIdx.x; cl < kTC; cl += kThreads) {
    const int64_t j = tl.j0 + cl;
    cf[cl] = j < d.W ? a.lr * rsqrtf(d.rcol[tl.b * d.W + j]) : 0.f;
  }
  __syncthreads();
  constexpr int CG = Lay<VEC>::CG;
  for (int64_t i = tl.i0 + warp; i < tl.i1; i += kWarps) {
    const float rf = rsqrtf(d.rrow[tl.b * d.H + i] / mR);
#pragma unroll
    for (int kg = 0; kg < CH; kg += CG) {
      if (tl.j0 + Lay<VEC>::col(kg, 0) >= d.W) break;
      float mv[CG][VEC], pv[CG][VEC];
#pragma unroll
      for (int k = 0; k < CG; ++k) {
        const int64_t j = tl.j0 + Lay<VEC>::col(kg + k, lane);
        if (j < d.W) {
          load_f<VEC>(mv[k], d.m + base + i * d.W + j);
          load_f<VEC>(pv[k], d.p + base + i * d.W + j);
        }
      }
#pragma unroll
      for (int k = 0; k < CG; ++k) {
        const int cl = Lay<VEC>::col(kg + k, lane);
        if (tl.j0 + cl < d.W) {
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const float upd = (mv[k][v] * rf) * cf[cl + v];
            pv[k][v] = fmaf(-a.wdl, pv[k][v], pv[k][v] - upd);
          }
          store_f<VEC>(d.p + base + i * d.W + tl.j0 + cl, pv[k]);
        }
      }
    }
  }
}

template <int VEC>
__global__ void __launch_bounds__(kThreads, 2) k_came_pass_d(const __grid_constant__ CArgs a, int cls) {
  __shared__ __align__(16) float cf[kTC];
  walk(a, kListCD, cls, [&](const CDev& d, int, int64_t local) { pass_d_tile<VEC>(d, a, local, cf); });
}

// ---- host side ------------------------------------------------------------------
adaf_status fail(adaf_status st, const std::string& msg) { return meo::set_last_error(st, msg.c_str()); }
adaf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ADAF_ERR_CUDA, std::string("came: ") + what + ": " + cudaGetErrorString(e));
}
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr size_t kColbufBytes = sizeof(float) * kWarps * kTC;
constexpr size_t kPassASmem = kColbufBytes + sizeof(double) * kWarps;
constexpr size_t kPassCSmem = kColbufBytes + sizeof(float) * kTC;

// Row-panel configurations (warps, column groups of 256 per lane, ring
// stages, CTAs per SM; rows per chunk): the Adafactor step's two.
constexpr int kP1NW = 8, kP1G = 2, kP1S = 3, kP1MinB = 2, kP1Rows = 256;   // 2048 <= W <= 4096
constexpr int kP2NW = 14, kP2G = 4, kP2S = 3, kP2MinB = 1, kP2Rows = 128;  // 4096 < W <= 14336
template <int NW, int G, int S>
constexpr size_t panel_smem() {
  return meo::panel::Cfg<__nv_bfloat16, NW, G, S>::kBytes + sizeof(double) * (NW + 1);
}

// The plan of one call: descriptors, class lists, statistics items, offsets.
struct Plan {
  std::vector<CDev> dev;
  std::vector<int64_t> pf[2][kClasses];
  std::vector<int32_t> idx[2][kClasses];
  std::vector<int64_t> ppf[kPanelCfgs];
  std::vector<int32_t> pidx[kPanelCfgs];
  std::vector<int64_t> item_pf;
  std::vector<int32_t> item_idx;
  int64_t rowpart = 0, colpart = 0, usp = 0, slices = 0, rchunks = 0, pcol = 0, prchunks = 0, dsums = 0;
  size_t off_hdr = 0, hdr_bytes = 0, off_pf[2][kClasses] = {}, off_idx[2][kClasses] = {}, off_ipf = 0, off_iidx = 0;
  size_t off_ppf[kPanelCfgs] = {}, off_pidx[kPanelCfgs] = {};
  size_t off_rowpart = 0, off_colpart = 0, off_usp = 0, off_rchunk = 0, off_mean0 = 0, off_mean1 = 0, off_coef = 0;
  size_t off_pcol = 0, off_pdpart = 0, off_prchunk = 0, off_dsum = 0;
  size_t bytes = 0;
};

adaf_status make_plan(const came_tensor* tensors, const came_state* states, int32_t n, bool need_ptrs, Plan* P) {
  if (n < 0) return fail(ADAF_ERR_INVALID_ARGUMENT, "came: n < 0");
  if (n > 0 && tensors == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "came: tensors is NULL");
  if (need_ptrs && n > 0 && states == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "came: states is NULL");
  P->dev.resize(n);
  for (int l = 0; l < 2; ++l)
    for (int c = 0; c < kClasses; ++c) P->pf[l][c].assign(1, 0);
  for (int q = 0; q < kPanelCfgs; ++q) P->ppf[q].assign(1, 0);
  P->item_pf.assign(1, 0);
  for (int32_t t = 0; t < n; ++t) {
    const came_tensor& x = tensors[t];
    const std::string who = "came: tensor " + std::to_string(t);
    if (x.ndim < 0 || x.ndim > ADAF_MAX_NDIM) return fail(ADAF_ERR_INVALID_ARGUMENT, who + ": bad ndim");
    if (x.grad_dtype != ADAF_FLOAT32 && x.grad_dtype != ADAF_BFLOAT16)
      return fail(ADAF_ERR_INVALID_ARGUMENT, who + ": unknown grad_dtype");
    int64_t numel = 1;
    for (int32_t k = 0; k < x.ndim; ++k) {
      if (x.shape[k] < 0) return fail(ADAF_ERR_INVALID_ARGUMENT, who + ": negative dim");
      if (x.shape[k] > INT32_MAX) return fail(ADAF_ERR_UNSUPPORTED, who + ": a dim above 2^31");
      numel = x.shape[k] == 0 ? 0 : numel;
      if (numel > 0 && numel > (int64_t{1} << 40) / x.shape[k]) return fail(ADAF_ERR_UNSUPPORTED, who + ": more than 2^40 values");
      numel *= x.shape[k];
    }
    CDev d{};
    d.n = numel;
    d.gdt = x.grad_dtype;
    const bool fact = x.ndim >= 2;
    d.H = fact ? x.shape[x.ndim - 2] : 1;
    d.W = fact ? x.shape[x.ndim - 1] : numel;
    d.B = (fact && d.H > 0 && d.W > 0) ? numel / (d.H * d.W) : 1;
    if (need_ptrs && numel > 0) {
      const came_state& s = states[t];
      if (!x.p || !x.g || !s.exp_avg) return fail(ADAF_ERR_INVALID_ARGUMENT, who + ": NULL p, g or exp_avg");
      if (fact && (!s.exp_avg_sq_row || !s.exp_avg_sq_col || !s.exp_avg_res_row || !s.exp_avg_res_col))
        return fail(ADAF_ERR_INVALID_ARGUMENT, who + ": factored state pointer is NULL");
      if (!fact && (!s.exp_avg_sq || !s.exp_avg_res))
        return fail(ADAF_ERR_INVALID_ARGUMENT, who + ": exp_avg_sq / exp_avg_res is NULL");
      const size_t ge = x.grad_dtype == ADAF_BFLOAT16 ? 2 : 4;
      if (!aligned(x.p, 4) || !aligned(x.g, ge) || !aligned(s.exp_avg, 4))
        return fail(ADAF_ERR_INVALID_ARGUMENT, who + ": not element-aligned");
      d.p = x.p;
      d.g = x.g;
      d.m = s.exp_avg;
      d.row = s.exp_avg_sq_row;
      d.col = s.exp_avg_sq_col;
      d.rrow = s.exp_avg_res_row;
      d.rcol = s.exp_avg_res_col;
      d.v = s.exp_avg_sq;
      d.res = s.exp_avg_res;
    }
    int64_t ntiles = 0;
    if (numel == 0) {
      d.cls = k1D;
    } else if (fact) {
      const bool vec = d.W % 8 == 0 && (!need_ptrs || (aligned(d.p, 16) && aligned(d.g, 16) && aligned(d.m, 16)));
      d.cls = vec ? (x.grad_dtype == ADAF_BFLOAT16 ? kVecBF : kVecF) : kScalar;
      d.cb = cdiv(d.W, kTC);
      d.rb = cdiv(d.H, kTR);
      ntiles = d.B * d.rb * d.cb;
      d.rowpart = P->rowpart;
      P->rowpart += d.cb * d.B * d.H;
      d.colpart = P->colpart;
      P->colpart += d.rb * d.B * d.W;
      d.slice0 = P->slices;
      P->slices += d.B;
      d.nrc = cdiv(d.H, kRowItem);
      d.ncc = cdiv(d.W, kColItem);
      d.rc0 = P->rchunks;
      P->rchunks += d.B * d.nrc;
      P->item_idx.push_back(t);
      P->item_pf.push_back(P->item_pf.back() + d.B * (d.nrc + d.ncc));
      // bf16 matrices of 2048 <= W <= 14336 on the vector path take the
      // row-panel pass instead of passes a and b
      if (d.cls == kVecBF && d.W >= 2048 && d.W <= meo::kMaxWideW) {
        d.panel = d.W <= 4096 ? 1 : 2;
        d.pr = d.panel == 1 ? kP1Rows : kP2Rows;
        d.prb = cdiv(d.H, d.pr);
        d.pcol = P->pcol;
        P->pcol += d.B * d.prb * d.W;
        d.prc0 = P->prchunks;
        P->prchunks += d.B * d.prb;
        d.dsum0 = P->dsums;
        P->dsums += d.B * d.ncc;
        P->pidx[d.panel - 1].push_back(t);
        P->ppf[d.panel - 1].push_back(P->ppf[d.panel - 1].back() + d.B * d.prb);
      }
    } else {
      d.cls = k1D;
      ntiles = cdiv(numel, kUnit1D);
    }
    d.sp0 = P->usp;
    d.nsp = d.panel ? 0 : ntiles;  // panel tensors: sum(u^2) from the column items
    P->usp += d.nsp;
    if (ntiles > 0) {
      for (int l = 0; l < 2; ++l) {
        if (l == kListAB && d.panel) continue;
        P->idx[l][d.cls].push_back(t);
        P->pf[l][d.cls].push_back(P->pf[l][d.cls].back() + ntiles);
      }
    }
    P->dev[t] = d;
  }
  for (int c = 0; c < kClasses; ++c)
    if (P->pf[kListCD][c].back() > INT32_MAX) return fail(ADAF_ERR_UNSUPPORTED, "came: more than 2^31 tiles");
  if (P->item_pf.back() > INT32_MAX) return fail(ADAF_ERR_UNSUPPORTED, "came: more than 2^31 statistics items");
  // layout: header (descriptors, class lists, items), then the scratch arrays
  size_t o = 0;
  P->off_hdr = o;
  o += sizeof(CDev) * n;
  for (int l = 0; l < 2; ++l) {
    for (int c = 0; c < kClasses; ++c) {
      o = round_up(o, 8);
      P->off_pf[l][c] = o;
      o += sizeof(int64_t) * P->pf[l][c].size();
      P->off_idx[l][c] = o;
      o += sizeof(int32_t) * P->idx[l][c].size();
    }
  }
  for (int q = 0; q < kPanelCfgs; ++q) {
    o = round_up(o, 8);
    P->off_ppf[q] = o;
    o += sizeof(int64_t) * P->ppf[q].size();
    P->off_pidx[q] = o;
    o += sizeof(int32_t) * P->pidx[q].size();
  }
  o = round_up(o, 8);
  P->off_ipf = o;
  o += sizeof(int64_t) * P->item_pf.size();
  P->off_iidx = o;
  o += sizeof(int32_t) * P->item_idx.size();
  P->hdr_bytes = o - P->off_hdr;
  o = round_up(o, 256);
  P->off_rowpart = o; o = round_up(o + sizeof(float) * P->rowpart, 256);
  P->off_colpart = o; o = round_up(o + sizeof(float) * P->colpart, 256);
  P->off_usp = o;     o = round_up(o + sizeof(double) * P->usp, 256);
  P->off_rchunk = o;  o = round_up(o + sizeof(double) * P->rchunks, 256);
  P->off_mean0 = o;   o = round_up(o + sizeof(double) * P->slices, 256);
  P->off_mean1 = o;   o = round_up(o + sizeof(double) * P->slices, 256);
  P->off_coef = o;    o = round_up(o + sizeof(double) * n, 256);
  P->off_pcol = o;    o = round_up(o + sizeof(float) * P->pcol, 256);
  P->off_pdpart = o;  o = round_up(o + sizeof(float) * P->pcol, 256);
  P->off_prchunk = o; o = round_up(o + sizeof(double) * P->prchunks, 256);
  P->off_dsum = o;    o = round_up(o + sizeof(double) * P->dsums, 256);
  P->bytes = o;
  return ADAF_OK;
}

adaf_status check_hp(const came_hparams* hp) {
  if (hp == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "came: hparams is NULL");
  if (!std::isfinite(hp->lr) || hp->lr < 0.0) return fail(ADAF_ERR_INVALID_ARGUMENT, "came: invalid learning rate");
  if (!std::isfinite(hp->eps1) || hp->eps1 < 0.0 || !std::isfinite(hp->eps2) || hp->eps2 < 0.0)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "came: invalid eps");
  if (!std::isfinite(hp->clip_threshold) || hp->clip_threshold <= 0.0)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "came: invalid clip_threshold (needs > 0)");
  const double b[3] = {hp->beta1, hp->beta2, hp->beta3};
  for (int k = 0; k < 3; ++k)
    if (!std::isfinite(b[k]) || b[k] < 0.0 || b[k] >= 1.0)
      return fail(ADAF_ERR_INVALID_ARGUMENT, "came: invalid beta" + std::to_string(k + 1) + " (needs 0 <= beta < 1)");
  if (!std::isfinite(hp->weight_decay) || hp->weight_decay < 0.0)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "came: invalid weight_decay");
  return ADAF_OK;
}

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
  int sms = 0;
  std::vector<cudaEvent_t> free_events;
  meo::TableCache tables;  // device copies of the descriptor table (host_copy.cuh)
};

enum KernelSlot { kSA = 0, kSStats, kSMeans, kSB, kSClip, kSC, kSD, kSPanel, kNumKernels };
const char* const kKernelNames[kNumKernels] = {"k_came_pass_a", "k_came_stats",  "k_came_means",
                                               "k_came_pass_b", "k_came_clip",   "k_came_pass_c",
                                               "k_came_pass_d", "k_came_panel"};
struct ProfRecord {
  int slot, device;
  cudaEvent_t start, stop;
  int count;  // kernels launched between the two events
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

bool g_attr_done = false;
cudaError_t set_smem_attrs() {
  if (g_attr_done) return cudaSuccess;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_came_pass_a<8, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassASmem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_came_pass_a<8, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassASmem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_came_pass_a<1, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassASmem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_came_pass_c<8, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassCSmem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_came_pass_c<8, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassCSmem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_came_pass_c<1, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassCSmem)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_came_panel<kP1NW, kP1G, kP1S, kP1MinB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(panel_smem<kP1NW, kP1G, kP1S>()))) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_came_panel<kP2NW, kP2G, kP2S, kP2MinB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(panel_smem<kP2NW, kP2G, kP2S>()))) != cudaSuccess) return e;
  g_attr_done = true;
  return cudaSuccess;
}

}  // namespace

extern "C" {

void came_default_hparams(came_hparams* hp) {
  if (hp == nullptr) return;
  hp->lr = 0.0;
  hp->eps1 = 1e-30;
  hp->eps2 = 1e-16;
  hp->clip_threshold = 1.0;
  hp->beta1 = 0.9;
  hp->beta2 = 0.999;
  hp->beta3 = 0.9999;
  hp->weight_decay = 0.0;
}

adaf_status came_validate(const came_hparams* hp) { return check_hp(hp); }

adaf_status came_workspace_size(const came_tensor* tensors, int32_t n, size_t* bytes) {
  if (bytes == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "came: bytes is NULL");
  Plan P;
  adaf_status st = make_plan(tensors, nullptr, n, false, &P);
  if (st != ADAF_OK) return st;
  *bytes = n == 0 ? 0 : P.bytes;
  return ADAF_OK;
}

adaf_status came_step(const came_tensor* tensors, const came_state* states, int32_t n, int64_t step,
                      const came_hparams* hp, void* workspace, size_t workspace_bytes, void* stream) {
  adaf_status st = check_hp(hp);
  if (st != ADAF_OK) return st;
  if (step < 1) return fail(ADAF_ERR_INVALID_ARGUMENT, "came: step must be >= 1");
  Plan P;
  st = make_plan(tensors, states, n, true, &P);
  if (st != ADAF_OK) return st;
  if (n == 0) return ADAF_OK;
  if (workspace == nullptr || !aligned(workspace, 256))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "came: workspace is NULL or not 256-byte aligned");
  if (workspace_bytes < P.bytes)
    return fail(ADAF_ERR_WORKSPACE_TOO_SMALL, "came: workspace needs " + std::to_string(P.bytes) + " bytes");

  std::vector<unsigned char> h(P.hdr_bytes);
  std::memcpy(h.data(), P.dev.data(), sizeof(CDev) * n);
  for (int l = 0; l < 2; ++l) {
    for (int c = 0; c < kClasses; ++c) {
      std::memcpy(h.data() + P.off_pf[l][c], P.pf[l][c].data(), sizeof(int64_t) * P.pf[l][c].size());
      if (!P.idx[l][c].empty())
        std::memcpy(h.data() + P.off_idx[l][c], P.idx[l][c].data(), sizeof(int32_t) * P.idx[l][c].size());
    }
  }
  for (int q = 0; q < kPanelCfgs; ++q) {
    std::memcpy(h.data() + P.off_ppf[q], P.ppf[q].data(), sizeof(int64_t) * P.ppf[q].size());
    if (!P.pidx[q].empty())
      std::memcpy(h.data() + P.off_pidx[q], P.pidx[q].data(), sizeof(int32_t) * P.pidx[q].size());
  }
  std::memcpy(h.data() + P.off_ipf, P.item_pf.data(), sizeof(int64_t) * P.item_pf.size());
  if (!P.item_idx.empty()) std::memcpy(h.data() + P.off_iidx, P.item_idx.data(), sizeof(int32_t) * P.item_idx.size());

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  CArgs a{};
  a.dev = reinterpret_cast<const CDev*>(ws + P.off_hdr);
  for (int l = 0; l < 2; ++l) {
    for (int c = 0; c < kClasses; ++c) {
      a.pf[l][c] = reinterpret_cast<const int64_t*>(ws + P.off_pf[l][c]);
      a.idx[l][c] = reinterpret_cast<const int32_t*>(ws + P.off_idx[l][c]);
      a.nmem[l][c] = static_cast<int32_t>(P.idx[l][c].size());
    }
  }
  for (int q = 0; q < kPanelCfgs; ++q) {
    a.ppf[q] = reinterpret_cast<const int64_t*>(ws + P.off_ppf[q]);
    a.pidx[q] = reinterpret_cast<const int32_t*>(ws + P.off_pidx[q]);
    a.pnmem[q] = static_cast<int32_t>(P.pidx[q].size());
  }
  a.pcolpart = reinterpret_cast<float*>(ws + P.off_pcol);
  a.pdpart = reinterpret_cast<float*>(ws + P.off_pdpart);
  a.prchunk = reinterpret_cast<double*>(ws + P.off_prchunk);
  a.dsum = reinterpret_cast<double*>(ws + P.off_dsum);
  a.item_pf = reinterpret_cast<const int64_t*>(ws + P.off_ipf);
  a.item_idx = reinterpret_cast<const int32_t*>(ws + P.off_iidx);
  a.nfact = static_cast<int32_t>(P.item_idx.size());
  a.rowpart = reinterpret_cast<float*>(ws + P.off_rowpart);
  a.colpart = reinterpret_cast<float*>(ws + P.off_colpart);
  a.uspart = reinterpret_cast<double*>(ws + P.off_usp);
  a.rchunk = reinterpret_cast<double*>(ws + P.off_rchunk);
  a.coef = reinterpret_cast<double*>(ws + P.off_coef);
  a.n = n;
  a.b1 = static_cast<float>(hp->beta1);
  a.omb1 = static_cast<float>(1.0 - hp->beta1);
  a.b2 = static_cast<float>(hp->beta2);
  a.omb2 = static_cast<float>(1.0 - hp->beta2);
  a.b3 = static_cast<float>(hp->beta3);
  a.omb3 = static_cast<float>(1.0 - hp->beta3);
  a.eps1 = static_cast<float>(hp->eps1);
  a.eps2 = static_cast<float>(hp->eps2);
  a.lr = static_cast<float>(hp->lr);
  a.wdl = static_cast<float>(hp->weight_decay * hp->lr);
  a.clip = static_cast<float>(hp->clip_threshold);
  double* mean0 = reinterpret_cast<double*>(ws + P.off_mean0);
  double* mean1 = reinterpret_cast<double*>(ws + P.off_mean1);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if ((err = set_smem_attrs()) != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute");
  DeviceState& ds = g_dev[device];
  if (ds.sms == 0 && (err = cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
    return cuda_fail(err, "cudaDeviceGetAttribute");
  // The descriptor table comes from a kept device copy when one holds the
  // same bytes (TableCache); otherwise it is staged in a pinned ring slot and
  // a kernel reads it from host memory (no copy engine, host_copy.cuh).
  auto upload = [&](unsigned char* dst) -> cudaError_t {
    Slot& sl = ds.ring[ds.next];
    ds.next = (ds.next + 1) % kRing;
    cudaError_t e = cudaSuccess;
    if (sl.used && (e = cudaEventSynchronize(sl.done)) != cudaSuccess) return e;
    const size_t up = round_up(P.hdr_bytes, 16);  // the upload moves whole 16-byte words
    if (sl.cap < up) {
      if (sl.host) cudaFreeHost(sl.host);
      sl.host = nullptr;
      sl.cap = 0;
      if ((e = cudaHostAlloc(&sl.host, up, cudaHostAllocPortable | cudaHostAllocMapped)) != cudaSuccess) return e;
      sl.cap = up;
    }
    if (sl.done == nullptr && (e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming)) != cudaSuccess)
      return e;
    std::memcpy(sl.host, h.data(), P.hdr_bytes);
    if ((e = meo::copy_from_host(dst, sl.host, up, s)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(sl.done, s)) != cudaSuccess) return e;
    sl.used = true;
    return cudaSuccess;
  };
  unsigned char* tab = nullptr;
  meo::RecordOnExit used_guard;
  if ((err = ds.tables.lookup(h.data(), P.hdr_bytes, s, upload, &tab, &used_guard.ev)) != cudaSuccess)
    return cuda_fail(err, "descriptor table upload");
  used_guard.s = s;
  // the table's arrays at their offsets within the kept copy
  auto at = [&](size_t off) { return tab + (off - P.off_hdr); };
  a.dev = reinterpret_cast<const CDev*>(at(P.off_hdr));
  for (int l = 0; l < 2; ++l) {
    for (int c = 0; c < kClasses; ++c) {
      a.pf[l][c] = reinterpret_cast<const int64_t*>(at(P.off_pf[l][c]));
      a.idx[l][c] = reinterpret_cast<const int32_t*>(at(P.off_idx[l][c]));
    }
  }
  for (int q = 0; q < kPanelCfgs; ++q) {
    a.ppf[q] = reinterpret_cast<const int64_t*>(at(P.off_ppf[q]));
    a.pidx[q] = reinterpret_cast<const int32_t*>(at(P.off_pidx[q]));
  }
  a.item_pf = reinterpret_cast<const int64_t*>(at(P.off_ipf));
  a.item_idx = reinterpret_cast<const int32_t*>(at(P.off_iidx));

  const int persist = 2 * ds.sms;  // 2 CTAs of 256 threads per SM
  auto grid_for = [&](int64_t units) { return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(persist, units))); };
  int64_t tiles[2][kClasses];
  for (int l = 0; l < 2; ++l)
    for (int c = 0; c < kClasses; ++c) tiles[l][c] = P.pf[l][c].back();
  const int64_t chunks[kPanelCfgs] = {P.ppf[0].back(), P.ppf[1].back()};
  const int64_t items = P.item_pf.back();

  // launch helper: profiling events around each launch
  int nk = 0;  // kernels launched so far by this call (a slot may launch one per class)
  auto launch = [&](int slot, auto&& fn) -> adaf_status {
    ProfRecord rec{slot, device, nullptr, nullptr, 0};
    cudaError_t e;
    if (g_profile) {
      if ((e = get_event(ds, &rec.start)) != cudaSuccess) return cuda_fail(e, "cudaEventCreate (profile)");
      if ((e = get_event(ds, &rec.stop)) != cudaSuccess) return cuda_fail(e, "cudaEventCreate (profile)");
      if ((e = cudaEventRecord(rec.start, s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord (profile)");
    }
    const int before = nk;
    fn();
    rec.count = nk - before;
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, kKernelNames[slot]);
    if (g_profile) {
      if ((e = cudaEventRecord(rec.stop, s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord (profile)");
      g_prof.push_back(rec);
    }
    return ADAF_OK;
  };
#define CAME_TRY(x)                 \
  do {                              \
    adaf_status st_ = (x);          \
    if (st_ != ADAF_OK) return st_; \
  } while (0)

  // row-panel pass of the bf16 matrices, pass a of the rest (and the 1D
  // second moment + sum(u^2))
  const int64_t* ta = tiles[kListAB];
  if (chunks[0] || chunks[1]) {
    CAME_TRY(launch(kSPanel, [&] {
      if (chunks[0]) {
        k_came_panel<kP1NW, kP1G, kP1S, kP1MinB><<<static_cast<int>(std::min<int64_t>(kP1MinB * ds.sms, chunks[0])),
                                                   kP1NW * 32, panel_smem<kP1NW, kP1G, kP1S>(), s>>>(a, 0);
        ++nk;
      }
      if (chunks[1]) {
        k_came_panel<kP2NW, kP2G, kP2S, kP2MinB><<<static_cast<int>(std::min<int64_t>(kP2MinB * ds.sms, chunks[1])),
                                                   kP2NW * 32, panel_smem<kP2NW, kP2G, kP2S>(), s>>>(a, 1);
        ++nk;
      }
    }));
  }
  if (ta[kVecBF] || ta[kVecF] || ta[kScalar] || ta[k1D]) {
    CAME_TRY(launch(kSA, [&] {
      if (ta[kVecBF]) { k_came_pass_a<8, 1><<<grid_for(ta[kVecBF]), kThreads, kPassASmem, s>>>(a, kVecBF); ++nk; }
      if (ta[kVecF]) { k_came_pass_a<8, 0><<<grid_for(ta[kVecF]), kThreads, kPassASmem, s>>>(a, kVecF); ++nk; }
      if (ta[kScalar]) { k_came_pass_a<1, 0><<<grid_for(ta[kScalar]), kThreads, kPassASmem, s>>>(a, kScalar); ++nk; }
      if (ta[k1D]) { k_came_pass_a<1, 0><<<grid_for(ta[k1D]), kThreads, kPassASmem, s>>>(a, k1D); ++nk; }
    }));
  }
  if (items) {
    a.phase = 0;
    a.mean = mean0;
    CAME_TRY(launch(kSStats, [&] { k_came_stats<<<grid_for(items), kThreads, 0, s>>>(a); ++nk; }));
    CAME_TRY(launch(kSMeans, [&] { k_came_means<<<a.nfact, kThreads, 0, s>>>(a); ++nk; }));
    if (ta[kVecBF] || ta[kVecF] || ta[kScalar]) {
      CAME_TRY(launch(kSB, [&] {
        if (ta[kVecBF]) { k_came_pass_b<8, 1><<<grid_for(ta[kVecBF]), kThreads, 0, s>>>(a, kVecBF); ++nk; }
        if (ta[kVecF]) { k_came_pass_b<8, 0><<<grid_for(ta[kVecF]), kThreads, 0, s>>>(a, kVecF); ++nk; }
        if (ta[kScalar]) { k_came_pass_b<1, 0><<<grid_for(ta[kScalar]), kThreads, 0, s>>>(a, kScalar); ++nk; }
      }));
    }
  }
  CAME_TRY(launch(kSClip, [&] { k_came_clip<<<n, kThreads, 0, s>>>(a); ++nk; }));
  const int64_t* tc = tiles[kListCD];
  CAME_TRY(launch(kSC, [&] {
    if (tc[kVecBF]) { k_came_pass_c<8, 1><<<grid_for(tc[kVecBF]), kThreads, kPassCSmem, s>>>(a, kVecBF); ++nk; }
    if (tc[kVecF]) { k_came_pass_c<8, 0><<<grid_for(tc[kVecF]), kThreads, kPassCSmem, s>>>(a, kVecF); ++nk; }
    if (tc[kScalar]) { k_came_pass_c<1, 0><<<grid_for(tc[kScalar]), kThreads, kPassCSmem, s>>>(a, kScalar); ++nk; }
    if (tc[k1D]) { k_came_pass_c<1, 0><<<grid_for(tc[k1D]), kThreads, kPassCSmem, s>>>(a, k1D); ++nk; }
  }));
  if (items) {
    a.phase = 1;
    a.mean = mean1;
    CAME_TRY(launch(kSStats, [&] { k_came_stats<<<grid_for(items), kThreads, 0, s>>>(a); ++nk; }));
    CAME_TRY(launch(kSMeans, [&] { k_came_means<<<a.nfact, kThreads, 0, s>>>(a); ++nk; }));
    CAME_TRY(launch(kSD, [&] {
      if (tc[kVecBF]) { k_came_pass_d<8><<<grid_for(tc[kVecBF]), kThreads, 0, s>>>(a, kVecBF); ++nk; }
      if (tc[kVecF]) { k_came_pass_d<8><<<grid_for(tc[kVecF]), kThreads, 0, s>>>(a, kVecF); ++nk; }
      if (tc[kScalar]) { k_came_pass_d<1><<<grid_for(tc[kScalar]), kThreads, 0, s>>>(a, kScalar); ++nk; }
    }));
  }
#undef CAME_TRY
  return ADAF_OK;
}

adaf_status came_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profile = on != 0;
  return ADAF_OK;
}

adaf_status came_profile_read(double* ms, int64_t* launches, int32_t nk) {
  std::lock_guard<std::mutex> lock(g_mu);
  adaf_status st = ADAF_OK;
  for (ProfRecord& r : g_prof) {
    float el = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&el, r.start, r.stop);
    if (e != cudaSuccess && st == ADAF_OK) st = cuda_fail(e, "profile event");
    if (r.slot < nk) {
      if (ms) ms[r.slot] += el;
      if (launches) launches[r.slot] += r.count;
    }
    DeviceState& ds = g_dev[r.device];
    ds.free_events.push_back(r.start);
    ds.free_events.push_back(r.stop);
  }
  g_prof.clear();
  return st;
}

int32_t came_num_kernels(void) { return kNumKernels; }

const char* came_kernel_name(int32_t k) { return (k >= 0 && k < kNumKernels) ? kKernelNames[k] : ""; }

}  // extern "C"

namespace meo {
void came_forget_tables() {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  const bool have_dev = cudaGetDevice(&cur) == cudaSuccess;
  for (auto& kv : g_dev) {
    if (cudaSetDevice(kv.first) == cudaSuccess) kv.second.tables.clear();
  }
  if (have_dev) cudaSetDevice(cur);
}
}  // namespace meo

