// Kernels of the GB300 Adafactor step.
//
// The step is bandwidth bound (a handful of flops per byte, no contraction),
// so the kernels are built around streaming the gradient (twice for the
// row-chunk classes, whose pass 1 also forms sum(u^2); three times for the
// tiled classes) and the parameter once (read + write), with persistent grids
// sized to the SM count and deterministic two-stage reductions: per-unit
// partials written once, then summed in a fixed order (no float atomics, so
// two runs give bit-identical results).
//
// Launch sequence of one step (one launch per tensor class and kind):
//   pass1   g (and p when RMS(p) must be recomputed) -> row/col partial sums
//           of g^2 (row-chunk classes: the updated row statistic and the
//           column partials of g^2 / row_i as well); tensors with ndim < 2
//           update exp_avg_sq in place and emit partial sum(u^2).
//   stats   row/col partials -> EMA of row/col means (exp_avg_sq_row/col),
//           plus per-chunk sums of the new row vector.
//   scalars per tensor: alpha = rho * max(eps2, RMS(p)), mean(row) per slice,
//           sum(u^2) of the row-chunk classes.
//   pass2   tiled classes: g -> partial sum(u^2), u = g (row_i/m)^-1/2 col_j^-1/2.
//   clip    per tensor: coef = alpha / max(1, RMS(u) / clip_threshold).
//   apply   g, p (exp_avg, or its 8-bit codes and scales) -> p (exp_avg);
//           partial sum(p_new^2).
//   psq     per tensor: sum(p_new^2) -> the optional carry slot.
// The row-sharded step runs the same kernels in three calls (phases 1-3 in
// StepArgs::phase), with the sums over the shards made by the caller.
// Method: Colossal-AI distributed-optimizer article, Step 3 (factored rows/
// cols, relative step, beta1), Step 4 (RMS), Step 5 (beta2t, clip, lr scale).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "adafactor_internal.h"
#include "row_panel.cuh"

namespace meo {
namespace {

// ---- small helpers --------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Deterministic CTA-wide sum: xor-butterfly inside each warp, then warp 0's
// lane 0 adds the kWarps warp sums in index order.  Every thread gets the
// result.  red must hold kWarps + 1 doubles.
__device__ __forceinline__ double block_sum(double v, double* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[w];
    red[kWarps] = s;
  }
  __syncthreads();
  const double s = red[kWarps];
  __syncthreads();
  return s;
}

// Index of the tensor owning unit u: largest t with pf[t] <= u < pf[t+1].
__device__ __forceinline__ int find_owner(const int32_t* pf, int ng, int64_t u) {
  int lo = 0, hi = ng;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pf[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

// Raw (not yet widened) gradient registers for VEC elements.
template <typename GT, int VEC> struct Raw;
template <> struct Raw<__nv_bfloat16, 8> { uint4 u; };
template <> struct Raw<float, 8> { float4 a, b; };
template <> struct Raw<__nv_bfloat16, 1> { unsigned short h; };
template <> struct Raw<float, 1> { float f; };

__device__ __forceinline__ void load_raw(Raw<__nv_bfloat16, 8>& r, const __nv_bfloat16* p) {
  r.u = __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void load_raw(Raw<float, 8>& r, const float* p) {
  r.a = __ldcs(reinterpret_cast<const float4*>(p));
  r.b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
}
__device__ __forceinline__ void load_raw(Raw<__nv_bfloat16, 1>& r, const __nv_bfloat16* p) {
  r.h = __ldcs(reinterpret_cast<const unsigned short*>(p));
}
__device__ __forceinline__ void load_raw(Raw<float, 1>& r, const float* p) { r.f = __ldcs(p); }

// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits.
__device__ __forceinline__ void widen(const Raw<__nv_bfloat16, 8>& r, float (&x)[8]) {
  const uint32_t w[4] = {r.u.x, r.u.y, r.u.z, r.u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}
__device__ __forceinline__ void widen(const Raw<float, 8>& r, float (&x)[8]) {
  x[0] = r.a.x; x[1] = r.a.y; x[2] = r.a.z; x[3] = r.a.w;
  x[4] = r.b.x; x[5] = r.b.y; x[6] = r.b.z; x[7] = r.b.w;
}
__device__ __forceinline__ void widen(const Raw<__nv_bfloat16, 1>& r, float (&x)[1]) {
  x[0] = __uint_as_float(static_cast<uint32_t>(r.h) << 16);
}
__device__ __forceinline__ void widen(const Raw<float, 1>& r, float (&x)[1]) { x[0] = r.f; }

__device__ __forceinline__ float load_g1(const void* g, int gdt, int64_t e) {
  if (gdt == kGradBF16) {
    const unsigned short h = __ldcs(static_cast<const unsigned short*>(g) + e);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  return __ldcs(static_cast<const float*>(g) + e);
}

// fp32 vectors of VEC elements (params, exp_avg).
template <int VEC> __device__ __forceinline__ void load_f(float (&y)[VEC], const float* p);
template <> __device__ __forceinline__ void load_f<8>(float (&y)[8], const float* p) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w; y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
}
template <> __device__ __forceinline__ void load_f<1>(float (&y)[1], const float* p) { y[0] = __ldcs(p); }
template <int VEC> __device__ __forceinline__ void store_f(float* p, const float (&y)[VEC]);
template <> __device__ __forceinline__ void store_f<1>(float* p, const float (&y)[1]) { __stcs(p, y[0]); }

// Position of tile `local` of a factored tensor: column block fastest, so
// neighbouring CTAs read neighbouring pieces of the same rows.
struct TilePos {
  int64_t b, r, c;
};
// Unit indices and their divisors fit 32 bits (the planner's prefix arrays
// are int32), and a 32-bit unsigned division is a short integer sequence,
// where a 64-bit one goes through the FP64 pipe, which is slow on this part.
__device__ __forceinline__ void udivmod32(int64_t n, int64_t d, int64_t& q, int64_t& r) {
  const uint32_t nn = static_cast<uint32_t>(n), dd = static_cast<uint32_t>(d);
  const uint32_t qq = nn / dd;
  q = qq;
  r = nn - qq * dd;
}
__device__ __forceinline__ TilePos tile_pos(const DevTensor& d, int64_t local) {
  TilePos t;
  int64_t q;
  udivmod32(local, d.cb, q, t.c);
  udivmod32(q, d.rb, t.b, t.r);
  return t;
}

// ---- per-tile column factors in shared memory -----------------------------
// On the vector path lane l reads the 8 factors of its columns k*256 + l*8 + v
// as two float4 loads; storing element v of lane l at
// k*256 + (v/4)*128 + l*4 + v%4 makes both loads conflict-free (consecutive
// lanes read consecutive 16-byte words).  The element-wise path needs no
// swizzle (lane l reads column k*32 + l).
template <int VEC> __device__ __forceinline__ int colf_index(int cl) {
  if (VEC == 1) return cl;
  const int k = cl >> 8, l = (cl >> 3) & 31, v = cl & 7;
  return (k << 8) + ((v >> 2) << 7) + (l << 2) + (v & 3);
}

template <int VEC> __device__ __forceinline__ void load_colf(float (&f)[VEC], const float* colf, int k, int lane);
template <> __device__ __forceinline__ void load_colf<8>(float (&f)[8], const float* colf, int k, int lane) {
  const float4 a = *reinterpret_cast<const float4*>(colf + (k << 8) + (lane << 2));
  const float4 b = *reinterpret_cast<const float4*>(colf + (k << 8) + 128 + (lane << 2));
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <> __device__ __forceinline__ void load_colf<1>(float (&f)[1], const float* colf, int k, int lane) {
  f[0] = colf[(k << 5) + lane];
}

// ---- pass 1: row / column partial sums of g^2 -----------------------------
// Lane column layout inside a tile: chunk k, element v -> k*32*VEC + lane*VEC + v.
// A row is streamed in groups of CG chunks; RPI rows are loaded per iteration
// so that ~128 bytes of gradient per lane are in flight before any use.
// ---- flat processing of narrow tiles (element-wise path, W <= kTileCols) ---
// Such a tile holds whole rows [i0, i1) and is one contiguous range of
// (i1 - i0) * W values; threads stream it by flat index (coalesced whatever
// W is) and recover (row, column) with row = (int)((e + 0.5f) * (1.0f / W)).
// In fp32 that is exact for every W <= 1024 and e < 256 * W (checked
// exhaustively): the fractional part of (e + 0.5) / W is at least 0.5 / W,
// far above the rounding error of the product.
// Where the tile's start is aligned, threads move 4 consecutive values per
// load (16 bytes of fp32, 8 of bf16) and step (row, column) along them.
constexpr int kFlatPass2 = 16;  // scalar values per thread in flight, pass 2
constexpr int kFlatApply = 8;   // scalar values per thread in flight, apply
constexpr int kFlatVec1 = kWarps * kTileCols / 4 / kThreads;  // 4-value loads per thread, pass-1 chunk
constexpr int kFlatVec2 = 8;    // 4-value loads per thread in flight, pass 2
constexpr int kFlatVecA = 4;    // 4-value loads per stream and thread in flight, apply (3 with exp_avg)
__device__ __forceinline__ int flat_row(int e, float invw) {
  return static_cast<int>(__fmul_rn(__fadd_rn(static_cast<float>(e), 0.5f), invw));
}
template <typename GT> __device__ __forceinline__ float load_g_scalar(const GT* p);
template <> __device__ __forceinline__ float load_g_scalar<float>(const float* p) { return __ldcs(p); }
template <> __device__ __forceinline__ float load_g_scalar<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldcs(reinterpret_cast<const unsigned short*>(p))) << 16);
}

template <typename GT> struct Raw4;
template <> struct Raw4<float> { float4 v; };
template <> struct Raw4<__nv_bfloat16> { uint2 v; };
__device__ __forceinline__ void load_raw4(Raw4<float>& r, const float* p) {
  r.v = __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void load_raw4(Raw4<__nv_bfloat16>& r, const __nv_bfloat16* p) {
  r.v = __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ void widen4(const Raw4<float>& r, float (&x)[4]) {
  x[0] = r.v.x; x[1] = r.v.y; x[2] = r.v.z; x[3] = r.v.w;
}
__device__ __forceinline__ void widen4(const Raw4<__nv_bfloat16>& r, float (&x)[4]) {
  x[0] = __uint_as_float(r.v.x << 16); x[1] = __uint_as_float(r.v.x & 0xffff0000u);
  x[2] = __uint_as_float(r.v.y << 16); x[3] = __uint_as_float(r.v.y & 0xffff0000u);
}
template <typename GT> __device__ __forceinline__ bool vec4_aligned(const GT* p) {
  return (reinterpret_cast<uintptr_t>(p) & (4 * sizeof(GT) - 1)) == 0;
}
// Next (row, column) of a flat walk over rows of w values.
__device__ __forceinline__ void flat_next(int& i, int& j, int w) {
  if (++j == w) { j = 0; ++i; }
}

template <int VEC> struct Layout {
  static constexpr int CH = kTileCols / (32 * VEC);  // chunks per tile row
  static constexpr int CG = VEC == 8 ? 4 : 8;          // chunks per load group
};

// Flat pass 1 of a narrow tile: chunks of whole rows are squared into the
// shared staging area (the column-buffer space, kWarps * kTileCols floats),
// then summed twice in fixed orders: down each column by the thread that owns
// it, and along each row by a segment of L = min(32, next power of 2 >= w)
// lanes.  The next chunk's loads are in flight meanwhile.  Returns false, with
// nothing done, where the tile does not qualify (wide rows, unaligned start).
template <typename GT, bool PSQ>
__device__ __forceinline__ void flat_chunk_issue(Raw4<GT> (&raw)[kFlatVec1], float& tail, const GT* src,
                                                 const float* psrc, int cn, float& psq) {
  const int nv = cn >> 2;
#pragma unroll
  for (int k = 0; k < kFlatVec1; ++k) {
    const int v = threadIdx.x + k * kThreads;
    if (v < nv) load_raw4(raw[k], src + 4 * v);
  }
  const int te = (nv << 2) + threadIdx.x;  // at most 3 values past the last whole load
  if (te < cn) tail = load_g_scalar<GT>(src + te);
  if (PSQ) {
#pragma unroll
    for (int k = 0; k < kFlatVec1; ++k) {
      const int v = threadIdx.x + k * kThreads;
      if (v < nv) {
        const float4 y = __ldcs(reinterpret_cast<const float4*>(psrc + 4 * v));
        psq = fmaf(y.x, y.x, psq); psq = fmaf(y.y, y.y, psq);
        psq = fmaf(y.z, y.z, psq); psq = fmaf(y.w, y.w, psq);
      }
    }
    if (te < cn) {
      const float y = __ldcs(psrc + te);
      psq = fmaf(y, y, psq);
    }
  }
}

template <typename GT, bool PSQ>
__device__ __forceinline__ bool pass1_flat(const DevTensor& d, const StepArgs& a, int64_t local, float* stage,
                                           double* red) {
  constexpr int kStage = kWarps * kTileCols;
  const int64_t H = d.H, W = d.W;
  if (W > kTileCols) return false;
  const TilePos tp = tile_pos(d, local);  // tp.c == 0: one column block
  const int64_t i0 = tp.r * kTileRows;
  const GT* gt = static_cast<const GT*>(d.g) + tp.b * H * W + i0 * W;
  const float* pt = d.p + tp.b * H * W + i0 * W;
  if (!vec4_aligned(gt) || (PSQ && !vec4_aligned(pt))) return false;
  const int w = static_cast<int>(W);
  const int nr = static_cast<int>(min(H, i0 + kTileRows) - i0);
  const int R = min(nr, (kStage / w) & ~3);  // rows per chunk: chunk starts stay on 4-value boundaries
  int lg = 0;
  while ((1 << lg) < w && lg < 5) ++lg;  // L = 1 << lg lanes per row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane >> lg, cl0 = lane & ((1 << lg) - 1);
  const int rpw = 32 >> lg;  // rows per warp pass
  float* rowpart = a.rowpart + d.rowpart + tp.b * H + i0;

  float cacc[kTileCols / kThreads];
#pragma unroll
  for (int k = 0; k < kTileCols / kThreads; ++k) cacc[k] = 0.f;
  float psq = 0.f, tail = 0.f;
  Raw4<GT> raw[kFlatVec1];
  flat_chunk_issue<GT, PSQ>(raw, tail, gt, pt, R * w, psq);
  for (int r0 = 0; r0 < nr; r0 += R) {
    const int rows = min(R, nr - r0);
    const int cn = rows * w, nv = cn >> 2;
#pragma unroll
    for (int k = 0; k < kFlatVec1; ++k) {
      const int v = threadIdx.x + k * kThreads;
      if (v < nv) {
        float x[4];
        widen4(raw[k], x);
        *reinterpret_cast<float4*>(stage + 4 * v) = make_float4(x[0] * x[0], x[1] * x[1], x[2] * x[2], x[3] * x[3]);
      }
    }
    const int te = (nv << 2) + threadIdx.x;
    if (te < cn) stage[te] = tail * tail;
    __syncthreads();
    const int r1 = r0 + R;
    if (r1 < nr) flat_chunk_issue<GT, PSQ>(raw, tail, gt + r1 * w, pt + r1 * w, min(R, nr - r1) * w, psq);
    // columns: thread c sums rows in order, four interleaved partials
#pragma unroll
    for (int k = 0; k < kTileCols / kThreads; ++k) {
      const int c = threadIdx.x + k * kThreads;
      if (c < w) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int r = 0;
        for (; r + 4 <= rows; r += 4) {
          s0 += stage[r * w + c];
          s1 += stage[(r + 1) * w + c];
          s2 += stage[(r + 2) * w + c];
          s3 += stage[(r + 3) * w + c];
        }
        for (; r < rows; ++r) s0 += stage[r * w + c];
        cacc[k] += (s0 + s1) + (s2 + s3);
      }
    }
    // rows: segments of L lanes, a xor tree inside each segment
    for (int rb = warp * rpw; rb < rows; rb += kWarps * rpw) {
      const int r = rb + sub;
      float sr = 0.f;
      if (r < rows)
        for (int c = cl0; c < w; c += 1 << lg) sr += stage[r * w + c];
      for (int o = (1 << lg) >> 1; o > 0; o >>= 1) sr += __shfl_xor_sync(0xffffffffu, sr, o);
      if (cl0 == 0 && r < rows) rowpart[r0 + r] = sr;
    }
    __syncthreads();  // the stage is rewritten next
  }
  float* colpart = a.colpart + d.colpart + (tp.b * d.rb + tp.r) * W;
#pragma unroll
  for (int k = 0; k < kTileCols / kThreads; ++k) {
    const int c = threadIdx.x + k * kThreads;
    if (c < w) colpart[c] = cacc[k];
  }
  if (PSQ) {
    const double tot = block_sum(static_cast<double>(psq), red);
    if (threadIdx.x == 0) a.ppart[d.p1_0 + local] = tot;
  }
  return true;
}

template <typename GT, int VEC, bool PSQ>
__device__ __forceinline__ void pass1_factored(const DevTensor& d, const StepArgs& a, int64_t local,
                               float* colbuf, double* red) {
  constexpr int CH = Layout<VEC>::CH, CG = Layout<VEC>::CG;
  constexpr int RPI = PSQ ? 1 : ((VEC == 8 && sizeof(GT) == 4) ? 1 : 2);
  if constexpr (VEC == 1) {
    if (pass1_flat<GT, PSQ>(d, a, local, colbuf, red)) return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const TilePos tp = tile_pos(d, local);
  const int64_t H = d.H, W = d.W;
  const int64_t i0 = tp.r * kTileRows;
  const int64_t i1 = min(H, i0 + kTileRows);
  const int64_t j0 = tp.c * kTileCols;
  const GT* gb = static_cast<const GT*>(d.g) + tp.b * H * W;
  const float* pb = d.p + tp.b * H * W;
  float* rowpart = a.rowpart + d.rowpart + tp.c * (int64_t)d.B * H + tp.b * H;

  float cacc[CH * VEC];
#pragma unroll
  for (int k = 0; k < CH * VEC; ++k) cacc[k] = 0.f;
  float psq = 0.f;

  for (int64_t i = i0 + warp; i < i1; i += RPI * kWarps) {
    float rs[RPI];
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr) rs[rr] = 0.f;
#pragma unroll
    for (int kg = 0; kg < CH; kg += CG) {
      if (j0 + kg * 32 * VEC >= W) break;  // the rest of the tile is past the row's end (warp-uniform)
      Raw<GT, VEC> raw[RPI][CG];
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr) {
        const int64_t ii = i + rr * kWarps;
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int64_t j = j0 + (kg + k) * 32 * VEC + lane * VEC;
          if (ii < i1 && j < W) load_raw(raw[rr][k], gb + ii * W + j);
        }
      }
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr) {
        const int64_t ii = i + rr * kWarps;
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int64_t j = j0 + (kg + k) * 32 * VEC + lane * VEC;
          if (ii < i1 && j < W) {
            float x[VEC];
            widen(raw[rr][k], x);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
              const float q = x[v] * x[v];
              cacc[(kg + k) * VEC + v] += q;
              rs[rr] += q;
            }
            if (PSQ) {
              float y[VEC];
              load_f<VEC>(y, pb + ii * W + j);
#pragma unroll
              for (int v = 0; v < VEC; ++v) psq = fmaf(y[v], y[v], psq);
            }
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr) {
      const int64_t ii = i + rr * kWarps;
      const float s = warp_sum(rs[rr]);
      if (lane == 0 && ii < i1) rowpart[ii] = s;
    }
  }

  // Column partials: the kWarps warps of the CTA covered disjoint rows of the
  // same columns; add their accumulators in warp order through shared memory.
  float* mine = colbuf + warp * kTileCols;
  const int ncl = static_cast<int>(min(static_cast<int64_t>(kTileCols), W - j0));  // columns of this tile
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    if (k * 32 * VEC >= ncl) break;
#pragma unroll
    for (int v = 0; v < VEC; ++v) mine[k * 32 * VEC + lane * VEC + v] = cacc[k * VEC + v];
  }
  __syncthreads();
  float* colpart = a.colpart + d.colpart + (tp.b * d.rb + tp.r) * W;
  for (int cl = threadIdx.x; cl < ncl; cl += kThreads) {
    const int64_t j = j0 + cl;
    {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += colbuf[w * kTileCols + cl];
      colpart[j] = s;
    }
  }
  if (PSQ) {
    const double tot = block_sum(static_cast<double>(psq), red);
    if (threadIdx.x == 0) a.ppart[d.p1_0 + local] = tot;
  } else {
    __syncthreads();  // colbuf is reused by the next tile
  }
}

constexpr int kBatch1D = 8;  // elements per thread in flight in the 1D kernels

// Full second moment (ndim < 2): v <- beta2 v + (1 - beta2)(g^2 + eps1) in
// place, partial sum(g^2 / v) = sum(u^2), and sum(p^2) when needed.
template <bool PSQ>
__device__ __forceinline__ void pass1_unfactored(const DevTensor& d, const StepArgs& a, int64_t local, double* red) {
  const int64_t e0 = local * kTile1D;
  const int64_t e1 = min(d.n, e0 + kTile1D);
  const float b2 = static_cast<float>(a.beta2);
  const float omb2 = static_cast<float>(1.0 - a.beta2);
  const float eps1 = static_cast<float>(a.eps1);
  float s = 0.f, ps = 0.f;
  // kBatch1D elements per thread are loaded before any is used, so their
  // loads are in flight together; the sums still run in element order.
  for (int64_t e00 = e0 + threadIdx.x; e00 < e1; e00 += kBatch1D * kThreads) {
    float x[kBatch1D], v[kBatch1D], y[kBatch1D];
#pragma unroll
    for (int k = 0; k < kBatch1D; ++k) {
      const int64_t e = e00 + k * kThreads;
      x[k] = v[k] = y[k] = 0.f;
      if (e < e1) {
        x[k] = load_g1(d.g, d.gdt, e);
        v[k] = d.v[e];
        if (PSQ) y[k] = d.p[e];
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch1D; ++k) {
      const int64_t e = e00 + k * kThreads;
      if (e < e1) {
        const float vn = fmaf(b2, v[k], omb2 * fmaf(x[k], x[k], eps1));
        d.v[e] = vn;
        s += (x[k] * x[k]) / vn;
        if (PSQ) ps = fmaf(y[k], y[k], ps);
      }
    }
  }
  const double S = block_sum(static_cast<double>(s), red);
  double P = 0.0;
  if (PSQ) P = block_sum(static_cast<double>(ps), red);
  if (threadIdx.x == 0) {
    a.spart[d.tile0 + local] = S;
    if (PSQ) a.ppart[d.p1_0 + local] = P;
  }
}

// Shared-memory layout of the persistent kernels.
constexpr size_t kColbufBytes = sizeof(float) * kWarps * kTileCols;
constexpr size_t kRedBytes = sizeof(double) * 16;
constexpr size_t kPrefixBytes = (sizeof(int32_t) * (kMaxGroup + 1) + 15) / 16 * 16;
constexpr size_t kColfBytes = sizeof(float) * kTileCols;
constexpr size_t kPartBytes = sizeof(float) * 2 * kWarps * kColChunk;
constexpr size_t kRowfBytes = sizeof(float) * kTileRows;

// Copies the launch's member prefix into shared memory; returns the member count.
__device__ __forceinline__ int load_prefix(int32_t* pf, const Range& r) {
  const int ng = r.m_end - r.m_begin;
  for (int k = threadIdx.x; k <= ng; k += blockDim.x) pf[k] = r.pf[r.m_begin + k];
  __syncthreads();
  return ng;
}

// Tensor index of member m (identity when the range has no index list).
__device__ __forceinline__ int member_tensor(const Range& r, int m) {
  return r.idx ? r.idx[r.m_begin + m] : r.m_begin + m;
}

template <typename GT, int VEC, bool PSQ>
__global__ void __launch_bounds__(kThreads, 2) k_pass1_f(const __grid_constant__ StepArgs a, const Range r) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* colbuf = reinterpret_cast<float*>(smem);
  double* red = reinterpret_cast<double*>(smem + kColbufBytes);
  int32_t* pf = reinterpret_cast<int32_t*>(smem + kColbufBytes + kRedBytes);
  const int ng = load_prefix(pf, r);
  const int64_t u1 = pf[ng];
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor d = a.tensors[member_tensor(r, m)];
    pass1_factored<GT, VEC, PSQ>(d, a, u - pf[m], colbuf, red);
  }
}

template <bool PSQ>
__global__ void __launch_bounds__(kThreads) k_pass1_u(const __grid_constant__ StepArgs a, const Range r) {
  extern __shared__ __align__(16) unsigned char smem[];
  double* red = reinterpret_cast<double*>(smem);
  int32_t* pf = reinterpret_cast<int32_t*>(smem + kRedBytes);
  const int ng = load_prefix(pf, r);
  const int64_t u1 = pf[ng];
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor d = a.tensors[member_tensor(r, m)];
    pass1_unfactored<PSQ>(d, a, u - pf[m], red);
  }
}

// Compensated (Kahan) fp32 accumulation: s += x with the running error in c.
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = x - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// ---- stats: EMA of row / column means -------------------------------------
__device__ __forceinline__ void stats_row_item(const DevTensor& d, const StepArgs& a, int64_t b, int64_t q, double* red) {
  const int64_t H = d.H;
  const int64_t i0 = q * kRowChunk;
  const int64_t i1 = min(H, i0 + kRowChunk);
  const float* rp = a.rowpart + d.rowpart + b * H;
  const int64_t stride = static_cast<int64_t>(d.B) * H;
  float* row = d.row + b * H;
  const float w = static_cast<float>(d.W), eps1 = static_cast<float>(a.eps1);
  const float b2 = static_cast<float>(a.beta2), omb2 = static_cast<float>(1.0 - a.beta2);
  float acc = 0.f;  // at most kRowChunk / kThreads = 4 rows per thread
  for (int64_t i = i0 + threadIdx.x; i < i1; i += kThreads) {
    float s = 0.f, c = 0.f;  // fp32 with Kahan compensation (see stats_col_item)
    for (int k = 0; k < d.cb; ++k) kahan_add(s, c, rp[k * stride + i]);
    const float mean = s / w + eps1;
    const float nr = fmaf(b2, row[i], omb2 * mean);
    row[i] = nr;
    acc += nr;
  }
  const double tot = block_sum(static_cast<double>(acc), red);
  if (threadIdx.x == 0) a.rowchunk[d.rowchunk + b * d.nrc + q] = tot;
}


// Column item: kColChunk (256) columns of one slice.  Warp w adds the row
// blocks r = w, w + 8, w + 16, ... of the column partials in that order, with
// compensated (Kahan) fp32 sums; the 8 warp sums are then added in warp order
// in double.  Fixed order throughout, so the result is deterministic.  With
// W % 4 == 0 lane l owns the column quads 4l and 128 + 4l (16-byte loads) and
// a warp has kStatsRows rows of loads in flight; otherwise lane l owns
// columns l + 32m, m < 8 (scalar loads, two rows in flight).  For fused
// tensors the weighted partials D_j are reduced the same way and the chunk's
// sum_j D_j / col_j goes to dsum.
constexpr int kStatsRows = 4;

template <bool Q4>
__device__ __forceinline__ void stats_col_item(const DevTensor& d, const StepArgs& a, int64_t b, int64_t q,
                                               float* part, double* red) {
  constexpr int kPer = kColChunk / 32;
  constexpr int R = Q4 ? kStatsRows : 2;  // row blocks per warp and iteration
  const bool fused = is_fused(d.kind);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t W = d.W;
  const int64_t c0 = q * kColChunk;
  const float* cp = a.colpart + d.colpart + b * d.prb * W;
  const float* dp = a.dpart + d.dpart + b * d.prb * W;
  // The old column statistic, loaded now so that its latency overlaps the row loop.
  const int64_t jt = c0 + threadIdx.x;
  float* colp = d.col + b * W + jt;
  const float col_old = (threadIdx.x < kColChunk && jt < W) ? *colp : 0.f;
  // lane's column of slot m: quads (Q4) or strided singles
  auto col_of = [&](int m) -> int64_t {
    return Q4 ? c0 + (m >> 2) * 128 + 4 * lane + (m & 3) : c0 + lane + 32 * m;
  };
  float s[kPer], comp[kPer], ds[kPer], dcomp[kPer];
#pragma unroll
  for (int m = 0; m < kPer; ++m) s[m] = comp[m] = ds[m] = dcomp[m] = 0.f;
  for (int r0 = warp; r0 < d.prb; r0 += R * kWarps) {
    float x[R][kPer], y[R][kPer];
#pragma unroll
    for (int h = 0; h < R; ++h) {
      const int r = r0 + h * kWarps;
      const int64_t roff = static_cast<int64_t>(r) * W;
      if (Q4) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t j = col_of(4 * e);
          const bool ok = r < d.prb && j < W;
          const float4 cv = ok ? *reinterpret_cast<const float4*>(cp + roff + j) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 dv = (fused && ok) ? *reinterpret_cast<const float4*>(dp + roff + j)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
          x[h][4 * e] = cv.x; x[h][4 * e + 1] = cv.y; x[h][4 * e + 2] = cv.z; x[h][4 * e + 3] = cv.w;
          y[h][4 * e] = dv.x; y[h][4 * e + 1] = dv.y; y[h][4 * e + 2] = dv.z; y[h][4 * e + 3] = dv.w;
        }
      } else {
#pragma unroll
        for (int m = 0; m < kPer; ++m) {
          const int64_t j = col_of(m);
          const bool ok = r < d.prb && j < W;
          x[h][m] = ok ? cp[roff + j] : 0.f;
          y[h][m] = (fused && ok) ? dp[roff + j] : 0.f;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < R; ++h) {
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        kahan_add(s[m], comp[m], x[h][m]);
        if (fused) kahan_add(ds[m], dcomp[m], y[h][m]);
      }
    }
  }
  __syncthreads();  // part is free (previous item done reading it)
#pragma unroll
  for (int m = 0; m < kPer; ++m) {
    const int cl = static_cast<int>(col_of(m) - c0);
    part[warp * kColChunk + cl] = s[m];
    if (fused) part[(kWarps + warp) * kColChunk + cl] = ds[m];
  }
  __syncthreads();
  // Per-column arithmetic in fp32 (this GPU's FP64 rate is a small fraction
  // of its FP32 rate); the 8 warp sums are added with Kahan compensation.
  if (a.phase == 1) {
    // Row-sharded begin: this shard's column sums go to the exchange buffer
    // (and D_j to the workspace); the column statistic waits for the sum
    // over all shards.
    if (threadIdx.x < kColChunk && jt < W) {
      float tot = 0.f, tc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) kahan_add(tot, tc, part[w * kColChunk + threadIdx.x]);
      a.round1[d.x1c + b * W + jt] = static_cast<double>(tot);
      if (fused) {
        float dt = 0.f, dc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) kahan_add(dt, dc, part[(kWarps + w) * kColChunk + threadIdx.x]);
        a.dloc[d.dloc + b * W + jt] = dt;
      }
    }
    return;
  }
  float term = 0.f;
  if (threadIdx.x < kColChunk && jt < W) {
    float tot = 0.f, tc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) kahan_add(tot, tc, part[w * kColChunk + threadIdx.x]);
    const float mean = tot / static_cast<float>(d.hg) + static_cast<float>(a.eps1);
    const float cn = fmaf(static_cast<float>(a.beta2), col_old, static_cast<float>(1.0 - a.beta2) * mean);
    *colp = cn;
    if (fused) {
      float dt = 0.f, dc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) kahan_add(dt, dc, part[(kWarps + w) * kColChunk + threadIdx.x]);
      term = dt / cn;
    }
  }
  if (fused) {
    const double tot = block_sum(static_cast<double>(term), red);
    if (threadIdx.x == 0) a.dsum[d.dsum + b * d.ncc + q] = tot;
  }
}

__device__ __forceinline__ void stats_col_any(const DevTensor& d, const StepArgs& a, int64_t b, int64_t q,
                                              float* part, double* red) {
  if (d.W % 4 == 0) stats_col_item<true>(d, a, b, q, part, red);
  else stats_col_item<false>(d, a, b, q, part, red);
}

// Row-sharded middle: the column statistic from the column sums of g^2 over
// all shards (exchange round 1), and for fused tensors this shard's
// sum_j D_j / col_j over the chunk's columns.
__device__ __forceinline__ void stats_col_global(const DevTensor& d, const StepArgs& a, int64_t b, int64_t q,
                                                 double* red) {
  const bool fused = is_fused(d.kind);
  const int64_t W = d.W;
  const int64_t jt = q * kColChunk + threadIdx.x;
  float term = 0.f;
  if (threadIdx.x < kColChunk && jt < W) {
    float* colp = d.col + b * W + jt;
    const float tot = static_cast<float>(a.round1[d.x1c + b * W + jt]);
    const float mean = tot / static_cast<float>(d.hg) + static_cast<float>(a.eps1);
    const float cn = fmaf(static_cast<float>(a.beta2), *colp, static_cast<float>(1.0 - a.beta2) * mean);
    *colp = cn;
    if (fused) term = a.dloc[d.dloc + b * W + jt] / cn;
  }
  if (fused) {
    const double tot = block_sum(static_cast<double>(term), red);
    if (threadIdx.x == 0) a.dsum[d.dsum + b * d.ncc + q] = tot;
  }
}

__global__ void __launch_bounds__(kThreads) k_stats(const __grid_constant__ StepArgs a, const Range r) {
  extern __shared__ __align__(16) unsigned char smem[];
  double* red = reinterpret_cast<double*>(smem);
  int32_t* pf = reinterpret_cast<int32_t*>(smem + kRedBytes);
  float* part = reinterpret_cast<float*>(smem + kRedBytes + kPrefixBytes);
  const int ng = load_prefix(pf, r);
  const int64_t u1 = pf[ng];
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor d = a.tensors[member_tensor(r, m)];
    const int64_t local = u - pf[m];
    if (is_fused(d.kind)) {  // rows were updated by the fused pass 1
      int64_t b, k;
      udivmod32(local, d.ncc, b, k);
      if (a.phase == 2) stats_col_global(d, a, b, k, red);
      else stats_col_any(d, a, b, k, part, red);
      continue;
    }
    int64_t b, k;
    udivmod32(local, d.nrc + d.ncc, b, k);
    if (k < d.nrc) {
      if (a.phase != 2) stats_row_item(d, a, b, k, red);  // rows are local to a shard
    } else if (a.phase == 2) {
      stats_col_global(d, a, b, k - d.nrc, red);
    } else {
      stats_col_any(d, a, b, k - d.nrc, part, red);
    }
  }
}

// ---- scalars: alpha, mean(row), fused sum(u^2); one CTA per tensor ----------
__global__ void __launch_bounds__(kThreads) k_scalars(const __grid_constant__ StepArgs a) {
  __shared__ double red[16];
  const int t = blockIdx.x;
  const DevTensor d = a.tensors[t];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (a.phase == 1) {
    // Row-sharded begin: this shard's sum(p^2) and sum_i row_i per slice go
    // to the exchange buffer.
    if (a.scale_parameter) {
      double psq;
      if (a.psq_valid) {
        psq = *d.psq;
      } else {
        double acc = 0.0;
        for (int64_t k = threadIdx.x; k < d.p1_n; k += kThreads) acc += a.ppart[d.p1_0 + k];
        psq = block_sum(acc, red);
      }
      if (threadIdx.x == 0) a.round1[d.x1p] = psq;
    } else if (threadIdx.x == 0) {
      a.round1[d.x1p] = 0.0;
    }
    if (d.kind != kUnfactored) {
      for (int64_t b = warp; b < d.B; b += kWarps) {
        double sr = 0.0;
        for (int64_t q = lane; q < d.nrc; q += 32) sr += a.rowchunk[d.rowchunk + b * d.nrc + q];
        sr = warp_sum(sr);
        if (lane == 0) a.round1[d.x1r + b] = sr;
      }
    }
    return;
  }
  double alpha = a.rho;
  if (a.scale_parameter) {
    double psq;
    if (a.phase == 2) {
      psq = a.round1[d.x1p];  // sum over all shards
    } else if (a.psq_valid) {
      psq = *d.psq;
    } else {
      double acc = 0.0;
      for (int64_t k = threadIdx.x; k < d.p1_n; k += kThreads) acc += a.ppart[d.p1_0 + k];
      psq = block_sum(acc, red);
    }
    const double r = sqrt(psq / static_cast<double>(d.ng));
    alpha = a.rho * (r > a.eps2 ? r : a.eps2);
  }
  if (threadIdx.x == 0) a.alpha[t] = alpha;
  if (d.kind != kUnfactored) {
    // mean(row) per slice; for fused tensors also sum(u^2) =
    // sum_b mean(row_b) * sum_j D_bj / col_bj (slices in order within a warp,
    // then warps in order).
    const bool fused = is_fused(d.kind);
    double su = 0.0;
    for (int64_t b = warp; b < d.B; b += kWarps) {
      double s = 0.0;
      if (a.phase == 2) {
        s = a.round1[d.x1r + b];  // sum over all shards
      } else {
        for (int64_t q = lane; q < d.nrc; q += 32) s += a.rowchunk[d.rowchunk + b * d.nrc + q];
        s = warp_sum(s);
      }
      const double mb = s / static_cast<double>(d.hg);
      if (lane == 0) a.mrow[d.mslot + b] = mb;
      if (fused) {
        double ds = 0.0;
        for (int64_t q = lane; q < d.ncc; q += 32) ds += a.dsum[d.dsum + b * d.ncc + q];
        su += mb * warp_sum(ds);
      }
    }
    if (fused) {
      if (lane == 0) red[warp] = su;
      __syncthreads();
      if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < kWarps; ++w) tot += red[w];
        a.ssum[t] = tot;
      }
    }
  }
}

// ---- pass 2: partial sum(u^2) ---------------------------------------------
// sum_ij u_ij^2 = sum_i (m / row_i) * sum_j g_ij^2 / col_j, so a lane keeps one
// running fp32 dot product per row and folds it into a double with m/row_i.
// colf holds 1/col_j for the tile's columns (shared memory).
template <typename GT, int VEC>
__device__ __forceinline__ void pass2_factored(const DevTensor& d, const StepArgs& a, int64_t local, float* colf,
                               float* rowf, double* red) {
  constexpr int CH = Layout<VEC>::CH, CG = Layout<VEC>::CG;
  constexpr int RPI = (VEC == 8 && sizeof(GT) == 4) ? 1 : 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const TilePos tp = tile_pos(d, local);
  const int64_t H = d.H, W = d.W;
  const int64_t i0 = tp.r * kTileRows;
  const int64_t i1 = min(H, i0 + kTileRows);
  const int64_t j0 = tp.c * kTileCols;
  const GT* gb = static_cast<const GT*>(d.g) + tp.b * H * W;
  const float* row = d.row + tp.b * H;
  const float m = static_cast<float>(a.mrow[d.mslot + tp.b]);

  __syncthreads();  // previous tile's readers of colf / rowf are done
  for (int cl = threadIdx.x; cl < kTileCols; cl += kThreads) {
    const int64_t j = j0 + cl;
    colf[colf_index<VEC>(cl)] = (j < W) ? 1.0f / d.col[tp.b * W + j] : 0.f;
  }
  for (int rl = threadIdx.x; rl < kTileRows; rl += kThreads) {
    const int64_t i = i0 + rl;
    rowf[rl] = (i < i1) ? m / row[i] : 0.f;
  }
  __syncthreads();

  if constexpr (VEC == 1) {
    if (W <= kTileCols) {  // whole rows: stream the tile by flat index
      const int cnt = static_cast<int>((i1 - i0) * W);
      const GT* gt = gb + i0 * W;
      const float invw = 1.0f / static_cast<float>(W);
      const int w32 = static_cast<int>(W);
      float acc = 0.f;
      int start = 0;  // first value left to the scalar loop
      if (vec4_aligned(gt)) {
        const int nv = cnt >> 2;
        for (int v0 = threadIdx.x; v0 < nv; v0 += kFlatVec2 * kThreads) {
          Raw4<GT> raw[kFlatVec2];
#pragma unroll
          for (int k = 0; k < kFlatVec2; ++k) {
            const int v = v0 + k * kThreads;
            if (v < nv) load_raw4(raw[k], gt + 4 * v);
          }
#pragma unroll
          for (int k = 0; k < kFlatVec2; ++k) {
            const int v = v0 + k * kThreads;
            if (v < nv) {
              float x[4];
              widen4(raw[k], x);
              int i = flat_row(4 * v, invw), j = 4 * v - i * w32;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                acc = fmaf(rowf[i], (x[q] * x[q]) * colf[j], acc);
                flat_next(i, j, w32);
              }
            }
          }
        }
        start = nv << 2;
      }
      for (int e0 = start + threadIdx.x; e0 < cnt; e0 += kFlatPass2 * kThreads) {
        float x[kFlatPass2];
#pragma unroll
        for (int k = 0; k < kFlatPass2; ++k) {
          const int e = e0 + k * kThreads;
          x[k] = e < cnt ? load_g_scalar<GT>(gt + e) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kFlatPass2; ++k) {
          const int e = e0 + k * kThreads;
          if (e < cnt) {
            const int i = flat_row(e, invw), j = e - i * w32;
            acc = fmaf(rowf[i], (x[k] * x[k]) * colf[j], acc);
          }
        }
      }
      const double tot = block_sum(static_cast<double>(acc), red);
      if (threadIdx.x == 0) a.spart[d.tile0 + local] = tot;
      return;
    }
  }

  float acc = 0.f;  // this lane's share of sum(u^2) over the tile (<= 32 rows)
  for (int64_t i = i0 + warp; i < i1; i += RPI * kWarps) {
    float ts[RPI];
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr) ts[rr] = 0.f;
#pragma unroll
    for (int kg = 0; kg < CH; kg += CG) {
      if (j0 + kg * 32 * VEC >= W) break;  // the rest of the tile is past the row's end (warp-uniform)
      Raw<GT, VEC> raw[RPI][CG];
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr) {
        const int64_t ii = i + rr * kWarps;
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int64_t j = j0 + (kg + k) * 32 * VEC + lane * VEC;
          if (ii < i1 && j < W) load_raw(raw[rr][k], gb + ii * W + j);
        }
      }
#pragma unroll
      for (int rr = 0; rr < RPI; ++rr) {
        const int64_t ii = i + rr * kWarps;
#pragma unroll
        for (int k = 0; k < CG; ++k) {
          const int cl = (kg + k) * 32 * VEC + lane * VEC;
          if (ii < i1 && j0 + cl < W) {
            float x[VEC], f[VEC];
            widen(raw[rr][k], x);
            load_colf<VEC>(f, colf, kg + k, lane);
#pragma unroll
            for (int v = 0; v < VEC; ++v) ts[rr] = fmaf(x[v] * x[v], f[v], ts[rr]);
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < RPI; ++rr) {
      const int64_t ii = i + rr * kWarps;
      if (ii < i1) {
        acc = fmaf(rowf[ii - i0], ts[rr], acc);
      }
    }
  }
  const double tot = block_sum(static_cast<double>(acc), red);
  if (threadIdx.x == 0) a.spart[d.tile0 + local] = tot;
}

template <typename GT, int VEC>
__global__ void __launch_bounds__(kThreads, 2) k_pass2_f(const __grid_constant__ StepArgs a, const Range r) {
  extern __shared__ __align__(16) unsigned char smem[];
  double* red = reinterpret_cast<double*>(smem);
  int32_t* pf = reinterpret_cast<int32_t*>(smem + kRedBytes);
  float* colf = reinterpret_cast<float*>(smem + kRedBytes + kPrefixBytes);
  float* rowf = colf + kTileCols;
  const int ng = load_prefix(pf, r);
  const int64_t u1 = pf[ng];
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor d = a.tensors[member_tensor(r, m)];
    pass2_factored<GT, VEC>(d, a, u - pf[m], colf, rowf, red);
  }
}

// ---- clip: coef = alpha / max(1, RMS(u) / d), one CTA per tensor ----------
__global__ void __launch_bounds__(kThreads) k_clip(const __grid_constant__ StepArgs a) {
  __shared__ double red[16];
  const int t = blockIdx.x;
  const DevTensor d = a.tensors[t];
  double S;
  if (a.phase == 3) {
    S = a.round2[t];  // sum over all shards
  } else if (is_fused(d.kind)) {
    S = a.ssum[t];
  } else {
    double acc = 0.0;
    for (int64_t k = threadIdx.x; k < d.ntiles; k += kThreads) acc += a.spart[d.tile0 + k];
    S = block_sum(acc, red);
  }
  if (a.phase == 2) {  // row-sharded middle: this shard's sum(u^2) to exchange round 2
    if (threadIdx.x == 0) a.round2[t] = S;
    return;
  }
  if (threadIdx.x == 0) {
    const double rms_u = sqrt(S / static_cast<double>(d.ng));
    double div = rms_u / a.clip;
    if (!(div > 1.0)) div = 1.0;
    a.coef[t] = a.alpha[t] / div;
  }
}

// ---- 8-bit first moment ----------------------------------------------------
// The ms-swift GaLore / Q-GaLore article's block quantisation ("Q-Galore"
// section, its quantize_tensor / dequantize_tensor listing) applied to
// exp_avg.  Groups are kQ8Group values along the last dim; a group's state is
// its codes and one fp32 scale, value = code * scale.  Per step and group:
// the old moment is dequantised, m = beta1 * old + (1 - beta1) * u, then the
// group is re-quantised as the listing does, scale = amax / 127 and code =
// round-half-even(m / scale) (both quotients correctly rounded fp32), and the
// update applied to the parameter is the dequantised new moment code * scale,
// the value the stored state holds (the listing dequantises before use).
__device__ __forceinline__ float q8_value(uint32_t codes4, int v, float scale) {
  const int c = static_cast<int>(static_cast<int8_t>((codes4 >> (8 * v)) & 0xffu));
  return __fmul_rn(static_cast<float>(c), scale);
}
// Warp maximum of non-negative floats: their bit patterns order like
// unsigned integers, so one redux.sync.max.u32 does it.
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}
// Reciprocal with at most 1 ulp of error (rcp.approx.f32: subnormals
// handled, 1 / 0 = +inf).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// Quantises NG groups of the new moment, each 128 values held 4 per lane by
// the 32 lanes of a warp (out-of-range values passed as 0; every lane of the
// warp must call).  sc[g] = amax / 127 of group g (correctly rounded; 0 for
// an all-zero group); c[g][v] = the code round-half-even(fl(m[g][v] /
// sc[g])), clamped to [-128, 127], as a float.
//
// Each code is first taken from x = fl(m * r) with r = 1 / scale to 1 ulp:
// |x - fl(m / scale)| <= |m / scale| (2^-23 + 2^-24 + 2^-24) < 3.1e-5, since
// |m| <= amax makes |m / scale| at most 127 (1 + 2^-23) for a normal scale.
// Where x lies farther than kQ8TieBand (> 3.1e-5) from every half-integer,
// rint(x) is therefore the page's code.  Where any value of the NG groups
// lies closer, or a scale is subnormal, all NG groups take the correctly
// rounded divisions instead (a warp-uniform branch, rarely taken: about 3 %
// of the groups).
constexpr float kQ8TieBand = 1.0f / 8192.0f;
template <int NG>
__device__ __forceinline__ void q8_groups(const float (&m)[NG][4], float (&c)[NG][4], float (&sc)[NG]) {
  bool near = false;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float amax = fmaxf(fmaxf(fabsf(m[g][0]), fabsf(m[g][1])), fmaxf(fabsf(m[g][2]), fabsf(m[g][3])));
    amax = warp_max_nonneg(amax);
    sc[g] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
    const float r = sc[g] > 0.f ? rcp_approx(sc[g]) : 0.f;
    near |= sc[g] > 0.f && sc[g] < 0x1p-126f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float x = __fmul_rn(m[g][v], r);
      c[g][v] = rintf(x);
      near |= fabsf(__fsub_rn(x, c[g][v])) > 0.5f - kQ8TieBand;
    }
  }
  if (__any_sync(0xffffffffu, near)) {
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int v = 0; v < 4; ++v)
        c[g][v] = sc[g] > 0.f ? fminf(fmaxf(rintf(__fdiv_rn(m[g][v], sc[g])), -128.f), 127.f) : 0.f;
  }
}
// p <- p - wd * alpha * p - code * scale: the dequantised moment is applied
// with one rounding (fl(code * scale), the stored state's value, differs
// from the exact product by at most half an ulp of it).
__device__ __forceinline__ float q8_update(float p, float wda, float c, float sc) {
  return fmaf(-wda, p, fmaf(-c, sc, p));
}
// Codes of 4 values (integral floats in [-128, 127]), packed little-endian.
__device__ __forceinline__ uint32_t q8_pack4(const float (&c)[4]) {
  uint32_t w = 0;
#pragma unroll
  for (int v = 0; v < 4; ++v) w |= (static_cast<uint32_t>(__float2int_rn(c[v])) & 0xffu) << (8 * v);
  return w;
}

// ---- apply: p <- p - wd*alpha*p - update ----------------------------------
// colf holds coef * col_j^-1/2 for the tile's columns (shared memory).
template <typename GT, int VEC, bool B1, bool Q8, bool PSQ>
__device__ __forceinline__ void apply_factored(const DevTensor& d, const StepArgs& a, int t, int64_t local, float* colf,
                               float* rowf, double* red) {
  static_assert(!Q8 || (B1 && VEC == 1 && Layout<VEC>::CG * 32 % kQ8Group == 0),
                "8-bit moment: element-wise layout, whole groups per load group");
  constexpr int CH = Layout<VEC>::CH, CG = Layout<VEC>::CG;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const TilePos tp = tile_pos(d, local);
  const int64_t H = d.H, W = d.W;
  const int64_t i0 = tp.r * kTileRows;
  const int64_t i1 = min(H, i0 + kTileRows);
  const int64_t j0 = tp.c * kTileCols;
  const int64_t base = tp.b * H * W;
  const GT* gb = static_cast<const GT*>(d.g) + base;
  float* pb = d.p + base;
  float* mb = (B1 && !Q8) ? d.m1 + base : nullptr;
  int8_t* qb = Q8 ? d.mq + base : nullptr;
  const float* row = d.row + tp.b * H;
  const float m = static_cast<float>(a.mrow[d.mslot + tp.b]);
  const float coef = static_cast<float>(a.coef[t]);
  const float wda = static_cast<float>(a.wd * a.alpha[t]);
  const float b1 = static_cast<float>(a.beta1), omb1 = static_cast<float>(1.0 - a.beta1);

  __syncthreads();  // previous tile's readers of colf are done
  for (int cl = threadIdx.x; cl < kTileCols; cl += kThreads) {
    const int64_t j = j0 + cl;
    colf[colf_index<VEC>(cl)] = (j < W) ? coef * rsqrtf(d.col[tp.b * W + j]) : 0.f;
  }
  constexpr bool kFlat = VEC == 1 && !Q8;  // 8-bit groups need the row-by-row layout
  if (kFlat && W <= kTileCols) {
    for (int rl = threadIdx.x; rl < kTileRows; rl += kThreads) {
      const int64_t i = i0 + rl;
      rowf[rl] = (i < i1) ? rsqrtf(row[i] / m) : 0.f;
    }
  }
  __syncthreads();

  float psq = 0.f;
  if constexpr (kFlat) {
    if (W <= kTileCols) {  // whole rows: stream the tile by flat index
      const int cnt = static_cast<int>((i1 - i0) * W);
      const int64_t o = i0 * W;
      const float invw = 1.0f / static_cast<float>(W);
      const int w32 = static_cast<int>(W);
      int start = 0;  // first value left to the scalar loop
      if (vec4_aligned(gb + o) && vec4_aligned(pb + o) && (!B1 || vec4_aligned(mb + o))) {
        constexpr int UA = B1 ? kFlatVecA - 1 : kFlatVecA;
        const int nv = cnt >> 2;
        for (int v0 = threadIdx.x; v0 < nv; v0 += UA * kThreads) {
          Raw4<GT> raw[UA];
          float4 p4[UA], m4[B1 ? UA : 1];
#pragma unroll
          for (int k = 0; k < UA; ++k) {
            const int v = v0 + k * kThreads;
            if (v < nv) {
              load_raw4(raw[k], gb + o + 4 * v);
              p4[k] = __ldcs(reinterpret_cast<const float4*>(pb + o + 4 * v));
              if (B1) m4[B1 ? k : 0] = __ldcs(reinterpret_cast<const float4*>(mb + o + 4 * v));
            }
          }
#pragma unroll
          for (int k = 0; k < UA; ++k) {
            const int v = v0 + k * kThreads;
            if (v < nv) {
              float x[4], pv[4] = {p4[k].x, p4[k].y, p4[k].z, p4[k].w}, mv[4];
              if (B1) {
                const float4 mm = m4[B1 ? k : 0];
                mv[0] = mm.x; mv[1] = mm.y; mv[2] = mm.z; mv[3] = mm.w;
              }
              widen4(raw[k], x);
              int i = flat_row(4 * v, invw), j = 4 * v - i * w32;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float upd = (x[q] * rowf[i]) * colf[j];
                if (B1) {
                  mv[q] = fmaf(b1, mv[q], omb1 * upd);
                  upd = mv[q];
                }
                pv[q] = fmaf(-wda, pv[q], pv[q] - upd);
                if (PSQ) psq = fmaf(pv[q], pv[q], psq);
                flat_next(i, j, w32);
              }
              __stcs(reinterpret_cast<float4*>(pb + o + 4 * v), make_float4(pv[0], pv[1], pv[2], pv[3]));
              if (B1) __stcs(reinterpret_cast<float4*>(mb + o + 4 * v), make_float4(mv[0], mv[1], mv[2], mv[3]));
            }
          }
        }
        start = nv << 2;
      }
      for (int e0 = start + threadIdx.x; e0 < cnt; e0 += kFlatApply * kThreads) {
        float x[kFlatApply], pv[kFlatApply], mv[B1 ? kFlatApply : 1];
#pragma unroll
        for (int k = 0; k < kFlatApply; ++k) {
          const int e = e0 + k * kThreads;
          if (e < cnt) {
            x[k] = load_g_scalar<GT>(gb + o + e);
            pv[k] = __ldcs(pb + o + e);
            if (B1) mv[B1 ? k : 0] = __ldcs(mb + o + e);
          }
        }
#pragma unroll
        for (int k = 0; k < kFlatApply; ++k) {
          const int e = e0 + k * kThreads;
          if (e < cnt) {
            const int i = flat_row(e, invw), j = e - i * w32;
            float upd = (x[k] * rowf[i]) * colf[j];
            if (B1) {
              mv[B1 ? k : 0] = fmaf(b1, mv[B1 ? k : 0], omb1 * upd);
              upd = mv[B1 ? k : 0];
              __stcs(mb + o + e, mv[B1 ? k : 0]);
            }
            const float pn = fmaf(-wda, pv[k], pv[k] - upd);
            __stcs(pb + o + e, pn);
            if (PSQ) psq = fmaf(pn, pn, psq);
          }
        }
      }
      if (PSQ) {
        const double tot = block_sum(static_cast<double>(psq), red);
        if (threadIdx.x == 0) a.ppart[d.tile0 + local] = tot;
      }
      return;
    }
  }
  for (int64_t i = i0 + warp; i < i1; i += kWarps) {
    const float r_i = rsqrtf(row[i] / m);
#pragma unroll
    for (int kg = 0; kg < CH; kg += CG) {
      if (j0 + kg * 32 * VEC >= W) break;  // the rest of the tile is past the row's end (warp-uniform)
      Raw<GT, VEC> raw[CG];
      float pv[CG][VEC];
      float mv[B1 ? CG : 1][VEC];
      constexpr int QPG = kQ8Group / 32;  // element-wise chunks per 8-bit group
      float qs[Q8 ? CG / QPG : 1];        // group scales of this load group
#pragma unroll
      for (int k = 0; k < CG; ++k) {
        const int64_t j = j0 + (kg + k) * 32 * VEC + lane * VEC;
        if (j < W) {
          load_raw(raw[k], gb + i * W + j);
          load_f<VEC>(pv[k], pb + i * W + j);
          if (B1 && !Q8) load_f<VEC>(mv[B1 ? k : 0], mb + i * W + j);
          if (Q8) mv[B1 ? k : 0][0] = static_cast<float>(qb[i * W + j]);
        }
      }
      if (Q8) {
#pragma unroll
        for (int q = 0; q < CG / QPG; ++q) {
          const int64_t jg = j0 + (kg + q * QPG) * 32;
          qs[Q8 ? q : 0] = jg < W ? d.ms[(tp.b * H + i) * d.qg + jg / kQ8Group] : 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < CG; ++k) {
        const int cl = (kg + k) * 32 * VEC + lane * VEC;
        const int64_t j = j0 + cl;
        if (j < W) {
          float x[VEC], f[VEC];
          widen(raw[k], x);
          load_colf<VEC>(f, colf, kg + k, lane);
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            float upd = (x[v] * r_i) * f[v];
            if (B1) {
              const float old = Q8 ? __fmul_rn(mv[B1 ? k : 0][v], qs[Q8 ? k / QPG : 0]) : mv[B1 ? k : 0][v];
              mv[B1 ? k : 0][v] = fmaf(b1, old, omb1 * upd);
              upd = mv[B1 ? k : 0][v];
            }
            if (!Q8) {  // (the 8-bit moment updates p after re-quantising)
              const float pn = fmaf(-wda, pv[k][v], pv[k][v] - upd);
              pv[k][v] = pn;
              if (PSQ) psq = fmaf(pn, pn, psq);
            }
          }
          if (!Q8) store_f<VEC>(pb + i * W + j, pv[k]);
          if (B1 && !Q8) store_f<VEC>(mb + i * W + j, mv[B1 ? k : 0]);
        }
      }
      if (Q8) {
        // re-quantise each group of QPG chunks (warp max of |m|, scale,
        // codes), then apply the dequantised moment to p
        static_assert(!Q8 || (QPG == 4 && CG / QPG == 2), "a lane holds 4 values of each of 2 groups");
        float mg[2][4], c[2][4], sc[2];
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int kk = 0; kk < QPG; ++kk) {
            const int k = q * QPG + kk;
            mg[q][kk] = (j0 + (kg + k) * 32 + lane < W) ? mv[B1 ? k : 0][0] : 0.f;
          }
        q8_groups<2>(mg, c, sc);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
#pragma unroll
          for (int kk = 0; kk < QPG; ++kk) {
            const int k = q * QPG + kk;
            const int64_t j = j0 + (kg + k) * 32 + lane;
            if (j < W) {
              qb[i * W + j] = static_cast<int8_t>(__float2int_rn(c[q][kk]));
              const float pn = q8_update(pv[k][0], wda, c[q][kk], sc[q]);
              pb[i * W + j] = pn;
              if (PSQ) psq = fmaf(pn, pn, psq);
            }
          }
          const int64_t jg = j0 + (kg + q * QPG) * 32;
          if (lane == 0 && jg < W) d.ms[(tp.b * H + i) * d.qg + jg / kQ8Group] = sc[q];
        }
      }
    }
  }
  if (PSQ) {
    const double tot = block_sum(static_cast<double>(psq), red);
    if (threadIdx.x == 0) a.ppart[d.tile0 + local] = tot;
  }
}

template <bool B1, bool PSQ>
__device__ __forceinline__ void apply_unfactored(const DevTensor& d, const StepArgs& a, int t, int64_t local, double* red) {
  const int64_t e0 = local * kTile1D;
  const int64_t e1 = min(d.n, e0 + kTile1D);
  const float coef = static_cast<float>(a.coef[t]);
  const float wda = static_cast<float>(a.wd * a.alpha[t]);
  const float b1 = static_cast<float>(a.beta1), omb1 = static_cast<float>(1.0 - a.beta1);
  float psq = 0.f;
  for (int64_t e00 = e0 + threadIdx.x; e00 < e1; e00 += kBatch1D * kThreads) {
    float x[kBatch1D], v[kBatch1D], m[kBatch1D], pv[kBatch1D];
#pragma unroll
    for (int k = 0; k < kBatch1D; ++k) {
      const int64_t e = e00 + k * kThreads;
      x[k] = m[k] = pv[k] = 0.f;
      v[k] = 1.f;
      if (e < e1) {
        x[k] = load_g1(d.g, d.gdt, e);
        v[k] = d.v[e];
        if (B1) m[k] = d.m1[e];
        pv[k] = d.p[e];
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch1D; ++k) {
      const int64_t e = e00 + k * kThreads;
      if (e < e1) {
        float upd = coef * (x[k] * rsqrtf(v[k]));
        if (B1) {
          const float mn = fmaf(b1, m[k], omb1 * upd);
          d.m1[e] = mn;
          upd = mn;
        }
        const float pn = fmaf(-wda, pv[k], pv[k] - upd);
        d.p[e] = pn;
        if (PSQ) psq = fmaf(pn, pn, psq);
      }
    }
  }
  if (PSQ) {
    const double tot = block_sum(static_cast<double>(psq), red);
    if (threadIdx.x == 0) a.ppart[d.tile0 + local] = tot;
  }
}

// 1D tensors with the 8-bit moment: warp w takes the groups w, w + 8, ... of
// the tile (lane l: values 4l .. 4l + 3 of a group), two groups per pass.
template <bool PSQ>
__device__ __forceinline__ void apply_unfactored_q8(const DevTensor& d, const StepArgs& a, int t, int64_t local,
                                                    double* red) {
  const int64_t e0 = local * kTile1D;
  const int64_t e1 = min(d.n, e0 + kTile1D);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float coef = static_cast<float>(a.coef[t]);
  const float wda = static_cast<float>(a.wd * a.alpha[t]);
  const float b1 = static_cast<float>(a.beta1), omb1 = static_cast<float>(1.0 - a.beta1);
  constexpr int GP = 2;  // groups per warp and pass
  float psq = 0.f;
  for (int64_t g0 = e0 / kQ8Group + warp * GP; g0 * kQ8Group < e1; g0 += kWarps * GP) {
    float x[GP][4], v[GP][4], pv[GP][4], m[GP][4], sc[GP];
#pragma unroll
    for (int q = 0; q < GP; ++q) {
      const int64_t gb = (g0 + q) * kQ8Group;
      sc[q] = gb < e1 ? d.ms[g0 + q] : 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t e = gb + lane * 4 + k;
        x[q][k] = pv[q][k] = m[q][k] = 0.f;
        v[q][k] = 1.f;
        if (e < e1) {
          x[q][k] = load_g1(d.g, d.gdt, e);
          v[q][k] = d.v[e];
          pv[q][k] = d.p[e];
          m[q][k] = static_cast<float>(d.mq[e]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < GP; ++q) {
      const int64_t gb = (g0 + q) * kQ8Group;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t e = gb + lane * 4 + k;
        if (e < e1) {
          const float upd = coef * (x[q][k] * rsqrtf(v[q][k]));
          m[q][k] = fmaf(b1, __fmul_rn(m[q][k], sc[q]), omb1 * upd);
        }
      }
    }
    float c[GP][4], s[GP];
    q8_groups<GP>(m, c, s);  // warp-uniform: a group is in range for the whole warp or not at all
#pragma unroll
    for (int q = 0; q < GP; ++q) {
      const int64_t gb = (g0 + q) * kQ8Group;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t e = gb + lane * 4 + k;
        if (e < e1) {
          d.mq[e] = static_cast<int8_t>(__float2int_rn(c[q][k]));
          const float pn = q8_update(pv[q][k], wda, c[q][k], s[q]);
          d.p[e] = pn;
          if (PSQ) psq = fmaf(pn, pn, psq);
        }
      }
      if (lane == 0 && gb < e1) d.ms[g0 + q] = s[q];
    }
  }
  if (PSQ) {
    const double tot = block_sum(static_cast<double>(psq), red);
    if (threadIdx.x == 0) a.ppart[d.tile0 + local] = tot;
  }
}

template <typename GT, int VEC, bool B1, bool Q8, bool PSQ>
__global__ void __launch_bounds__(kThreads, 2) k_apply_f(const __grid_constant__ StepArgs a, const Range r) {
  extern __shared__ __align__(16) unsigned char smem[];
  double* red = reinterpret_cast<double*>(smem);
  int32_t* pf = reinterpret_cast<int32_t*>(smem + kRedBytes);
  float* colf = reinterpret_cast<float*>(smem + kRedBytes + kPrefixBytes);
  float* rowf = colf + kTileCols;  // allocated for the element-wise layout only
  const int ng = load_prefix(pf, r);
  const int64_t u1 = pf[ng];
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const int t = member_tensor(r, m);
    const DevTensor d = a.tensors[t];
    apply_factored<GT, VEC, B1, Q8, PSQ>(d, a, t, u - pf[m], colf, rowf, red);
  }
}

template <bool B1, bool Q8, bool PSQ>
__global__ void __launch_bounds__(kThreads) k_apply_u(const __grid_constant__ StepArgs a, const Range r) {
  extern __shared__ __align__(16) unsigned char smem[];
  double* red = reinterpret_cast<double*>(smem);
  int32_t* pf = reinterpret_cast<int32_t*>(smem + kRedBytes);
  const int ng = load_prefix(pf, r);
  const int64_t u1 = pf[ng];
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const int t = member_tensor(r, m);
    const DevTensor d = a.tensors[t];
    if (Q8) apply_unfactored_q8<PSQ>(d, a, t, u - pf[m], red);
    else apply_unfactored<B1, PSQ>(d, a, t, u - pf[m], red);
  }
}

// ---- vector path of apply: bulk-copy (TMA) staged rows ----------------------
// One CTA per SM: warp 8 is the producer, warps 0-7 the consumers.  The
// producer streams the tile rows of g, p (and exp_avg) into a ring of
// shared-memory stages of 8 rows with cp.async.bulk, one
// copy per row segment, completion counted on the stage's "full" mbarrier.
// Consumer warp w takes row w % kTmaRows of every stage, column block
// w / kTmaRows of kTileCols / SPLIT, and releases the stage on its
// "empty" mbarrier.  The bytes in flight are set by the ring depth, not by
// registers.  In each 256-column chunk k, lane l handles the column quads
// k*256 + 4l and k*256 + 128 + 4l, so shared-memory reads and global stores
// are contiguous across the warp.
// Every wait is bounded (kWaitCycles): after a timeout the kernel sets
// kStatusWaitTimeout in the status word; the warp keeps meeting the consumer
// barriers without touching the stages, so no warp is left waiting at one,
// and all consumers leave together at the next tile boundary.
constexpr int kTmaRows = kWarps;  // rows per stage
// SPLIT consumer warps per row (column blocks of kTileCols / SPLIT): 1 for
// the plain apply, 2 for the 8-bit moment, whose per-group re-quantisation
// needs more warps to hide its dependent arithmetic, and 2 for the fp32
// moment, whose stages hold 4 rows (RS) instead of 8: its rows are 10 KB
// (bf16 g, p, exp_avg), and 8-row stages left only two in the ring.
template <int SPLIT, int RS = kTmaRows> struct TmaCfg {
  static constexpr int kConsumers = RS * SPLIT;
  static constexpr int kThreads = (kConsumers + 1) * 32;
  static_assert(kTileCols % (256 * SPLIT) == 0, "a consumer warp takes whole 256-column chunks");
  static_assert(kConsumers <= 32, "consumer warp sums fit the reduction buffer");
};

template <typename GT, bool WP, bool WM, size_t kBudget, int RS = kTmaRows>
struct Ring {
  static constexpr int kRows = RS;  // tile rows per stage
  static constexpr int kG = kTileCols * sizeof(GT);
  static constexpr int kP = WP ? kTileCols * 4 : 0;
  static constexpr int kM = WM ? kTileCols * 4 : 0;
  static constexpr int kRow = kG + kP + kM;
  static constexpr int kStage = RS * kRow;
  static constexpr int kStages = kBudget / kStage < 16 ? static_cast<int>(kBudget / kStage) : 16;
  static constexpr size_t kBytes = static_cast<size_t>(kStages) * kStage;
  static_assert(kStages >= 2, "stage ring too small");
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of parity `parity` to complete; false after kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}
// Bulk copy global -> this CTA's shared memory, completion on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
template <int NC>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NC * 32) : "memory");
}

// Shared prologue: prefix copy and barrier init (all threads of the CTA;
// NC consumer warps arrive on each "empty" barrier).
template <int kStages, int NC>
__device__ __forceinline__ int tma_setup(int32_t* pf, const Range& r, uint64_t* full, uint64_t* empty) {
  const int ng = r.m_end - r.m_begin;
  for (int k = threadIdx.x; k <= ng; k += blockDim.x) pf[k] = r.pf[r.m_begin + k];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  return ng;
}

// The producer (one thread): every RG::kRows-row stage of every tile of this CTA.
template <typename GT, class RG>
__device__ __forceinline__ void tma_produce(const StepArgs& a, const Range& r, const int32_t* pf, int ng,
                                            unsigned char* ring, uint64_t* full, uint64_t* empty) {
  if (a.stall_copies) return;  // testing hook: the consumers' waits run out
  const int64_t u1 = pf[ng];
  uint32_t it = 0;
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor d = a.tensors[member_tensor(r, m)];
    const TilePos tp = tile_pos(d, u - pf[m]);
    const int64_t i0 = tp.r * kTileRows, i1 = min(d.H, i0 + kTileRows);
    const int64_t j0 = tp.c * kTileCols;
    const uint32_t ncol = static_cast<uint32_t>(min(static_cast<int64_t>(kTileCols), d.W - j0));
    const int64_t base = tp.b * d.H * d.W;
    for (int64_t rs = i0; rs < i1; rs += RG::kRows, ++it) {
      const uint32_t slot = it % RG::kStages, ph = (it / RG::kStages) & 1u;
      if (!mbar_wait(&empty[slot], ph ^ 1u)) {
        atomicOr(a.status, kStatusWaitTimeout);
        return;
      }
      const int nrows = static_cast<int>(min(static_cast<int64_t>(RG::kRows), i1 - rs));
      const uint32_t per_row = ncol * static_cast<uint32_t>(sizeof(GT) + (RG::kP ? 4 : 0) + (RG::kM ? 4 : 0));
      mbar_arrive_expect_tx(&full[slot], nrows * per_row);
      unsigned char* st = ring + slot * RG::kStage;
      for (int rr = 0; rr < nrows; ++rr) {
        const int64_t off = base + (rs + rr) * d.W + j0;
        unsigned char* row = st + rr * RG::kRow;
        bulk_g2s(row, static_cast<const GT*>(d.g) + off, ncol * sizeof(GT), &full[slot]);
        if (RG::kP) bulk_g2s(row + RG::kG, d.p + off, ncol * 4, &full[slot]);
        if (RG::kM) bulk_g2s(row + RG::kG + RG::kP, d.m1 + off, ncol * 4, &full[slot]);
      }
    }
  }
}

// Consumer-side wait for a stage; on timeout flags the status and `stop`.
__device__ __forceinline__ bool tma_acquire(uint64_t* bar, uint32_t parity, const StepArgs& a, int* stop) {
  if (mbar_wait(bar, parity)) return true;
  if ((threadIdx.x & 31) == 0) atomicOr(a.status, kStatusWaitTimeout);
  *stop = 1;
  return false;
}

// After a timeout: give copies still in flight a bounded chance to land
// before the CTA's shared memory goes away.
template <int kStages>
__device__ __forceinline__ void tma_drain(uint64_t* full, uint32_t it) {
  for (uint32_t k = 0; k < static_cast<uint32_t>(kStages); ++k) {
    const uint32_t j = it + k;
    const long long t0 = clock64();
    while (!mbar_try_wait(&full[j % kStages], (j / kStages) & 1u)) {
      if (clock64() - t0 > kWaitCycles / 8) break;
    }
  }
}

// 4 gradient values of one column quad from a staged row.
template <typename GT>
__device__ __forceinline__ void quad_g(float (&x)[4], const unsigned char* row, int cl) {
  if (sizeof(GT) == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + cl * 2);
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xffff0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xffff0000u);
  } else {
    const float4 w = *reinterpret_cast<const float4*>(row + cl * 4);
    x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
  }
}

// Consumer-only deterministic CTA sum over NC consumer warps (warp
// xor-trees, then warps in order); valid in consumer thread 0.
template <int NC>
__device__ __forceinline__ double consumer_sum(float v, double* red) {
  const float w = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = static_cast<double>(w);
  consumer_sync<NC>();
  double s = 0.0;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < NC; ++k) s += red[k];
  }
  return s;
}

// ---- fused flat pass 1 (kFactoredFlat) ------------------------------------
// Tensors whose rows fit one tile (W <= kTileCols): a work unit is a chunk of
// d.pr whole rows [i0, i1) of one slice (chosen by the planner so that a
// unit holds about 64K values), so the row statistic can be formed in pass 1,
// and with it D_j = sum_i g_ij^2 / row_i, as in the row-panel pass:
// sum(u^2) = mean(row) * sum_j D_j / col_j (k_stats, k_scalars), and g is
// read once for the statistics and sum(u^2) instead of twice (no pass 2).
//
// A unit's rows are one contiguous range of g.  One producer thread streams
// it, in chunks of R whole rows (at most kFlatChunkBytes, chunk starts on
// 16-byte boundaries), with cp.async.bulk into a ring of kFlatSlots slots;
// the 8 consumer warps read the rows back from shared memory.  Each row is
// taken by a segment of L = min(32, p) lanes (p the power of 2 >= W; 32 / L
// rows per warp at once), lane c of the segment holding columns c, c + L, ...
// (CPL = ceil(W / L) <= 16 of them).  Rows wider than 512 values are split
// between the two warps of a pair (warps w and w + 4): columns [0, 512) and
// [512, W), 16 per lane each; the pair adds its two half-row sums (low half
// first) through shared memory at a named barrier of its own.  Warp w (pair
// p) takes row groups w, w + 8 (p, p + 4), ... of every chunk.  Per row: the
// segment's xor-butterfly gives every lane the same total (each level adds
// the same two values, in either order), hence the same row EMA and
// 1 / row_i; each lane then adds its values to C_j and g^2 / row_i to D_j in
// registers.  The old row statistics of a warp's rows in a chunk are loaded
// kFlatRoldAhead chunks ahead, one per lane.  At the unit's end the warps' (pairs')
// column partials meet in shared memory and are added in warp (pair) order,
// while the producer already streams the next unit.  The values past a
// slice's last 16-byte boundary (fewer than 16 bytes) are read from global
// memory by their lanes.  All orders are fixed, so two runs give bit-identical
// results.  Every wait is bounded as in k_apply_tma.
constexpr int kFlatChunkBytes = 16384;         // one ring slot
constexpr int kFlatSlots = 4;                  // ring slots
constexpr int kFlatHalfW = 512;                // widest row one warp takes
constexpr int kFlatPairs = kWarps / 2;         // warp pairs of the wide form
constexpr int kFlatThreads = (kWarps + 1) * 32;  // 8 consumer warps + the producer warp
constexpr int kFlatMinB = 2;                   // CTAs per SM
constexpr int kFlatRoldAhead = 4;              // chunks of old row statistics in flight per warp
// Named barrier 2 + pair, the pair's two warps only (barrier 1 is the
// consumers' barrier).
__device__ __forceinline__ void pair_sync(int pair) {
  static_assert(kFlatPairs == 4, "one named barrier per pair");
  switch (pair) {
    case 0: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
    case 1: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
    case 2: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
    default: asm volatile("bar.sync 5, 64;" ::: "memory"); break;
  }
}
// Rows per chunk for rows of w values: as many whole rows as fit one slot
// (at most kTileRows), a multiple of the rows that keep every chunk start on
// a 16-byte boundary (16 / gcd(16, w * sizeof(GT)) rows).
template <typename GT>
__device__ __forceinline__ int flat_chunk_rows(int w) {
  constexpr int A = 16 / static_cast<int>(sizeof(GT));  // values per 16 bytes
  const int low = w & -w;                               // largest power of 2 dividing w
  const int rmin = A / (low < A ? low : A);
  int R = kFlatChunkBytes / static_cast<int>(sizeof(GT)) / w;
  if (R > kTileRows) R = kTileRows;
  return R - R % rmin;
}
// One gradient value from shared memory, widened to fp32.
template <typename GT> __device__ __forceinline__ float smem_val(const GT* p);
template <> __device__ __forceinline__ float smem_val<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float smem_val<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
}
// A unit of the flat pass: slice b, chunk q of d.pr rows from row i0.
struct FlatUnit {
  int64_t b, q, i0;
  int w, nr;
  int cnt, cpy;  // values of the unit; those before its last 16-byte boundary
};
template <typename GT>
__device__ __forceinline__ FlatUnit flat_unit(const DevTensor* d, int64_t local) {
  FlatUnit f;
  udivmod32(local, d->prb, f.b, f.q);
  f.i0 = f.q * d->pr;
  f.w = static_cast<int>(d->W);
  f.nr = static_cast<int>(min(d->H, f.i0 + d->pr) - f.i0);
  f.cnt = f.nr * f.w;  // at most kTileRows * kTileCols
  f.cpy = f.cnt & ~(16 / static_cast<int>(sizeof(GT)) - 1);
  return f;
}

template <typename GT>
__device__ __forceinline__ void flat_produce(const StepArgs& a, const Range& r, const int32_t* pf, int ng,
                                             unsigned char* ring, uint64_t* full, uint64_t* empty) {
  if (a.stall_copies) return;  // testing hook: the consumers' waits run out
  const int64_t u1 = pf[ng];
  uint32_t it = 0;
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor* d = a.tensors + member_tensor(r, m);
    const FlatUnit f = flat_unit<GT>(d, u - pf[m]);
    const int R = flat_chunk_rows<GT>(f.w);
    const GT* g = static_cast<const GT*>(d->g) + (f.b * d->H + f.i0) * f.w;
    for (int r0 = 0; r0 < f.nr; r0 += R, ++it) {
      const uint32_t slot = it % kFlatSlots, ph = (it / kFlatSlots) & 1u;
      if (!mbar_wait(&empty[slot], ph ^ 1u)) {
        atomicOr(a.status, kStatusWaitTimeout);
        return;
      }
      const int e0 = r0 * f.w, e1 = min(min(r0 + R, f.nr) * f.w, f.cpy);
      const uint32_t bytes = e1 > e0 ? static_cast<uint32_t>(e1 - e0) * static_cast<uint32_t>(sizeof(GT)) : 0u;
      mbar_arrive_expect_tx(&full[slot], bytes);
      if (bytes) bulk_g2s(ring + slot * kFlatChunkBytes, g + e0, bytes, &full[slot]);
    }
  }
}

// One unit's rows on the consumer side (CPL columns per lane; HALF: the
// pair form).  `it` counts the ring's chunks; `dead` is set after a wait ran
// out (the warp then keeps the control flow, for the pair barriers, but
// neither waits nor reads).
template <typename GT, int CPL, bool PSQ, bool HALF>
__device__ __forceinline__ void flat_consume(const DevTensor* dt, const StepArgs& a, int64_t local,
                                             const unsigned char* ring, uint64_t* full, uint64_t* empty, float* cw,
                                             float* xs, float* rq, double* red, uint32_t& it, bool& dead, int* stop,
                                             const float3 bc) {
  // Fields are read where they are used (dt is not restrict: the stores in
  // between make the compiler read the epilogue's fields again instead of
  // holding them in registers across the row loop).
  const DevTensor& d = *dt;
  static_assert(!HALF || CPL == 16, "a half row is 512 columns, 16 per lane");
  constexpr int NS = HALF ? kFlatPairs : kWarps;     // column-partial sets
  constexpr int CS = HALF ? kTileCols : kFlatHalfW;  // columns per set
  const FlatUnit f = flat_unit<GT>(dt, local);
  const int w = f.w, nr = f.nr;
  const int R = flat_chunk_rows<GT>(w);
  const GT* gt = static_cast<const GT*>(d.g) + (f.b * d.H + f.i0) * w;
  float* rowst = d.row + f.b * d.H + f.i0;
  int lg = 5;  // W > 32 whenever CPL > 1
  if (CPL == 1)
    while (lg > 0 && (1 << (lg - 1)) >= w) --lg;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = HALF ? warp / kFlatPairs : 0;   // column half of the wide form
  const int set = HALF ? warp % kFlatPairs : warp;  // pair (wide form) or warp
  const int sub = lane >> lg, cl = lane & ((1 << lg) - 1);
  const int c0 = half * kFlatHalfW + cl;  // this lane's first column
  const int spg = 32 >> lg;               // rows per row group
  const int nk = c0 < w ? (w - c0 + (1 << lg) - 1) >> lg : 0;  // this lane's columns per row
  const float b2 = bc.x, omb2 = bc.y, eps1 = bc.z;
  const float invw = 1.0f / static_cast<float>(w);
  // lane j holds the old row statistic of this warp's j-th row of a chunk:
  // row group set + (j / spg) * NS, row j % spg of the group (at most 32 rows)
  // (the groups of a chunk go round the warps starting where the previous
  // chunk's left off, so a warp's extra rows move to the next warps chunk by
  // chunk instead of always falling to the same ones)
  auto first_group = [&](int goff) { return (set - goff + NS) % NS; };
  // The old row statistics are copied kFlatRoldAhead chunks ahead (a chunk
  // is a few hundred cycles of work per warp, less than a load from HBM
  // takes while the copies stream), each lane's value with a 4-byte
  // cp.async into its slot of this warp's queue rq (kFlatRoldAhead + 1
  // slots of 32 floats: the slot being refilled is never the one being
  // read), one commit group per chunk.  Every chunk before the last has
  // gpc row groups, so the chunk kFlatRoldAhead ahead of one with group
  // offset goff starts at group offset goff + kFlatRoldAhead * gpc.
  const int gpc = (R + spg - 1) / spg;
  auto prefetch = [&](int c0r, int cgoff, int slot) {
    if (c0r < nr) {
      const int rl = (first_group(cgoff) + (lane / spg) * NS) * spg + lane % spg;
      if (rl < min(R, nr - c0r))
        panel::cp_async4(static_cast<uint32_t>(__cvta_generic_to_shared(rq + slot * 32 + lane)), rowst + c0r + rl);
    }
    panel::cp_async_commit();  // (empty past the unit's end: the group count stays in step)
  };
#pragma unroll 1
  for (int k = 0; k < kFlatRoldAhead; ++k) prefetch(k * R, (k * gpc) % NS, k);
  int cq = 0;  // slot of the current chunk

  // column sums in pairs of columns (k, k + 1): packed fp32x2 arithmetic
  constexpr int NP = (CPL + 1) / 2;
  float2 cacc[NP], dacc[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) cacc[k] = dacc[k] = make_float2(0.f, 0.f);
  float rsum = 0.f;
  int parity = 0;  // exchange buffer of the wide form
  int goff = 0;  // row groups of the unit's earlier chunks, mod NS
#pragma unroll 1
  for (int r0 = 0; r0 < nr; r0 += R, ++it) {
    const int rows = min(R, nr - r0);
    const int ngc = (min(R, nr - r0) + spg - 1) / spg;  // row groups in the chunk
    const int gi0 = first_group(goff);
    const int goff_next = (goff + ngc) % NS;
    // this chunk's group is complete once at most kFlatRoldAhead - 1 are pending
    panel::cp_async_wait<kFlatRoldAhead - 1>();
    const float rcur = (gi0 + (lane / spg) * NS) * spg + lane % spg < rows ? rq[cq * 32 + lane] : 0.f;
    prefetch(r0 + kFlatRoldAhead * R, (goff + kFlatRoldAhead * gpc) % NS, cq == 0 ? kFlatRoldAhead : cq - 1);
    cq = cq == kFlatRoldAhead ? 0 : cq + 1;
    const uint32_t slot = it % kFlatSlots, ph = (it / kFlatSlots) & 1u;
    if (!dead && !mbar_wait(&full[slot], ph)) {
      if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
      *stop = 1;
      dead = true;
    }
    const GT* sb = reinterpret_cast<const GT*>(ring + slot * kFlatChunkBytes);
    // the row group that reaches past the unit's last 16-byte boundary (in
    // the last chunk of a slice) is read from global memory: the bulk copy
    // stops at the boundary
    const bool tail = (r0 + rows) * w > f.cpy;
#pragma unroll 1
    for (int gi = gi0, t = 0; gi < ngc; gi += NS, ++t) {
      const int rl = gi * spg + sub;  // row within the chunk
      const bool ok = rl < rows && !dead;
      const bool from_g = tail && (r0 + min((gi + 1) * spg, rows)) * w > f.cpy;  // warp-uniform
      float x[2 * NP];
      x[2 * NP - 1] = 0.f;
      if (from_g) {
        const GT* src = gt + (r0 + rl) * w + c0;
#pragma unroll
        for (int k = 0; k < CPL; ++k) x[k] = (ok && k < nk) ? load_g_scalar<GT>(src + (k << lg)) : 0.f;
      } else {
        // CPL is ceil(W / 32) rounded up to even, so every lane holds columns
        // k < CPL - 2 of a row; only the last two need the lane's count
        // (narrow rows and the upper half of the pair form: all of them)
        const GT* src = sb + rl * w + c0;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const bool v = (HALF || CPL < 4 || k >= CPL - 2) ? (ok && k < nk) : ok;
          x[k] = v ? smem_val<GT>(src + (k << lg)) : 0.f;
        }
      }
      float2 q[NP];
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < NP; ++m) {
        const float2 xv = make_float2(x[2 * m], x[2 * m + 1]);
        q[m] = __fmul2_rn(xv, xv);
        s2 = __fadd2_rn(s2, q[m]);
      }
      float s = s2.x + s2.y;
      for (int o = (1 << lg) >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (HALF) {
        // the pair's two half-row sums, low half first in both warps
        if (lane == 0) xs[parity * kWarps + warp] = s;
        pair_sync(set);
        const float other = xs[parity * kWarps + (warp ^ kFlatPairs)];
        s = half == 0 ? s + other : other + s;
        parity ^= 1;
      }
      const float ro = __shfl_sync(0xffffffffu, rcur, t * spg + sub);
      float ri = 0.f;
      if (ok) {
        const float rn = fmaf(b2, ro, omb2 * fmaf(s, invw, eps1));
        ri = __frcp_rn(rn);  // correctly rounded 1 / rn
        if (cl == 0 && half == 0) {
          rowst[r0 + rl] = rn;
          rsum += rn;
        }
      }
      const float2 ri2 = make_float2(ri, ri);
#pragma unroll
      for (int m = 0; m < NP; ++m) {
        cacc[m] = __fadd2_rn(cacc[m], q[m]);
        dacc[m] = __ffma2_rn(q[m], ri2, dacc[m]);
      }
    }
    __syncwarp();
    if (lane == 0 && !dead) mbar_arrive(&empty[slot]);
    goff = goff_next;
  }
  // narrow rows: add the warp's row segments column by column (lanes with
  // the same column differ in the bits above lg)
  if (lg < 5) {
    for (int o = 16; o >= (1 << lg); o >>= 1) {
      cacc[0].x += __shfl_xor_sync(0xffffffffu, cacc[0].x, o);
      dacc[0].x += __shfl_xor_sync(0xffffffffu, dacc[0].x, o);
    }
  }
  float psq = 0.f;
  if (PSQ && !dead) {
    const float* pt = d.p + (f.b * d.H + f.i0) * w;
    for (int e0 = threadIdx.x; e0 < f.cnt; e0 += 8 * kThreads) {
      float y[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int e = e0 + k * kThreads;
        y[k] = e < f.cnt ? __ldcs(pt + e) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) psq = fmaf(y[k], y[k], psq);
    }
  }
  // the column partials, C then D, through cw[set][j]
  const int64_t off = (f.b * d.prb + f.q) * w;
  consumer_sync<kWarps>();  // cw of the previous unit is read
  if (sub == 0) {
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int j = c0 + (k << lg);
      if (j < w) cw[set * CS + j] = (k & 1) ? cacc[k >> 1].y : cacc[k >> 1].x;
    }
  }
  // (warp sums in fp32: the row statistics and p^2 of one warp's rows)
  const double rw = warp_sum(rsum);
  const double pw = PSQ ? warp_sum(psq) : 0.f;
  if (lane == 0) {
    red[warp] = rw;
    if (PSQ) red[kWarps + warp] = pw;  // red holds 2 * kWarps doubles
  }
  consumer_sync<kWarps>();
  float* cp = a.colpart + d.colpart + off;
  for (int j = threadIdx.x; j < w; j += kThreads) {
    float tc = 0.f;
#pragma unroll
    for (int v = 0; v < NS; ++v) tc += cw[v * CS + j];
    cp[j] = tc;
  }
  if (threadIdx.x == 0 && !*stop) {
    double rt = 0.0, pt2 = 0.0;
#pragma unroll
    for (int v = 0; v < kWarps; ++v) {
      rt += red[v];
      if (PSQ) pt2 += red[kWarps + v];
    }
    a.rowchunk[d.rowchunk + f.b * d.nrc + f.q] = rt;
    if (PSQ) a.ppart[d.p1_0 + local] = pt2;
  }
  consumer_sync<kWarps>();
  if (sub == 0) {
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int j = c0 + (k << lg);
      if (j < w) cw[set * CS + j] = (k & 1) ? dacc[k >> 1].y : dacc[k >> 1].x;
    }
  }
  consumer_sync<kWarps>();
  float* dp = a.dpart + d.dpart + off;
  for (int j = threadIdx.x; j < w; j += kThreads) {
    float td = 0.f;
#pragma unroll
    for (int v = 0; v < NS; ++v) td += cw[v * CS + j];
    dp[j] = td;
  }
}

// Shared memory of k_pass1_flat: the ring, the column partials (8 sets of
// 512 columns or 4 pairs of 1024), the pair exchange (2 buffers x 8 warps),
// the warps' queues of old row statistics, CTA-sum scratch (2 x 8 doubles),
// mbarriers, member prefix.
constexpr size_t kFlatRing = static_cast<size_t>(kFlatChunkBytes) * kFlatSlots;
constexpr size_t kFlatCw = sizeof(float) * kWarps * kFlatHalfW;
constexpr size_t kFlatXs = sizeof(float) * 2 * kWarps;
constexpr size_t kFlatRqWarp = static_cast<size_t>(kFlatRoldAhead + 1) * 32;  // floats per warp
constexpr size_t kFlatRq = sizeof(float) * kWarps * kFlatRqWarp;
constexpr size_t kFlatSmem = kFlatRing + kFlatCw + kFlatXs + kFlatRq + kRedBytes +
                             sizeof(uint64_t) * 2 * kFlatSlots + kPrefixBytes;
static_assert(kWarps * kFlatHalfW == kFlatPairs * kTileCols && kRedBytes >= sizeof(double) * 2 * kWarps &&
                  (kFlatRing + kFlatCw + kFlatXs + kFlatRq) % 8 == 0,
              "shared-memory layout of the flat pass");
template <typename GT, bool PSQ>
__global__ void __launch_bounds__(kFlatThreads, kFlatMinB)
    k_pass1_flat(const __grid_constant__ StepArgs a, const Range r) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  float* cw = reinterpret_cast<float*>(smem + kFlatRing);
  float* xs = reinterpret_cast<float*>(smem + kFlatRing + kFlatCw);
  double* red = reinterpret_cast<double*>(smem + kFlatRing + kFlatCw + kFlatXs + kFlatRq);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kRedBytes / sizeof(double));
  uint64_t* empty = full + kFlatSlots;
  int32_t* pf = reinterpret_cast<int32_t*>(empty + kFlatSlots);
  __shared__ int stop;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) stop = 0;
  const int ng = tma_setup<kFlatSlots, kWarps>(pf, r, full, empty);
  if (warp == kWarps) {
    if (lane == 0) flat_produce<GT>(a, r, pf, ng, ring, full, empty);
    return;
  }
  float* rq = reinterpret_cast<float*>(smem + kFlatRing + kFlatCw + kFlatXs) + warp * kFlatRqWarp;  // this warp's
  const int64_t u1 = pf[ng];
  uint32_t it = 0;
  bool dead = false;
  // beta2, 1 - beta2 and eps1 in fp32, once (conversions from fp64 run on
  // the FP64 pipe, which is slow on this part)
  const float3 bc = make_float3(static_cast<float>(a.beta2), static_cast<float>(1.0 - a.beta2),
                                static_cast<float>(a.eps1));
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor* d = a.tensors + member_tensor(r, m);
    const int64_t local = u - pf[m];
    // columns per lane, rounded up to even (whole rows per warp up to 512)
    const int64_t cpl = (d->W + 31) / 32;
#define MEO_FLAT(C, HF) flat_consume<GT, C, PSQ, HF>(d, a, local, ring, full, empty, cw, xs, rq, red, it, dead, &stop, bc)
    switch (cpl) {
      case 1: MEO_FLAT(1, false); break;
      case 2: MEO_FLAT(2, false); break;
      case 3: case 4: MEO_FLAT(4, false); break;
      case 5: case 6: MEO_FLAT(6, false); break;
      case 7: case 8: MEO_FLAT(8, false); break;
      case 9: case 10: MEO_FLAT(10, false); break;
      case 11: case 12: MEO_FLAT(12, false); break;
      case 13: case 14: MEO_FLAT(14, false); break;
      case 15: case 16: MEO_FLAT(16, false); break;
      default: MEO_FLAT(16, true); break;
    }
#undef MEO_FLAT
    consumer_sync<kWarps>();  // stop is settled for every consumer
    if (stop) break;
  }
  if (stop && threadIdx.x == 0) tma_drain<kFlatSlots>(full, it);
}

// ---- fused pass 1 over row chunks (kFactoredRows) --------------------------
// The shared row-panel pass (row_panel.cuh) over chunks of d.pr full rows:
// the updated row statistic, the column partials C_j of g^2 and D_j of
// g^2 / row_i, the row-chunk sums of the new row statistic and, when RMS(p)
// is not carried, sum(p^2).  With the column statistic of the step,
// sum(u^2) = mean(row) * sum_j D_j / col_j (k_stats, k_scalars), so g is read
// from HBM once here instead of twice.  Configurations: NW = 8 warps, G = 2
// column groups of 256 per lane for 2048 <= W <= 4096 (2 CTAs per SM);
// NW = 14, G = 4 for W <= 14336 (1 CTA per SM; the 56 column groups of
// W = 14336 give every warp four: with 16 warps, half had three and waited
// at each sub-panel's barrier for the others), in the split form (a ring of
// 4 stages of 2-row sub-panels; the row shares meet at an mbarrier that each
// warp waits on one sub-panel later, instead of at a CTA barrier).
constexpr int kRowsNW = 8, kRowsG = 2, kRowsS = 3, kRowsMinB = 2;

// Dynamic shared memory of k_pass1_panel: ring and row shares, CTA-sum
// scratch (64 doubles), and the member prefix where it still fits the CTA's
// 227 KB (a ring of 4 stages of 56 KB does not leave room for it; the prefix
// is then read from global memory, a few loads per chunk of rows).
template <typename GT, int NW, int G, int S> struct PanelCfg {
  static constexpr size_t kRedOff = panel::Cfg<GT, NW, G, S>::kBytes;
  static constexpr size_t kBase = kRedOff + sizeof(double) * 64;
  static constexpr bool kSmemPrefix = kBase + kPrefixBytes <= 227 * 1024;
  static constexpr size_t kSmem = kBase + (kSmemPrefix ? kPrefixBytes : 0);
  static_assert(kRedOff % 8 == 0 && NW + 1 <= 64, "the CTA sum needs NW + 1 aligned doubles");
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
};

template <typename GT, int NW, int G, int S, int MINB, bool PSQ>
__global__ void __launch_bounds__(NW * 32, MINB)
    k_pass1_panel(const __grid_constant__ StepArgs a, const Range r) {
  using PC = PanelCfg<GT, NW, G, S>;
  extern __shared__ __align__(16) unsigned char smem[];
  double* red = reinterpret_cast<double*>(smem + PC::kRedOff);
  const int32_t* pf;
  int ng;
  if constexpr (PC::kSmemPrefix) {
    int32_t* spf = reinterpret_cast<int32_t*>(red + 64);
    ng = load_prefix(spf, r);
    pf = spf;
  } else {
    ng = r.m_end - r.m_begin;
    pf = r.pf + r.m_begin;
  }
  constexpr bool kSplit = panel::Cfg<GT, NW, G, S>::kSplit;
  if constexpr (kSplit) {
    if (threadIdx.x == 0) panel::split_init<GT, NW, G, S>(smem);
    __syncthreads();
  }
  uint32_t q = 0;     // sub-panels done (split form)
  bool dead = false;  // a split-form wait ran out
  const int64_t u1 = pf[ng];
  const float b2 = static_cast<float>(a.beta2), omb2 = static_cast<float>(1.0 - a.beta2);
  const float eps1 = static_cast<float>(a.eps1);
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor d = a.tensors[member_tensor(r, m)];
    // Row indices within a slice fit in int32 (the plan requires H <= INT32_MAX).
    const int32_t local = static_cast<int32_t>(u - pf[m]);
    const int32_t b = local / d.prb, chunk = local % d.prb;
    const int32_t H = static_cast<int32_t>(d.H), W = static_cast<int32_t>(d.W);
    const int32_t c0 = chunk * d.pr, c1 = min(H, c0 + d.pr);
    const GT* gb = static_cast<const GT*>(d.g) + static_cast<int64_t>(b) * H * W;
    const float* pb = d.p + static_cast<int64_t>(b) * H * W;
    auto where = [&]() {
      const int64_t off = static_cast<int64_t>(b * d.prb + chunk) * W;
      return panel::Partials{a.colpart + d.colpart + off, a.dpart + d.dpart + off};
    };
    float rsum = 0.f, psq = 0.f;
    if constexpr (kSplit)
      panel::run_chunk_split<GT, NW, G, S, PSQ>(smem, gb, pb, d.row + static_cast<int64_t>(b) * H, W, c0, c1, b2,
                                                omb2, eps1, where, rsum, psq, q, dead, a.status);
    else
      panel::run_chunk<GT, NW, G, S, PSQ>(smem, gb, pb, d.row + static_cast<int64_t>(b) * H, W, c0, c1, b2, omb2,
                                          eps1, where, rsum, psq);
    // (the barriers of the CTA sums also order this chunk's last reads of
    // the ring before the next chunk's prologue refills it)
    const double rtot = panel::block_sum<NW>(static_cast<double>(rsum), red);
    if (PSQ) {
      const double ptot = panel::block_sum<NW>(static_cast<double>(psq), red);
      if (threadIdx.x == 0) a.ppart[d.p1_0 + local] = ptot;
    }
    if (threadIdx.x == 0) a.rowchunk[d.rowchunk + b * d.nrc + chunk] = rtot;
  }
  panel::cp_async_wait_all();  // only empty groups can be pending here
}

// ---- apply (vector path) ---------------------------------------------------
template <typename GT, bool B1, int RS = kTmaRows>
using ApplyRing = Ring<GT, true, B1, 200 * 1024, RS>;

// Codes (4 per lane and 128-column half-chunk: exactly one 8-bit group) and
// this lane's group scale (lanes 0..7: the segment's 8 groups) of one row
// segment, read straight from global memory one row ahead of their use.
constexpr int kQ8Split = 2;                             // consumer warps per row with the 8-bit moment
constexpr int kQ8PerWarp = kTileCols / 128 / kQ8Split;  // 8-bit groups of one consumer warp's columns
struct Q8Row {
  uint32_t q[kQ8PerWarp];
  float s;
};
// jw: the warp's first column in the row (tile start + column block).
__device__ __forceinline__ void q8_load_row(Q8Row& out, const DevTensor& d, int64_t rowg, int64_t base_row,
                                            int64_t jw, int lane) {
  const int8_t* qb = d.mq + base_row + jw;
#pragma unroll
  for (int q = 0; q < kQ8PerWarp; ++q) {
    const int cl = q * 128 + lane * 4;
    out.q[q] = (jw + cl < d.W) ? *reinterpret_cast<const uint32_t*>(qb + cl) : 0u;
  }
  out.s = (lane < kQ8PerWarp && jw + lane * 128 < d.W) ? d.ms[rowg * d.qg + jw / 128 + lane] : 0.f;
}

// What a consumer thread needs of a tile before its rows: the tensor, the
// tile index within it, coef and mean(row), and the raw column / row
// statistics behind this thread's entries of the per-tile factors.
template <int NC> struct TileStats {
  static constexpr int kCols = kTileCols / (NC * 32);
  static_assert(kTileCols % (NC * 32) == 0 && kTileRows <= NC * 32, "one row factor per thread at most");
  int t;
  int64_t local;
  float coef, mr;
  float col[kCols];
  float row;
};
template <int NC>
__device__ __forceinline__ void tile_stats_load(TileStats<NC>& s, const StepArgs& a, const Range& r,
                                                const int32_t* pf, int ng, int64_t u) {
  const int m = find_owner(pf, ng, u);
  s.t = member_tensor(r, m);
  const DevTensor& d = a.tensors[s.t];
  s.local = u - pf[m];
  const TilePos tp = tile_pos(d, s.local);
  const int64_t j0 = tp.c * kTileCols, i0 = tp.r * kTileRows;
  s.coef = static_cast<float>(a.coef[s.t]);
  s.mr = static_cast<float>(a.mrow[d.mslot + tp.b]);
#pragma unroll
  for (int q = 0; q < TileStats<NC>::kCols; ++q) {
    const int64_t j = j0 + threadIdx.x + q * NC * 32;
    s.col[q] = j < d.W ? d.col[tp.b * d.W + j] : 1.f;
  }
  const int64_t i = i0 + threadIdx.x;
  s.row = (threadIdx.x < kTileRows && i < d.H) ? d.row[tp.b * d.H + i] : 1.f;
}

template <bool B1, bool Q8> struct ApplyShape {  // rows per stage, consumer warps per row
  static constexpr int kRows = (B1 && !Q8) ? 4 : kTmaRows;
  static constexpr int kSplit = Q8 ? kQ8Split : (B1 ? 2 : 1);
};
template <typename GT, bool B1, bool Q8, bool PSQ>
__global__ void __launch_bounds__(TmaCfg<ApplyShape<B1, Q8>::kSplit, ApplyShape<B1, Q8>::kRows>::kThreads, 1)
    k_apply_tma(const __grid_constant__ StepArgs a, const Range r) {
  constexpr int SPLIT = ApplyShape<B1, Q8>::kSplit;
  constexpr int RS = ApplyShape<B1, Q8>::kRows;
  constexpr int NC = TmaCfg<SPLIT, RS>::kConsumers;
  static_assert(!Q8 || B1, "the 8-bit moment needs beta1");
  static_assert(kQ8Group == 128, "a 128-column half-chunk is one 8-bit group");
  using RG = ApplyRing<GT, B1 && !Q8, RS>;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* ring = smem;
  float* colf = reinterpret_cast<float*>(smem + RG::kBytes);  // coef * col_j^-1/2
  float* rowf = colf + kTileCols;                              // (row_i / mean(row))^-1/2
  double* red = reinterpret_cast<double*>(rowf + kTileRows);  // NC <= 32 warp sums
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 32);
  uint64_t* empty = full + RG::kStages;
  int32_t* pf = reinterpret_cast<int32_t*>(empty + RG::kStages);
  __shared__ int stop;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ng = tma_setup<RG::kStages, NC>(pf, r, full, empty);
  if (warp == NC) {
    if (lane == 0) tma_produce<GT, RG>(a, r, pf, ng, ring, full, empty);
    return;
  }
  if (threadIdx.x == 0) stop = 0;
  const float b1 = static_cast<float>(a.beta1), omb1 = static_cast<float>(1.0 - a.beta1);
  const int64_t u1 = pf[ng];
  uint32_t it = 0;
  // The per-tile statistics (this thread's column and row values, coef,
  // mean(row)) are loaded one tile ahead, while the previous tile's rows are
  // processed, so a tile starts without a round trip to global memory.  Not
  // with the 8-bit moment: that variant has no registers to spare, and the
  // prefetch measured 0.3 % faster for the others but 0.5 % slower for it.
  constexpr bool kAhead = !Q8;
  TileStats<NC> next;
  if (kAhead && pf[0] + blockIdx.x < u1) tile_stats_load(next, a, r, pf, ng, pf[0] + blockIdx.x);
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    TileStats<NC> cur;
    if (kAhead) cur = next;
    else tile_stats_load(cur, a, r, pf, ng, u);
    const int t = cur.t;
    const DevTensor d = a.tensors[t];
    const TilePos tp = tile_pos(d, cur.local);
    const int64_t H = d.H, W = d.W;
    const int64_t i0 = tp.r * kTileRows, i1 = min(H, i0 + kTileRows);
    const int64_t j0 = tp.c * kTileCols;
    const int64_t base = tp.b * H * W;
    const float wda = static_cast<float>(a.wd * a.alpha[t]);
    consumer_sync<NC>();  // stop is settled; colf / rowf / red of the previous tile are read
    if (stop) break;
#pragma unroll
    for (int q = 0; q < TileStats<NC>::kCols; ++q) {
      const int cl = threadIdx.x + q * NC * 32;
      colf[cl] = (j0 + cl < W) ? cur.coef * rsqrtf(cur.col[q]) : 0.f;
    }
    if (threadIdx.x < kTileRows) rowf[threadIdx.x] = (i0 + threadIdx.x < i1) ? rsqrtf(cur.row / cur.mr) : 0.f;
    consumer_sync<NC>();
    if (kAhead && u + gridDim.x < u1) tile_stats_load(next, a, r, pf, ng, u + gridDim.x);
    float psq = 0.f;
    bool ok = true;
    const int wr = warp % RS;                                    // row of the stage
    constexpr int KW = kTileCols / 256 / SPLIT;                   // 256-column chunks per warp
    const int k0 = (warp / RS) * KW;                              // first chunk of this warp
    const int64_t jw = j0 + k0 * 256;
    Q8Row qnext;  // codes / scales of this warp's next row
    if (Q8 && i0 + wr < i1) q8_load_row(qnext, d, tp.b * H + i0 + wr, base + (i0 + wr) * W, jw, lane);
    for (int64_t rs = i0; rs < i1 && ok; rs += RS, ++it) {
      const int64_t i = rs + wr;
      Q8Row qcur;
      if (Q8) {
        qcur = qnext;
        const int64_t inext = i + RS;
        if (inext < i1) q8_load_row(qnext, d, tp.b * H + inext, base + inext * W, jw, lane);
      }
      const uint32_t slot = it % RG::kStages, ph = (it / RG::kStages) & 1u;
      if (!tma_acquire(&full[slot], ph, a, &stop)) {
        ok = false;
        break;
      }
      if (i < i1) {
        const unsigned char* row = ring + slot * RG::kStage + wr * RG::kRow;
        const float r_i = rowf[i - i0];
        float* pg = d.p + base + i * W + j0;
        float* mg = (B1 && !Q8) ? d.m1 + base + i * W + j0 : nullptr;
#pragma unroll
        for (int kk = 0; kk < KW; ++kk) {
          const int k = k0 + kk;
          if constexpr (Q8) {
            // each 128-column group: new moments, re-quantisation (the whole
            // warp, in or out of range), then p from the dequantised moments
            // (one group at a time: two at once spill under the 96-register cap)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int cl = k * 256 + h * 128 + lane * 4;
              const float gs = __shfl_sync(0xffffffffu, qcur.s, kk * 2 + h);  // old group scale
              float mq[1][4] = {{0.f, 0.f, 0.f, 0.f}}, c[1][4], sc[1];
              float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
              if (j0 + cl < W) {
                float x[4];
                quad_g<GT>(x, row, cl);
                const float4 f = *reinterpret_cast<const float4*>(colf + cl);
                pv = *reinterpret_cast<const float4*>(row + RG::kG + cl * 4);
                const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const float upd = (x[v] * r_i) * fv[v];
                  mq[0][v] = fmaf(b1, q8_value(qcur.q[kk * 2 + h], v, gs), omb1 * upd);
                }
              }
              q8_groups<1>(mq, c, sc);
              if (j0 + cl < W) {
                float* pp = &pv.x;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  pp[v] = q8_update(pp[v], wda, c[0][v], sc[0]);
                  if (PSQ) psq = fmaf(pp[v], pp[v], psq);
                }
                __stcs(reinterpret_cast<float4*>(pg + cl), pv);
                *reinterpret_cast<uint32_t*>(d.mq + base + i * W + j0 + cl) = q8_pack4(c[0]);
              }
              if (lane == 0 && j0 + k * 256 + h * 128 < W)
                d.ms[(tp.b * H + i) * d.qg + (j0 + k * 256 + h * 128) / 128] = sc[0];
            }
          } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int cl = k * 256 + h * 128 + lane * 4;
            if (j0 + cl < W) {
              float x[4];
              quad_g<GT>(x, row, cl);
              const float4 f = *reinterpret_cast<const float4*>(colf + cl);
              float4 pv = *reinterpret_cast<const float4*>(row + RG::kG + cl * 4);
              float4 mv = make_float4(0.f, 0.f, 0.f, 0.f);
              if (B1) mv = *reinterpret_cast<const float4*>(row + RG::kG + RG::kP + cl * 4);
              float* pp = &pv.x;
              float* mp = &mv.x;
              const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float upd = (x[v] * r_i) * fv[v];
                if (B1) {
                  mp[v] = fmaf(b1, mp[v], omb1 * upd);
                  upd = mp[v];
                }
                const float pn = fmaf(-wda, pp[v], pp[v] - upd);
                pp[v] = pn;
                if (PSQ) psq = fmaf(pn, pn, psq);
              }
              __stcs(reinterpret_cast<float4*>(pg + cl), pv);
              if (B1) __stcs(reinterpret_cast<float4*>(mg + cl), mv);
            }
          }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (PSQ) {
      const double tot = consumer_sum<NC>(psq, red);
      if (threadIdx.x == 0 && !stop) a.ppart[d.tile0 + cur.local] = tot;
    }
  }
  if (stop && threadIdx.x == 0) tma_drain<RG::kStages>(full, it);
}

// ---- apply of the flat class: bulk-copy staged runs of whole rows ---------
// A flat tile (whole rows [i0, i1) of one slice, W <= kTileCols) is one
// contiguous range of (i1 - i0) * W values of g, p (and exp_avg).  The
// producer streams it in spans of kTmaRows * kTileCols values into the ring
// of k_apply_tma, one copy per stream and span (a stage holds the span's g,
// then its p, then its exp_avg); consumer warp w takes piece w (kTileCols
// values) of every span.  Lane l handles the quads k*256 + h*128 + 4l of its
// piece: the quad's first (row, column) comes from its flat index
// (flat_row), the other three by stepping along the row.  A tile's copies
// stop at its last multiple of kFlatAlign<GT> values (16-byte pieces); the
// up to kFlatAlign - 1 values after that, at the end of a slice only, are
// read and written with plain loads and stores by the last piece's warp.
// A tenth warp builds each tile's factor tables (coef * col_j^-1/2,
// (row_i / mean)^-1/2) and geometry one or two tiles ahead in two table
// slots, so the consumer warps never wait on one another: each waits for
// its tile's table and its stages, and releases both.  Waits are bounded as
// in k_apply_tma.
template <typename GT> constexpr int64_t kFlatAlign = 16 / sizeof(GT);  // 4 fp32, 8 bf16 values

template <typename GT, class RG>
__device__ __forceinline__ void tma_produce_flat(const StepArgs& a, const Range& r, const int32_t* pf, int ng,
                                                 unsigned char* ring, uint64_t* full, uint64_t* empty) {
  if (a.stall_copies) return;  // testing hook: the consumers' waits run out
  constexpr int64_t kSpan = kTmaRows * kTileCols;
  const int64_t u1 = pf[ng];
  uint32_t it = 0;
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x) {
    const int m = find_owner(pf, ng, u);
    const DevTensor d = a.tensors[member_tensor(r, m)];
    const TilePos tp = tile_pos(d, u - pf[m]);
    const int64_t i0 = tp.r * kTileRows, i1 = min(d.H, i0 + kTileRows);
    const int64_t o = tp.b * d.H * d.W + i0 * d.W;
    const int64_t cnt = (i1 - i0) * d.W, cpy = cnt & ~(kFlatAlign<GT> - 1);
    const GT* g = static_cast<const GT*>(d.g) + o;
    const float* p = d.p + o;
    const float* mm = RG::kM ? d.m1 + o : nullptr;
    for (int64_t e0 = 0; e0 < cnt; e0 += kSpan, ++it) {
      const uint32_t slot = it % RG::kStages, ph = (it / RG::kStages) & 1u;
      if (!mbar_wait(&empty[slot], ph ^ 1u)) {
        atomicOr(a.status, kStatusWaitTimeout);
        return;
      }
      const int64_t e1 = min(cpy, e0 + kSpan);
      const uint32_t per_value = static_cast<uint32_t>(sizeof(GT) + (RG::kP ? 4 : 0) + (RG::kM ? 4 : 0));
      const uint32_t n = e1 > e0 ? static_cast<uint32_t>(e1 - e0) : 0u;
      mbar_arrive_expect_tx(&full[slot], n * per_value);
      unsigned char* st = ring + slot * RG::kStage;
      if (n) {
        bulk_g2s(st, g + e0, n * sizeof(GT), &full[slot]);
        if (RG::kP) bulk_g2s(st + kTmaRows * RG::kG, p + e0, n * 4, &full[slot]);
        if (RG::kM) bulk_g2s(st + kTmaRows * (RG::kG + RG::kP), mm + e0, n * 4, &full[slot]);
      }
    }
  }
}

// One flat tile's factors and geometry, built ahead by the table warp.
struct FlatTab {
  float colf[kTileCols];  // coef * col_j^-1/2
  float rowf[kTileRows];  // (row_i / mean(row))^-1/2
  double psq[kTmaRows];   // the consumer warps' sum(p_new^2) over the tile
  const void* g;
  float* p;
  float* m;
  int64_t ppart;  // the tile's entry of the sum(p^2) partials
  float wda;      // wd * alpha
  int w, cnt, cpy;
};
constexpr int kFlatTabs = 2;  // table slots
constexpr int kFlatApplyThreads = (kTmaRows + 2) * 32;  // consumers, producer warp, table warp

// The table warp: every tile of this CTA in turn, into table slot k % 2
// once the consumers released it; before refilling a slot it adds the
// consumer warps' sum(p^2) partials of the slot's previous tile in warp
// order (and those of the last tiles at the end).
template <typename GT, bool B1, bool PSQ>
__device__ __forceinline__ void flat_tables(const StepArgs& a, const Range& r, const int32_t* pf, int ng,
                                            FlatTab* tab, uint64_t* tfull, uint64_t* tempty) {
  const int lane = threadIdx.x & 31;
  const int64_t u1 = pf[ng];
  uint32_t k = 0;
  auto flush = [&](const FlatTab& T) {
    if (PSQ && lane == 0) {
      double tot = 0.0;
#pragma unroll
      for (int v = 0; v < kTmaRows; ++v) tot += T.psq[v];
      a.ppart[T.ppart] = tot;
    }
  };
  for (int64_t u = pf[0] + blockIdx.x; u < u1; u += gridDim.x, ++k) {
    const uint32_t s = k % kFlatTabs, ph = (k / kFlatTabs) & 1u;
    if (!mbar_wait(&tempty[s], ph ^ 1u)) {
      if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
      return;
    }
    FlatTab& T = tab[s];
    if (k >= kFlatTabs) flush(T);
    __syncwarp();
    const int m = find_owner(pf, ng, u);
    const int t = member_tensor(r, m);
    const DevTensor* d = a.tensors + t;
    const int64_t local = u - pf[m];
    const TilePos tp = tile_pos(*d, local);
    const int64_t H = d->H, W = d->W;
    const int64_t i0 = tp.r * kTileRows, i1 = min(H, i0 + kTileRows);
    const int64_t o = tp.b * H * W + i0 * W;
    const float coef = static_cast<float>(a.coef[t]);
    const float mr = static_cast<float>(a.mrow[d->mslot + tp.b]);
    const float* col = d->col + tp.b * W;
    const float* row = d->row + tp.b * H + i0;
    // all of the lane's loads first, so they are in flight together
    float cv[kTileCols / 32], rv[kTileRows / 32];
#pragma unroll
    for (int q = 0; q < kTileCols / 32; ++q) {
      const int j = lane + 32 * q;
      cv[q] = j < W ? col[j] : 1.f;
    }
#pragma unroll
    for (int q = 0; q < kTileRows / 32; ++q) {
      const int i = lane + 32 * q;
      rv[q] = i0 + i < i1 ? row[i] : 1.f;
    }
#pragma unroll
    for (int q = 0; q < kTileCols / 32; ++q) {
      const int j = lane + 32 * q;
      T.colf[j] = j < W ? coef * rsqrtf(cv[q]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kTileRows / 32; ++q) {
      const int i = lane + 32 * q;
      T.rowf[i] = i0 + i < i1 ? rsqrtf(rv[q] / mr) : 0.f;
    }
    if (lane == 0) {
      T.g = static_cast<const GT*>(d->g) + o;
      T.p = d->p + o;
      T.m = B1 ? d->m1 + o : nullptr;
      T.ppart = d->tile0 + local;
      T.wda = static_cast<float>(a.wd * a.alpha[t]);
      T.w = static_cast<int>(W);
      T.cnt = static_cast<int>((i1 - i0) * W);  // at most kTileRows * kTileCols
      T.cpy = T.cnt & ~static_cast<int>(kFlatAlign<GT> - 1);
    }
    mbar_arrive(&tfull[s]);  // every lane (count 32): its own writes are released
  }
  // the partials of the last tiles
  for (uint32_t q = k > kFlatTabs ? k - kFlatTabs : 0; q < k; ++q) {
    const uint32_t s = q % kFlatTabs, ph = (q / kFlatTabs) & 1u;
    if (!mbar_wait(&tempty[s], ph)) {
      if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
      return;
    }
    flush(tab[s]);
  }
}

template <typename GT, bool B1, bool PSQ>
__global__ void __launch_bounds__(kFlatApplyThreads, 1)
    k_apply_tma_flat(const __grid_constant__ StepArgs a, const Range r) {
  constexpr int NC = kTmaRows;  // consumer warps, one piece of a span each
  constexpr int64_t kSpan = kTmaRows * kTileCols;
  using RG = ApplyRing<GT, B1>;
  static_assert(RG::kP == kTileCols * 4 && (!B1 || RG::kM == RG::kP), "stage layout: g, p, exp_avg blocks");
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* ring = smem;
  FlatTab* tab = reinterpret_cast<FlatTab*>(smem + RG::kBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(tab + kFlatTabs);
  uint64_t* empty = full + RG::kStages;
  uint64_t* tfull = empty + RG::kStages;
  uint64_t* tempty = tfull + kFlatTabs;
  int32_t* pf = reinterpret_cast<int32_t*>(tempty + kFlatTabs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ng = load_prefix(pf, r);
  if (threadIdx.x == 0) {
    for (int s = 0; s < RG::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    for (int s = 0; s < kFlatTabs; ++s) {
      mbar_init(&tfull[s], 32);
      mbar_init(&tempty[s], NC);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == NC) {
    if (lane == 0) tma_produce_flat<GT, RG>(a, r, pf, ng, ring, full, empty);
    return;
  }
  if (warp == NC + 1) {
    flat_tables<GT, B1, PSQ>(a, r, pf, ng, tab, tfull, tempty);
    return;
  }
  const float b1 = static_cast<float>(a.beta1), omb1 = static_cast<float>(1.0 - a.beta1);
  const int64_t u1 = pf[ng];
  uint32_t it = 0, k = 0;
  bool ok = true;
  for (int64_t u = pf[0] + blockIdx.x; u < u1 && ok; u += gridDim.x, ++k) {
    const uint32_t ts = k % kFlatTabs, tph = (k / kFlatTabs) & 1u;
    if (!mbar_wait(&tfull[ts], tph)) {
      if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
      ok = false;
      break;
    }
    const FlatTab& T = tab[ts];
    const float* colf = T.colf;
    const float* rowf = T.rowf;
    const int cnt = T.cnt, cpy = T.cpy, w = T.w;
    const float invw = 1.0f / static_cast<float>(w);
    const float wda = T.wda;
    const GT* gt = static_cast<const GT*>(T.g);
    float* pt = T.p;
    float* mt = T.m;
    float psq = 0.f;
    for (int e0 = 0; e0 < cnt; e0 += static_cast<int>(kSpan), ++it) {
      const uint32_t slot = it % RG::kStages, ph = (it / RG::kStages) & 1u;
      if (!mbar_wait(&full[slot], ph)) {
        if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
        ok = false;
        break;
      }
      const int s0 = e0 + warp * kTileCols;  // this warp's piece
      if (s0 < cnt) {
        const unsigned char* st = ring + slot * RG::kStage;
        const unsigned char* gs = st + warp * RG::kG;                                   // this piece's g
        const unsigned char* ps = st + kTmaRows * RG::kG + warp * RG::kP;                // its p
        const unsigned char* ms = st + kTmaRows * (RG::kG + RG::kP) + warp * RG::kP;     // its exp_avg
        const int nc = s0 < cpy ? min(kTileCols, cpy - s0) : 0;  // staged values (whole quads)
#pragma unroll
        for (int kk = 0; kk < kTileCols / 256; ++kk) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int cl = kk * 256 + h * 128 + lane * 4;
            if (cl < nc) {
              float x[4];
              quad_g<GT>(x, gs, cl);
              float4 pv = *reinterpret_cast<const float4*>(ps + cl * 4);
              float4 mv = make_float4(0.f, 0.f, 0.f, 0.f);
              if (B1) mv = *reinterpret_cast<const float4*>(ms + cl * 4);
              float* pp = &pv.x;
              float* mp = &mv.x;
              const int e = s0 + cl;
              int i = flat_row(e, invw), j = e - i * w;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float upd = (x[v] * rowf[i]) * colf[j];
                if (B1) {
                  mp[v] = fmaf(b1, mp[v], omb1 * upd);
                  upd = mp[v];
                }
                const float pn = fmaf(-wda, pp[v], pp[v] - upd);
                pp[v] = pn;
                if (PSQ) psq = fmaf(pn, pn, psq);
                flat_next(i, j, w);
              }
              __stcs(reinterpret_cast<float4*>(pt + e), pv);
              if (B1) __stcs(reinterpret_cast<float4*>(mt + e), mv);
            }
          }
        }
        // values past the last 16-byte piece of the tile (end of a slice)
        const int e = s0 + nc + lane;
        if (nc < kTileCols && e < cnt && e >= cpy) {
          const int i = flat_row(e, invw), j = e - i * w;
          float upd = (load_g_scalar<GT>(gt + e) * rowf[i]) * colf[j];
          if (B1) {
            const float mn = fmaf(b1, mt[e], omb1 * upd);
            mt[e] = mn;
            upd = mn;
          }
          const float pv = pt[e];
          const float pn = fmaf(-wda, pv, pv - upd);
          pt[e] = pn;
          if (PSQ) psq = fmaf(pn, pn, psq);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (!ok) break;
    if (PSQ) {
      const float ws = warp_sum(psq);
      if (lane == 0) tab[ts].psq[warp] = static_cast<double>(ws);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tempty[ts]);  // the tile's tables are read
  }
  if (!ok && threadIdx.x == 0) tma_drain<RG::kStages>(full, it);
}

// ---- psq: sum(p_new^2) carry, one CTA per tensor --------------------------
__global__ void __launch_bounds__(kThreads) k_psq(const __grid_constant__ StepArgs a) {
  __shared__ double red[16];
  const int t = blockIdx.x;
  const DevTensor d = a.tensors[t];
  if (d.psq == nullptr) return;
  double acc = 0.0;
  for (int64_t k = threadIdx.x; k < d.ntiles; k += kThreads) acc += a.ppart[d.tile0 + k];
  const double S = block_sum(acc, red);
  if (threadIdx.x == 0) *d.psq = S;
}

}  // namespace

const char* kernel_name(int k) {
  static const char* names[kNumKernels] = {"k_pass1", "k_stats", "k_scalars", "k_pass2",
                                           "k_clip", "k_apply", "k_psq"};
  return (k >= 0 && k < kNumKernels) ? names[k] : "";
}

namespace {

// Dynamic shared memory of the bulk-copy kernels: ring, per-tile factors or
// column buffer, reduction scratch, mbarriers, prefix.
template <class RG>
constexpr size_t tma_smem(size_t extra) {
  return RG::kBytes + extra + sizeof(double) * 32 + sizeof(uint64_t) * 2 * RG::kStages + kPrefixBytes;
}
constexpr size_t kFactorBytes = sizeof(float) * (kTileCols + kTileRows);
// k_apply_tma_flat: ring, table slots, mbarriers (stages and tables), prefix.
template <class RG>
constexpr size_t flat_apply_smem() {
  return RG::kBytes + sizeof(FlatTab) * kFlatTabs + sizeof(uint64_t) * 2 * (RG::kStages + kFlatTabs) + kPrefixBytes;
}

using KernelFn = void (*)(StepArgs, Range);

// One launchable instantiation: function, block size, dynamic shared memory.
struct Inst {
  KernelFn fn = nullptr;
  int threads = kThreads;
  size_t smem = 0;
};

template <typename GT, int VEC>
Inst pick_f(KernelId k, bool psq_in, int mom, bool psq_out) {
  const bool b1 = mom != 0;
  Inst x;
  switch (k) {
    case kKPass1:
      x.fn = psq_in ? k_pass1_f<GT, VEC, true> : k_pass1_f<GT, VEC, false>;
      x.smem = kColbufBytes + kRedBytes + kPrefixBytes;
      return x;
    case kKPass2:
      x.fn = k_pass2_f<GT, VEC>;
      x.smem = kRedBytes + kPrefixBytes + kColfBytes + kRowfBytes;
      return x;
    case kKApply:
      if constexpr (VEC == 8) {  // vector path: bulk-copy staged rows
        if (mom == 2) {
          x.threads = TmaCfg<ApplyShape<true, true>::kSplit, ApplyShape<true, true>::kRows>::kThreads;
          x.fn = psq_out ? k_apply_tma<GT, true, true, true> : k_apply_tma<GT, true, true, false>;
          x.smem = tma_smem<ApplyRing<GT, false, ApplyShape<true, true>::kRows>>(kFactorBytes);
        } else if (b1) {
          x.threads = TmaCfg<ApplyShape<true, false>::kSplit, ApplyShape<true, false>::kRows>::kThreads;
          x.fn = psq_out ? k_apply_tma<GT, true, false, true> : k_apply_tma<GT, true, false, false>;
          x.smem = tma_smem<ApplyRing<GT, true, ApplyShape<true, false>::kRows>>(kFactorBytes);
        } else {
          x.threads = TmaCfg<1>::kThreads;
          x.fn = psq_out ? k_apply_tma<GT, false, false, true> : k_apply_tma<GT, false, false, false>;
          x.smem = tma_smem<ApplyRing<GT, false>>(kFactorBytes);
        }
        return x;
      } else {
        if (mom == 2) x.fn = psq_out ? k_apply_f<GT, VEC, true, true, true> : k_apply_f<GT, VEC, true, true, false>;
        else if (b1) x.fn = psq_out ? k_apply_f<GT, VEC, true, false, true> : k_apply_f<GT, VEC, true, false, false>;
        else x.fn = psq_out ? k_apply_f<GT, VEC, false, false, true> : k_apply_f<GT, VEC, false, false, false>;
        x.smem = kRedBytes + kPrefixBytes + kColfBytes + (VEC == 1 ? kRowfBytes : 0);
        return x;
      }
    default: return x;
  }
}

// Fused pass 1 (NW warps, G column groups per lane) and the bulk-copy apply
// of the row-chunk classes.
template <typename GT, int NW, int G, int S, int MINB>
Inst pick_rows(KernelId k, bool psq_in, int mom, bool psq_out) {
  Inst x;
  if (k == kKPass1) {
    x.fn = psq_in ? k_pass1_panel<GT, NW, G, S, MINB, true> : k_pass1_panel<GT, NW, G, S, MINB, false>;
    x.threads = NW * 32;
    x.smem = PanelCfg<GT, NW, G, S>::kSmem;
  } else if (k == kKApply) {
    x = pick_f<GT, 8>(k, psq_in, mom, psq_out);
  }
  return x;
}

// The flat class: fused flat pass 1, no pass 2, the bulk-copy flat apply
// (the element-wise apply, row by row, with the 8-bit moment).
template <typename GT>
Inst pick_flat(KernelId k, bool psq_in, int mom, bool psq_out) {
  Inst x;
  if (k == kKPass1) {
    x.fn = psq_in ? k_pass1_flat<GT, true> : k_pass1_flat<GT, false>;
    x.threads = kFlatThreads;
    x.smem = kFlatSmem;
  } else if (k == kKApply) {
    if (mom == 2) return pick_f<GT, 1>(k, psq_in, mom, psq_out);
    x.threads = kFlatApplyThreads;
    if (mom == 1) {
      x.fn = psq_out ? k_apply_tma_flat<GT, true, true> : k_apply_tma_flat<GT, true, false>;
      x.smem = flat_apply_smem<ApplyRing<GT, true>>();
    } else {
      x.fn = psq_out ? k_apply_tma_flat<GT, false, true> : k_apply_tma_flat<GT, false, false>;
      x.smem = flat_apply_smem<ApplyRing<GT, false>>();
    }
  }
  return x;
}

// mom: first moment none (0), fp32 exp_avg (1), 8-bit codes + scales (2).
Inst pick(KernelId k, TensorClass c, bool psq_in, int mom, bool psq_out) {
  Inst x;
  switch (c) {
    case kClsVecBF16: return pick_f<__nv_bfloat16, 8>(k, psq_in, mom, psq_out);
    case kClsVecF32: return pick_f<float, 8>(k, psq_in, mom, psq_out);
    case kClsScalarBF16: return pick_f<__nv_bfloat16, 1>(k, psq_in, mom, psq_out);
    case kClsScalarF32: return pick_f<float, 1>(k, psq_in, mom, psq_out);
    case kClsRowsBF16: return pick_rows<__nv_bfloat16, kRowsNW, kRowsG, kRowsS, kRowsMinB>(k, psq_in, mom, psq_out);
    case kClsWideBF16: return pick_rows<__nv_bfloat16, 14, 4, 4, 1>(k, psq_in, mom, psq_out);
    case kClsFlatBF16: return pick_flat<__nv_bfloat16>(k, psq_in, mom, psq_out);
    case kClsFlatF32: return pick_flat<float>(k, psq_in, mom, psq_out);
    case kClsUnfactored:
      x.smem = kRedBytes + kPrefixBytes;
      if (k == kKPass1) x.fn = psq_in ? k_pass1_u<true> : k_pass1_u<false>;
      if (k == kKApply) {
        if (mom == 2) x.fn = psq_out ? k_apply_u<true, true, true> : k_apply_u<true, true, false>;
        else if (mom == 1) x.fn = psq_out ? k_apply_u<true, false, true> : k_apply_u<true, false, false>;
        else x.fn = psq_out ? k_apply_u<false, false, true> : k_apply_u<false, false, false>;
      }
      return x;
    default: return x;
  }
}

}  // namespace

int kernel_variant(const StepArgs& a) {
  const int psq_in = (a.scale_parameter && !a.psq_valid) ? 1 : 0;
  const int mom = a.has_beta1 ? (a.q8 ? 2 : 1) : 0;
  return psq_in + 2 * mom + (a.want_psq_out != 0 ? 6 : 0);
}

int kernel_grid_limit(KernelId k, TensorClass c, int variant, int device, cudaError_t* err) {
  // (resident CTAs per SM) x SM count of the instantiation that (kind, class,
  // variant) launches, cached per device.  Also raises the dynamic
  // shared-memory limit of that instantiation where it needs more than the
  // 48 KB default.
  constexpr int kMaxDev = 64, kVariants = 12;
  static int cache[kMaxDev][kNumKernels][kNumClasses][kVariants] = {};
  *err = cudaSuccess;
  if (device < 0 || device >= kMaxDev || variant < 0 || variant >= kVariants) {
    *err = device < 0 || device >= kMaxDev ? cudaErrorInvalidDevice : cudaErrorInvalidValue;
    return 0;
  }
  if (cache[device][k][c][variant] > 0) return cache[device][k][c][variant];
  int sms = 0;
  *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (*err != cudaSuccess) return 0;
  int per_sm = 1 << 30;
  auto visit = [&](const void* fn, int threads, size_t smem) {
    if (*err != cudaSuccess || fn == nullptr) return;
    if (smem > 48 * 1024) {
      *err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (*err != cudaSuccess) return;
    }
    int b = 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem);
    if (*err == cudaSuccess && b < per_sm) per_sm = b;
  };
  if (k == kKPass1 || k == kKPass2 || k == kKApply) {
    const Inst x = pick(k, c, variant & 1, (variant >> 1) % 3, variant >= 6);
    visit(reinterpret_cast<const void*>(x.fn), x.threads, x.smem);
  } else if (k == kKStats) {
    visit(reinterpret_cast<const void*>(k_stats), kThreads, kRedBytes + kPrefixBytes + kPartBytes);
  } else {
    per_sm = 8;  // per-tensor kernels: grid = tensor count, not limited here
  }
  if (*err != cudaSuccess) return 0;
  if (per_sm < 1) per_sm = 1;
  if (per_sm == (1 << 30)) per_sm = 1;
  cache[device][k][c][variant] = per_sm * sms;
  return cache[device][k][c][variant];
}

cudaError_t launch_stream(KernelId k, TensorClass c, const StepArgs& a, const Range& r, int grid,
                          cudaStream_t s) {
  if (grid <= 0 || r.m_end <= r.m_begin) return cudaSuccess;
  const int v = kernel_variant(a);
  const Inst x = pick(k, c, v & 1, (v >> 1) % 3, v >= 6);
  if (x.fn == nullptr) return cudaErrorInvalidValue;
  x.fn<<<grid, x.threads, x.smem, s>>>(a, r);
  return cudaGetLastError();
}

cudaError_t launch_stats(const StepArgs& a, const Range& r, int grid, cudaStream_t s) {
  if (grid <= 0 || r.m_end <= r.m_begin) return cudaSuccess;
  k_stats<<<grid, kThreads, kRedBytes + kPrefixBytes + kPartBytes, s>>>(a, r);
  return cudaGetLastError();
}

cudaError_t launch_per_tensor(KernelId k, const StepArgs& a, int ntensors, cudaStream_t s) {
  if (ntensors <= 0) return cudaSuccess;
  switch (k) {
    case kKScalars: k_scalars<<<ntensors, kThreads, 0, s>>>(a); break;
    case kKClip: k_clip<<<ntensors, kThreads, 0, s>>>(a); break;
    case kKPsq: k_psq<<<ntensors, kThreads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace meo
