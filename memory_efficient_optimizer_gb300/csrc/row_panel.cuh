// Fused statistics pass over chunks of full rows, shared by the Adafactor
// step (k_pass1_panel) and the CAME step (k_came_panel).
//
// Both rules factor the second moment of an [H, W] slice into a row
// statistic r_i (an EMA of the row means of g^2 + eps1) and a column
// statistic c_j, and both need sum(u^2) = sum_ij g_ij^2 mean(r) / (r_i c_j)
// for the RMS clip (Colossal-AI distributed-optimizer article, Step 5 for
// Adafactor; the DistributedCAME paragraph for CAME).  Written as
//   sum(u^2) = mean(r) * sum_j D_j / c_j,   D_j = sum_i g_ij^2 / r_i,
// D_j can be accumulated in the same read of g as the statistics, as long as
// r_i is known while the row's values are still on chip: a CTA takes whole
// rows.  g is then read from HBM once for the statistics and sum(u^2)
// instead of twice.
//
// A work unit is a chunk of full rows [c0, c1) of one slice, taken by one CTA
// of NW warps in sub-panels of SR rows (32 / NW for NW <= 8, else 2).  Lane l of warp w owns the
// column groups c * NW + w (c < G) of 256 columns, 8 consecutive columns
// (256 (c NW + w) + 8 l + [0, 8)) in each, and keeps their column sums C_j
// and D_j in registers.
//
// Staging: every lane copies its own 16-byte pieces of each sub-panel into
// its own shared-memory slots with cp.async (completion tracked per thread by
// commit/wait groups: no spin loop, no mbarrier).  A ring of S sub-panels
// per CTA keeps S - 1 sub-panels in flight while one is processed, so the
// bytes in flight do not cost registers, and the second use of the values
// (phase B) reads shared memory instead of L2 or HBM.  Since a lane only ever
// reads the slots it filled, the staged data needs no barrier.
// Per sub-panel k:
//   wait for this thread's copies of sub-panel k;
//   A. add the squares into C_j; the warp's share of each row total goes to
//      shared memory (one reduce-scatter over the lanes covers the SR rows);
//   -- barrier -- (row shares complete; every lane has finished sub-panel
//      k - 1, whose stage is refilled now with sub-panel k + S - 1)
//   every warp sums the NW shares of each row (lane l: row l / NW, warp
//   l % NW) and forms r = b2 r + (1 - b2)(sum_j g_rj^2 / W + eps1) and its
//   reciprocal; warp 0 stores r;
//   B. add g_rj^2 / r into D_j from the same staged values.
// Per chunk the warps write C_j and D_j (column partials of the chunk), and
// warp 0 accumulates sum_r r (for mean(r)).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace meo {
namespace panel {

// Shared-memory ring: per stage and warp, slot ((rr * G + c) * kPieces + q)
// * 32 + lane holds 16 bytes (piece q of the 8 values of row rr, column
// group c, lane), so every warp-wide copy and read touches 512 contiguous
// bytes.  After the ring: the row shares [2][32] floats (kPartOff).
template <typename GT, int NW, int G, int S> struct Cfg {
  static constexpr int kSubRows = NW <= 8 ? 32 / NW : 2;
  // a warp's total of row r is complete in lane r * kShareLanes after row_shares
  static constexpr int kShareLanes = 32 / kSubRows;
  static constexpr int kPieces = static_cast<int>(sizeof(GT)) / 2;  // 16-byte pieces per 8 values
  static constexpr int kWarpBytes = kSubRows * G * kPieces * 32 * 16;
  static constexpr int kStageBytes = kWarpBytes * NW;
  static constexpr size_t kPartOff = static_cast<size_t>(S) * kStageBytes;
  static constexpr size_t kBytes = kPartOff + sizeof(float) * 2 * 32;  // ring + row shares
  static_assert(kSubRows * NW <= 32 && kShareLanes * kSubRows == 32 && (kSubRows == 2 || kSubRows == 4),
                "the row statistics take at most one (row, warp) share per lane");
  static_assert(S >= 2, "the ring needs the stage in use and one in flight");
};

// 16-byte asynchronous global -> shared copy (bypasses L1).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// 4-byte asynchronous global -> shared copy (the 4-byte form goes through L1).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

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

// This lane's copies of rows [q0, min(q0 + SR, q1)) into its slots of one
// stage (dst: shared address of the lane's first slot in that stage).  FULL:
// all SR rows and all of the lane's column groups are in range.
template <bool FULL, typename GT, int NW, int G, int S>
__device__ __forceinline__ void issue(uint32_t dst, const GT* gb, int32_t W, int32_t q0, int32_t q1, int warp,
                                      int lane) {
  using C = Cfg<GT, NW, G, S>;
  constexpr int P = C::kPieces;
  const GT* src0 = gb + static_cast<int64_t>(q0) * W + warp * 256 + lane * 8;
#pragma unroll
  for (int rr = 0; rr < C::kSubRows; ++rr) {
#pragma unroll
    for (int c = 0; c < G; ++c) {
      const int32_t j = (c * NW + warp) * 256 + lane * 8;
      if (FULL || (q0 + rr < q1 && j < W)) {
        const GT* src = src0 + static_cast<int64_t>(rr) * W + c * NW * 256;
#pragma unroll
        for (int q = 0; q < P; ++q)
          cp_async16(dst + ((rr * G + c) * P + q) * 512, src + q * (16 / static_cast<int>(sizeof(GT))));
      }
    }
  }
}

// The 8 bf16 values of one slot as 4 pairs (bf16 -> fp32 is exact: the bf16
// bits are the high half of the fp32 bits), for the paired fp32 instructions.
__device__ __forceinline__ void read_pairs(float2 (&x)[4], const unsigned char* slot) {
  const uint4 u = *reinterpret_cast<const uint4*>(slot);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) x[k] = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
}

// Reduce-scatter of 4 per-lane values over the warp: afterwards lane l holds
// the warp total of value ((l >> 4) & 1) * 2 + ((l >> 3) & 1), complete in
// lanes 0, 8, 16, 24.  Fixed exchange pattern, so the sums are deterministic.
__device__ __forceinline__ float reduce_scatter4(const float (&v)[4], int lane) {
  const bool h16 = lane & 16, h8 = lane & 8;
  float k0 = h16 ? v[2] : v[0], k1 = h16 ? v[3] : v[1];
  const float s0 = h16 ? v[0] : v[2], s1 = h16 ? v[1] : v[3];
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  float k = h8 ? k1 : k0;
  const float s = h8 ? k0 : k1;
  k += __shfl_xor_sync(0xffffffffu, s, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}
// Two-row version: lane l gets the warp total of value l >> 4 (complete in
// lanes 0 and 16).
__device__ __forceinline__ float reduce_scatter2(const float (&v)[2], int lane) {
  const bool h16 = lane & 16;
  float k = h16 ? v[1] : v[0];
  k += __shfl_xor_sync(0xffffffffu, h16 ? v[0] : v[1], 16);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
  return k;
}
__device__ __forceinline__ float row_shares(const float (&v)[4], int lane) { return reduce_scatter4(v, lane); }
__device__ __forceinline__ float row_shares(const float (&v)[2], int lane) { return reduce_scatter2(v, lane); }

// CTA-wide sum over NW warps in a fixed order (red: NW + 1 doubles); every
// thread gets the result.
template <int NW>
__device__ __forceinline__ double block_sum(double v, double* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += red[w];
    red[NW] = s;
  }
  __syncthreads();
  const double s = red[NW];
  __syncthreads();
  return s;
}

// Phase A over the staged values of one sub-panel: squares into C_j and this
// warp's share of each row total (rp); with PSQ also sum(p^2) of the same
// elements, read from pb.  FULL: every row of the sub-panel and every column
// group of the lane is in range, so no per-element predicates.  x^2 is exact
// in fp32 for a bf16 x, so fma(x, x, acc) equals acc + x * x.
template <bool FULL, typename GT, int NW, int G, int S, bool PSQ>
__device__ __forceinline__ void phase_a(const unsigned char* st, int32_t s0, int32_t s1, int32_t W, int warp,
                                        int lane, const float* pb, float2 (&cacc)[G][4], float (&rp)[32 / NW],
                                        float& psq) {
  constexpr int SR = 32 / NW, P = Cfg<GT, NW, G, S>::kPieces;
#pragma unroll
  for (int rr = 0; rr < SR; ++rr) {
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < G; ++c) {
      const int32_t j = (c * NW + warp) * 256 + lane * 8;
      if (FULL || (s0 + rr < s1 && j < W)) {
        float2 x[4];
        read_pairs(x, st + (rr * G + c) * P * 512);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          cacc[c][v] = __ffma2_rn(x[v], x[v], cacc[c][v]);
          s2 = __ffma2_rn(x[v], x[v], s2);
        }
        if (PSQ) {
          const float* py = pb + static_cast<int64_t>(s0 + rr) * W + j;
          const float4 ya = __ldcs(reinterpret_cast<const float4*>(py));
          const float4 yb = __ldcs(reinterpret_cast<const float4*>(py) + 1);
          const float y[8] = {ya.x, ya.y, ya.z, ya.w, yb.x, yb.y, yb.z, yb.w};
#pragma unroll
          for (int v = 0; v < 8; ++v) psq = fmaf(y[v], y[v], psq);
        }
      }
    }
    rp[rr] = s2.x + s2.y;
  }
}

// Phase B: g^2 / r into D_j (lane rr * NW holds 1 / r of row rr).
template <bool FULL, typename GT, int NW, int G, int S>
__device__ __forceinline__ void phase_b(const unsigned char* st, int32_t s0, int32_t s1, int32_t W, int warp,
                                        int lane, float winv, float2 (&dacc)[G][4]) {
  constexpr int SR = 32 / NW, P = Cfg<GT, NW, G, S>::kPieces;
#pragma unroll
  for (int rr = 0; rr < SR; ++rr) {
    const float wr = __shfl_sync(0xffffffffu, winv, rr * NW);
    const float2 w2 = make_float2(wr, wr);
#pragma unroll
    for (int c = 0; c < G; ++c) {
      const int32_t j = (c * NW + warp) * 256 + lane * 8;
      if (FULL || (s0 + rr < s1 && j < W)) {
        float2 x[4];
        read_pairs(x, st + (rr * G + c) * P * 512);
#pragma unroll
        for (int v = 0; v < 4; ++v) dacc[c][v] = __ffma2_rn(__fmul2_rn(x[v], w2), x[v], dacc[c][v]);
      }
    }
  }
}

// Where a chunk's column partials go: C_j to cp[0, W), D_j to dp[0, W).
struct Partials {
  float* cp;
  float* dp;
};

// One chunk of rows [c0, c1) of one slice (gb: the slice's gradient, pb its
// parameter, read only with PSQ; rowst: the slice's row statistic, updated in
// place).  Writes the chunk's column partials to where(), a callable that
// returns a Partials (evaluated after the rows, so that its operands need not
// stay in registers through the loop).  On return rsum holds, in lanes
// l % NW == 0 of warp 0, this thread's part of sum_r r over the chunk (0
// elsewhere), and psq this thread's part of sum(p^2); the caller adds them
// over the CTA.  smem: the ring and row shares of Cfg (kBytes).  Every
// thread of the CTA must call; the next call may follow directly (the
// caller's CTA barrier, e.g. the one in block_sum, separates this chunk's
// last reads of the ring from the next chunk's first copies).
template <typename GT, int NW, int G, int S, bool PSQ, typename Where>
__device__ __forceinline__ void run_chunk(unsigned char* smem, const GT* gb, const float* pb, float* rowst,
                                          int32_t W, int32_t c0, int32_t c1, float b2, float omb2, float eps1,
                                          Where&& where, float& rsum, float& psq) {
  using C = Cfg<GT, NW, G, S>;
  constexpr int SR = C::kSubRows;
  float* part = reinterpret_cast<float*>(smem + C::kPartOff);  // [2][SR][NW]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned char* mine = smem + warp * C::kWarpBytes + lane * 16;
  const uint32_t mine_s = static_cast<uint32_t>(__cvta_generic_to_shared(mine));
  const int rl = lane / NW;  // row of this lane's (row, warp) share
  const int32_t nsub = (c1 - c0 + SR - 1) / SR;
  const float invw = 1.0f / static_cast<float>(W);
  float2 cacc[G][4], dacc[G][4];
#pragma unroll
  for (int c = 0; c < G; ++c) {
#pragma unroll
    for (int v = 0; v < 4; ++v) cacc[c][v] = dacc[c][v] = make_float2(0.f, 0.f);
  }
  rsum = 0.f;
  // Prologue: sub-panels 0 .. S - 2 (one commit group each, empty past the
  // chunk's end, so the group count stays in step).
#pragma unroll
  for (int k = 0; k < S - 1; ++k) {
    if (k < nsub) issue<false, GT, NW, G, S>(mine_s + k * C::kStageBytes, gb, W, c0 + k * SR, c1, warp, lane);
    cp_async_commit();
  }
  // Column groups of this warp all inside the row (warp-uniform).
  const bool cols_full = ((G - 1) * NW + warp + 1) * 256 <= W;
  int stage = 0;
  for (int32_t k = 0; k < nsub; ++k) {
    const int32_t s0 = c0 + k * SR, s1 = min(c1, s0 + SR);
    const bool full = cols_full && s1 - s0 == SR;
    const float row_old = (s0 + rl < s1) ? rowst[s0 + rl] : 0.f;
    cp_async_wait<S - 2>();  // groups up to sub-panel k are complete
    const unsigned char* st = mine + stage * C::kStageBytes;
    float* pk = part + (k & 1) * 32;
    float rp[SR];
    if (full) phase_a<true, GT, NW, G, S, PSQ>(st, s0, s1, W, warp, lane, pb, cacc, rp, psq);
    else phase_a<false, GT, NW, G, S, PSQ>(st, s0, s1, W, warp, lane, pb, cacc, rp, psq);
    const float tot = row_shares(rp, lane);  // warp total of row lane / kShareLanes
    if (lane % C::kShareLanes == 0) pk[(lane / C::kShareLanes) * NW + warp] = tot;
    __syncthreads();
    // Refill the stage of sub-panel k - 1 (every lane is past it) with k + S - 1.
    {
      const int32_t kk = k + S - 1;
      const int fill = stage == 0 ? S - 1 : stage - 1;
      if (kk < nsub) {
        if (cols_full && c0 + (kk + 1) * SR <= c1)
          issue<true, GT, NW, G, S>(mine_s + fill * C::kStageBytes, gb, W, c0 + kk * SR, c1, warp, lane);
        else
          issue<false, GT, NW, G, S>(mine_s + fill * C::kStageBytes, gb, W, c0 + kk * SR, c1, warp, lane);
      }
      cp_async_commit();
    }
    // Row statistics of the sub-panel, in every warp: lane l adds the shares
    // of row l / NW over the warps (a fixed xor tree where SR * NW = 32, else
    // in warp order; lanes past SR * NW hold no row).
    float R = 0.f;
    if constexpr (SR * NW == 32) {
      R = pk[lane];
#pragma unroll
      for (int o = NW / 2; o > 0; o >>= 1) R += __shfl_xor_sync(0xffffffffu, R, o);
    } else {
      if (rl < SR) {
#pragma unroll
        for (int w = 0; w < NW; ++w) R += pk[rl * NW + w];
      }
    }
    const float rn = fmaf(b2, row_old, omb2 * fmaf(R, invw, eps1));
    const float winv = __frcp_rn(rn);  // correctly rounded 1 / rn
    if (warp == 0 && lane % NW == 0 && s0 + rl < s1) {
      rowst[s0 + rl] = rn;
      rsum += rn;
    }
    if (full) phase_b<true, GT, NW, G, S>(st, s0, s1, W, warp, lane, winv, dacc);
    else phase_b<false, GT, NW, G, S>(st, s0, s1, W, warp, lane, winv, dacc);
    stage = stage == S - 1 ? 0 : stage + 1;
  }
  // column partials of the chunk
  const Partials out = where();
  float* cp = out.cp;
  float* dp = out.dp;
#pragma unroll
  for (int c = 0; c < G; ++c) {
    const int32_t j = (c * NW + warp) * 256 + lane * 8;
    if (j < W) {
      *reinterpret_cast<float4*>(cp + j) = make_float4(cacc[c][0].x, cacc[c][0].y, cacc[c][1].x, cacc[c][1].y);
      *reinterpret_cast<float4*>(cp + j + 4) = make_float4(cacc[c][2].x, cacc[c][2].y, cacc[c][3].x, cacc[c][3].y);
      *reinterpret_cast<float4*>(dp + j) = make_float4(dacc[c][0].x, dacc[c][0].y, dacc[c][1].x, dacc[c][1].y);
      *reinterpret_cast<float4*>(dp + j + 4) = make_float4(dacc[c][2].x, dacc[c][2].y, dacc[c][3].x, dacc[c][3].y);
    }
  }
}

}  // namespace panel
}  // namespace meo
