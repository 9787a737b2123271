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
//
// Split form (rings of S >= 4 stages, run_chunk_split): the CTA barrier is
// replaced by an mbarrier per sub-panel that the lanes holding row shares
// arrive on after phase A, and the warps wait on it only one sub-panel later:
// iteration k runs phase A of sub-panel k, then the row statistics and phase
// B of sub-panel k - 1.  A warp that is ahead no longer stops at every
// sub-panel for the slowest one; it waits only when it is a whole phase
// ahead.  Two sub-panels are in use per lane (k and k - 1), so the ring needs
// a fourth stage to keep two in flight.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "adafactor_internal.h"

namespace meo {
namespace panel {

// Shared-memory ring: per stage and warp, slot ((rr * G + c) * kPieces + q)
// * 32 + lane holds 16 bytes (piece q of the 8 values of row rr, column
// group c, lane), so every warp-wide copy and read touches 512 contiguous
// bytes.  After the ring: the row shares, kShareBufs buffers of 32 floats
// (kPartOff; share of row r from warp w at r * kShareLanes + w), then, in
// the split form, its two mbarriers (kBarOff).
template <typename GT, int NW, int G, int S> struct Cfg {
  static constexpr int kSubRows = NW <= 8 ? 32 / NW : 2;
  // a warp's total of row r is complete in lane r * kShareLanes after
  // row_shares; after the row statistics, lane r * kShareLanes holds 1 / r
  static constexpr int kShareLanes = 32 / kSubRows;
  static constexpr int kPieces = static_cast<int>(sizeof(GT)) / 2;  // 16-byte pieces per 8 values
  static constexpr int kWarpBytes = kSubRows * G * kPieces * 32 * 16;
  static constexpr int kStageBytes = kWarpBytes * NW;
  static constexpr bool kSplit = S >= 4;
  // share buffers: written at sub-panel q, read at q + 1; in the split form
  // a warp can write q + 3 only after every warp has arrived for q + 2, so
  // after every warp has read q (4 buffers)
  static constexpr int kShareBufs = kSplit ? 4 : 2;
  static constexpr size_t kPartOff = static_cast<size_t>(S) * kStageBytes;
  static constexpr size_t kBarOff = kPartOff + sizeof(float) * 32 * kShareBufs;
  static constexpr size_t kBytes = kBarOff + (kSplit ? 2 * sizeof(uint64_t) : 0);
  static_assert(kSubRows * NW <= 32 && kShareLanes * kSubRows == 32 && NW <= kShareLanes &&
                    (kSubRows == 2 || kSubRows == 4),
                "the row statistics take at most one (row, warp) share per lane");
  static_assert(S >= 2, "the ring needs the stage in use and one in flight");
  static_assert(kBarOff % 8 == 0, "mbarrier alignment");
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
                                        int lane, const float* pb, float2 (&cacc)[G][4],
                                        float (&rp)[Cfg<GT, NW, G, S>::kSubRows], float& psq) {
  constexpr int SR = Cfg<GT, NW, G, S>::kSubRows, P = Cfg<GT, NW, G, S>::kPieces;
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

// Phase B: g^2 / r into D_j (lane rr * kShareLanes holds 1 / r of row rr).
template <bool FULL, typename GT, int NW, int G, int S>
__device__ __forceinline__ void phase_b(const unsigned char* st, int32_t s0, int32_t s1, int32_t W, int warp,
                                        int lane, float winv, float2 (&dacc)[G][4]) {
  constexpr int SR = Cfg<GT, NW, G, S>::kSubRows, P = Cfg<GT, NW, G, S>::kPieces;
#pragma unroll
  for (int rr = 0; rr < SR; ++rr) {
    const float wr = __shfl_sync(0xffffffffu, winv, rr * Cfg<GT, NW, G, S>::kShareLanes);
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


// Row statistics of a sub-panel from its row shares pk (share of row r from
// warp w at r * kShareLanes + w): lane l adds the NW shares of row
// l / kShareLanes with a fixed xor tree over its kShareLanes lanes (slots
// past NW hold no share and count 0), forms r = b2 r_old + (1 - b2)(sum / W +
// eps1) and returns 1 / r; r is stored (and added to rsum) by warp 0's lane
// of each row inside [s0, s1).
template <typename GT, int NW, int G, int S>
__device__ __forceinline__ float row_stats(const float* pk, int lane, int warp, float row_old, int32_t s0,
                                           int32_t s1, float* rowst, float invw, float b2, float omb2, float eps1,
                                           float& rsum) {
  constexpr int SL = Cfg<GT, NW, G, S>::kShareLanes;
  const int rl = lane / SL;
  float R = (lane % SL < NW) ? pk[lane] : 0.f;
#pragma unroll
  for (int o = SL / 2; o > 0; o >>= 1) R += __shfl_xor_sync(0xffffffffu, R, o);
  const float rn = fmaf(b2, row_old, omb2 * fmaf(R, invw, eps1));
  if (warp == 0 && lane % SL == 0 && s0 + rl < s1) {
    rowst[s0 + rl] = rn;
    rsum += rn;
  }
  return __frcp_rn(rn);  // correctly rounded 1 / rn
}

// Where a chunk's column partials go: C_j to cp[0, W), D_j to dp[0, W).
struct Partials {
  float* cp;
  float* dp;
};

template <int NW, int G>
__device__ __forceinline__ void store_partials(const Partials& out, int32_t W, int warp, int lane,
                                               const float2 (&cacc)[G][4], const float2 (&dacc)[G][4]) {
#pragma unroll
  for (int c = 0; c < G; ++c) {
    const int32_t j = (c * NW + warp) * 256 + lane * 8;
    if (j < W) {
      float* cp = out.cp + j;
      float* dp = out.dp + j;
      *reinterpret_cast<float4*>(cp) = make_float4(cacc[c][0].x, cacc[c][0].y, cacc[c][1].x, cacc[c][1].y);
      *reinterpret_cast<float4*>(cp + 4) = make_float4(cacc[c][2].x, cacc[c][2].y, cacc[c][3].x, cacc[c][3].y);
      *reinterpret_cast<float4*>(dp) = make_float4(dacc[c][0].x, dacc[c][0].y, dacc[c][1].x, dacc[c][1].y);
      *reinterpret_cast<float4*>(dp + 4) = make_float4(dacc[c][2].x, dacc[c][2].y, dacc[c][3].x, dacc[c][3].y);
    }
  }
}

// One chunk of rows [c0, c1) of one slice (gb: the slice's gradient, pb its
// parameter, read only with PSQ; rowst: the slice's row statistic, updated in
// place).  Writes the chunk's column partials to where(), a callable that
// returns a Partials (evaluated after the rows, so that its operands need not
// stay in registers through the loop).  On return rsum holds, in lanes
// l % kShareLanes == 0 of warp 0, this thread's part of sum_r r over the
// chunk (0 elsewhere), and psq this thread's part of sum(p^2); the caller
// adds them over the CTA.  smem: the ring and row shares of Cfg (kBytes).
// Every thread of the CTA must call; the next call may follow directly (the
// caller's CTA barrier, e.g. the one in block_sum, separates this chunk's
// last reads of the ring from the next chunk's first copies).
template <typename GT, int NW, int G, int S, bool PSQ, typename Where>
__device__ __forceinline__ void run_chunk(unsigned char* smem, const GT* gb, const float* pb, float* rowst,
                                          int32_t W, int32_t c0, int32_t c1, float b2, float omb2, float eps1,
                                          Where&& where, float& rsum, float& psq) {
  using C = Cfg<GT, NW, G, S>;
  constexpr int SR = C::kSubRows;
  float* part = reinterpret_cast<float*>(smem + C::kPartOff);  // [2][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned char* mine = smem + warp * C::kWarpBytes + lane * 16;
  const uint32_t mine_s = static_cast<uint32_t>(__cvta_generic_to_shared(mine));
  const int rl = lane / C::kShareLanes;  // row of this lane's row statistic
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
    if (lane % C::kShareLanes == 0) pk[lane + warp] = tot;
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
    const float winv = row_stats<GT, NW, G, S>(pk, lane, warp, row_old, s0, s1, rowst, invw, b2, omb2, eps1, rsum);
    if (full) phase_b<true, GT, NW, G, S>(st, s0, s1, W, warp, lane, winv, dacc);
    else phase_b<false, GT, NW, G, S>(st, s0, s1, W, warp, lane, winv, dacc);
    stage = stage == S - 1 ? 0 : stage + 1;
  }
  store_partials<NW, G>(where(), W, warp, lane, cacc, dacc);
}

// The split form's barriers: two mbarriers at kBarOff, each completed by the
// NW * kSubRows lanes that hold row shares.  One thread of the CTA, before
// the first chunk; the caller's CTA barrier makes the initialisation visible.
template <typename GT, int NW, int G, int S>
__device__ __forceinline__ void split_init(unsigned char* smem) {
  using C = Cfg<GT, NW, G, S>;
  static_assert(C::kSplit, "the split form needs a ring of 4 stages or more");
  const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(smem + C::kBarOff));
  for (int b = 0; b < 2; ++b)
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar + 8 * b), "r"(NW * C::kSubRows) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Waits for the phase of parity `parity` of the mbarrier at `bar`; false
// after meo::kWaitCycles.
__device__ __forceinline__ bool split_wait(uint32_t bar, uint32_t parity) {
  auto done = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (done()) return true;
  const long long t0 = clock64();
  while (!done()) {
    if (clock64() - t0 > meo::kWaitCycles) return false;
  }
  return true;
}

// run_chunk in the split form (S >= 4; arguments and results as there).  q
// counts the sub-panels this CTA has finished over all its chunks (it picks
// the mbarrier, its phase and the share buffer) and is advanced by the
// chunk's sub-panels.  A wait that runs out sets kStatusWaitTimeout in
// *status and `dead`, after which the thread waits no more (the step's
// results are then not used).
template <typename GT, int NW, int G, int S, bool PSQ, typename Where>
__device__ __forceinline__ void run_chunk_split(unsigned char* smem, const GT* gb, const float* pb, float* rowst,
                                                int32_t W, int32_t c0, int32_t c1, float b2, float omb2,
                                                float eps1, Where&& where, float& rsum, float& psq, uint32_t& q,
                                                bool& dead, int32_t* status) {
  using C = Cfg<GT, NW, G, S>;
  static_assert(C::kSplit, "the split form needs a ring of 4 stages or more");
  constexpr int SR = C::kSubRows, SL = C::kShareLanes;
  float* part = reinterpret_cast<float*>(smem + C::kPartOff);  // [4][32]
  const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(smem + C::kBarOff));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned char* mine = smem + warp * C::kWarpBytes + lane * 16;
  const uint32_t mine_s = static_cast<uint32_t>(__cvta_generic_to_shared(mine));
  const int rl = lane / SL;  // row of this lane's share and row statistic
  const int32_t nsub = (c1 - c0 + SR - 1) / SR;
  const float invw = 1.0f / static_cast<float>(W);
  float2 cacc[G][4], dacc[G][4];
#pragma unroll
  for (int c = 0; c < G; ++c) {
#pragma unroll
    for (int v = 0; v < 4; ++v) cacc[c][v] = dacc[c][v] = make_float2(0.f, 0.f);
  }
  rsum = 0.f;
  // Prologue: sub-panels 0 .. S - 1, one commit group each (empty past the
  // chunk's end).  Iteration k >= 1 commits one group (sub-panel k - 1 + S),
  // so when sub-panel k is waited for, the groups of sub-panels up to
  // k + S - 2 are committed and sub-panel k is complete once at most S - 2
  // are pending.
#pragma unroll
  for (int k = 0; k < S; ++k) {
    if (k < nsub) issue<false, GT, NW, G, S>(mine_s + k * C::kStageBytes, gb, W, c0 + k * SR, c1, warp, lane);
    cp_async_commit();
  }
  const bool cols_full = ((G - 1) * NW + warp + 1) * 256 <= W;
  float old_prev = 0.f;  // old row statistic of this lane's row in sub-panel k - 1
  for (int32_t k = 0; k <= nsub; ++k) {
    float old_cur = 0.f;
    if (k < nsub) {
      const int32_t s0 = c0 + k * SR, s1 = min(c1, s0 + SR);
      const bool full = cols_full && s1 - s0 == SR;
      old_cur = (s0 + rl < s1) ? rowst[s0 + rl] : 0.f;
      cp_async_wait<S - 2>();
      const unsigned char* st = mine + (k % S) * C::kStageBytes;
      float rp[SR];
      if (full) phase_a<true, GT, NW, G, S, PSQ>(st, s0, s1, W, warp, lane, pb, cacc, rp, psq);
      else phase_a<false, GT, NW, G, S, PSQ>(st, s0, s1, W, warp, lane, pb, cacc, rp, psq);
      const float tot = row_shares(rp, lane);  // warp total of row lane / SL
      if (lane % SL == 0) {
        const uint32_t qk = q + static_cast<uint32_t>(k);
        part[(qk % 4) * 32 + lane + warp] = tot;
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar + 8 * (qk & 1)) : "memory");
      }
    }
    if (k > 0) {
      // row statistics and phase B of sub-panel k - 1
      const uint32_t qp = q + static_cast<uint32_t>(k) - 1;
      if (!dead && !split_wait(bar + 8 * (qp & 1), (qp >> 1) & 1)) {
        dead = true;
        if (lane == 0) atomicOr(status, meo::kStatusWaitTimeout);
      }
      const int32_t s0 = c0 + (k - 1) * SR, s1 = min(c1, s0 + SR);
      const bool full = cols_full && s1 - s0 == SR;
      const float winv = row_stats<GT, NW, G, S>(part + (qp % 4) * 32, lane, warp, old_prev, s0, s1, rowst, invw,
                                                 b2, omb2, eps1, rsum);
      const int stage = (k - 1) % S;
      const unsigned char* st = mine + stage * C::kStageBytes;
      if (full) phase_b<true, GT, NW, G, S>(st, s0, s1, W, warp, lane, winv, dacc);
      else phase_b<false, GT, NW, G, S>(st, s0, s1, W, warp, lane, winv, dacc);
      // this lane is past sub-panel k - 1: refill its stage with k - 1 + S
      const int32_t kk = k - 1 + S;
      if (kk < nsub) {
        if (cols_full && c0 + (kk + 1) * SR <= c1)
          issue<true, GT, NW, G, S>(mine_s + stage * C::kStageBytes, gb, W, c0 + kk * SR, c1, warp, lane);
        else
          issue<false, GT, NW, G, S>(mine_s + stage * C::kStageBytes, gb, W, c0 + kk * SR, c1, warp, lane);
      }
      cp_async_commit();
    }
    old_prev = old_cur;
  }
  q += static_cast<uint32_t>(nsub);
  store_partials<NW, G>(where(), W, warp, lane, cacc, dacc);
}

}  // namespace panel
}  // namespace meo
