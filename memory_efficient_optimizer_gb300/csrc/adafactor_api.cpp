// Host side of the C ABI declared in include/adafactor.h: argument checks,
// the per-call plan (tiling, workspace layout, device descriptor table), the
// pinned staging of that table, the launch sequence and the optional
// per-kernel event timing.
#include "adafactor.h"

#include <cmath>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "adafactor_internal.h"
#include "host_copy.cuh"

namespace {

using meo::DevTensor;
using meo::KernelId;
using meo::StepArgs;

thread_local std::string g_last_error;

adaf_status fail(adaf_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

adaf_status cuda_fail(cudaError_t e, const char* what) {
  std::string m = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return fail(ADAF_ERR_CUDA, m);
}

bool finite_nonneg(double x) { return std::isfinite(x) && x >= 0.0; }

adaf_status check_hparams(const adaf_hparams* hp) {
  if (hp == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "hparams is NULL");
  // Step 3 of the article: manual lr and relative_step exclude each other;
  // warmup_init forces relative_step.
  if (hp->has_lr && hp->relative_step)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "Cannot combine manual lr and relative_step=True options");
  if (hp->warmup_init && !hp->relative_step)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "warmup_init=True requires relative_step=True");
  if (!hp->has_lr && !hp->relative_step)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "relative_step=False requires a manual lr");
  if (!(std::isfinite(hp->clip_threshold) && hp->clip_threshold > 0.0))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "clip_threshold must be finite and > 0");
  if (hp->has_lr && !finite_nonneg(hp->lr))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "lr must be finite and >= 0");
  if (!finite_nonneg(hp->eps1) || !finite_nonneg(hp->eps2))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "eps values must be finite and >= 0");
  if (!std::isfinite(hp->decay_rate)) return fail(ADAF_ERR_INVALID_ARGUMENT, "decay_rate must be finite");
  if (!finite_nonneg(hp->weight_decay))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "weight_decay must be finite and >= 0");
  if (hp->has_beta1 && !(hp->beta1 >= 0.0 && hp->beta1 < 1.0))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "beta1 must be in [0, 1)");
  if (hp->exp_avg_int8 && !hp->has_beta1)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "exp_avg_int8 needs beta1 (there is no first moment without it)");
  return ADAF_OK;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The device status word lives at workspace offset 0; the descriptor table
// starts at kTableOffset.
constexpr size_t kTableOffset = 256;
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Geometry of one call: device descriptors (pointers filled later) and the
// workspace layout.  Tensors with no elements are dropped.
struct Plan {
  std::vector<DevTensor> dev;       // one per non-empty tensor
  std::vector<int32_t> pf_tiles, pf_items;
  // Per tensor class: member tensor indices and, per streaming kind, the
  // prefix of their work units (pass 1, pass 2, apply).
  std::vector<int32_t> cls_idx[meo::kNumClasses];
  std::vector<int32_t> cls_pf[3][meo::kNumClasses];
  size_t off_pf_tiles = 0, off_pf_items = 0, header_bytes = 0;
  size_t off_cls_idx[meo::kNumClasses] = {}, off_cls_pf[3][meo::kNumClasses] = {};
  size_t off_alpha = 0, off_coef = 0, off_ssum = 0, off_mrow = 0, off_rowchunk = 0, off_dsum = 0;
  size_t off_spart = 0, off_ppart = 0, off_rowpart = 0, off_colpart = 0, off_dpart = 0, total_bytes = 0;
  size_t off_dloc = 0;                       // row-sharded plans only
  size_t round1_doubles = 0, round2_doubles = 0;  // row-sharded plans only
  bool any_factored = false;
};

// Index of a streaming kind in Plan::cls_pf.
int stream_slot(KernelId k) { return k == meo::kKPass1 ? 0 : (k == meo::kKPass2 ? 1 : 2); }

// Rows per work unit of the fused pass.
int32_t panel_rows(int64_t W) { return W <= meo::kMaxRowsW ? meo::kRowsChunk : meo::kWideChunk; }
// Rows per pass-1 unit of the fused flat pass: about 64K values per unit, a
// multiple of 8 rows (so every unit of a slice starts on a 16-byte boundary
// of g, fp32 or bf16), at most 1024 rows.  (32K-value units measured 8 %
// slower on small matrices: the per-unit combine of column partials.)
int32_t flat_rows(int64_t W) {
  const int64_t r = (65536 / W) & ~int64_t{7};
  return static_cast<int32_t>(r < 8 ? 8 : (r > 1024 ? 1024 : r));
}

// Checks the tensor list and builds the plan.  With full == false (size
// query) only the shapes and dtypes are read; states and hp are not touched.
// The workspace layout is the same either way: it reserves room for both
// factored paths a tensor may take (which one depends on pointer alignment,
// known only at step time).  shards != NULL: every tensor is one row shard
// of a larger tensor (global rows in shards[k]); the plan then also lays out
// the exchange buffers and the shard's D_j region.
adaf_status make_plan(const adaf_tensor* tensors, const adaf_state* states, int32_t n,
                      const adaf_hparams* hp, bool full, Plan* plan, const adaf_shard* shards = nullptr) {
  if (n < 0) return fail(ADAF_ERR_INVALID_ARGUMENT, "n must be >= 0");
  if (n > 0 && tensors == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "tensors is NULL");
  int64_t tiles = 0, p1units = 0, p1bound = 0, items = 0, nmrow = 0, nrowchunk = 0, ndsum = 0;
  int64_t nrowpart = 0, ncolpart = 0, ndpart = 0;
  int64_t nx1col = 0, nx1row = 0, ndloc = 0;
  plan->dev.clear();
  plan->dev.reserve(n);
  for (int32_t k = 0; k < n; ++k) {
    const adaf_tensor& t = tensors[k];
    char pre[64];
    std::snprintf(pre, sizeof(pre), "tensor %d: ", k);
    if (t.ndim < 0 || t.ndim > ADAF_MAX_NDIM)
      return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "ndim must be in [0, 8]");
    if (t.grad_dtype != ADAF_FLOAT32 && t.grad_dtype != ADAF_BFLOAT16)
      return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "grad_dtype must be ADAF_FLOAT32 or ADAF_BFLOAT16");
    int64_t numel = 1;
    for (int32_t d = 0; d < t.ndim; ++d) {
      if (t.shape[d] < 0) return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "negative dimension");
      if (t.shape[d] != 0 && numel > (int64_t(1) << 50) / t.shape[d])
        return fail(ADAF_ERR_UNSUPPORTED, std::string(pre) + "more than 2^50 elements");
      numel *= t.shape[d];
    }
    if (numel == 0) {
      if (shards != nullptr)
        return fail(ADAF_ERR_INVALID_ARGUMENT,
                    std::string(pre) + "a row shard must hold at least one row of every tensor");
      continue;
    }
    const size_t gsz = t.grad_dtype == ADAF_BFLOAT16 ? 2 : 4;
    if (full) {
      if (t.param == nullptr || !aligned(t.param, 4))
        return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "param is NULL or not 4-byte aligned");
      if (t.grad == nullptr || !aligned(t.grad, gsz))
        return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "grad is NULL or misaligned");
    }
    DevTensor d;
    std::memset(&d, 0, sizeof(d));
    d.n = numel;
    d.gdt = t.grad_dtype == ADAF_BFLOAT16 ? meo::kGradBF16 : meo::kGradF32;
    if (full) {
      const adaf_state& s = states[k];
      d.p = t.param;
      d.g = t.grad;
      if (t.ndim >= 2) {
        if (s.exp_avg_sq_row == nullptr || s.exp_avg_sq_col == nullptr || !aligned(s.exp_avg_sq_row, 4) ||
            !aligned(s.exp_avg_sq_col, 4))
          return fail(ADAF_ERR_INVALID_ARGUMENT,
                      std::string(pre) + "factored tensor needs exp_avg_sq_row and exp_avg_sq_col");
        d.row = s.exp_avg_sq_row;
        d.col = s.exp_avg_sq_col;
      } else {
        if (s.exp_avg_sq == nullptr || !aligned(s.exp_avg_sq, 4))
          return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "tensor with ndim < 2 needs exp_avg_sq");
        d.v = s.exp_avg_sq;
      }
      if (hp->has_beta1 && hp->exp_avg_int8) {
        if (s.exp_avg_codes == nullptr || !aligned(s.exp_avg_codes, 4) || s.exp_avg_scales == nullptr ||
            !aligned(s.exp_avg_scales, 4))
          return fail(ADAF_ERR_INVALID_ARGUMENT,
                      std::string(pre) + "exp_avg_int8 needs 4-byte aligned exp_avg_codes and exp_avg_scales");
        d.mq = s.exp_avg_codes;
        d.ms = s.exp_avg_scales;
      } else if (hp->has_beta1) {
        if (s.exp_avg == nullptr || !aligned(s.exp_avg, 4))
          return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "beta1 is set but exp_avg is NULL");
        d.m1 = s.exp_avg;
      }
      if (s.param_sq_sum != nullptr && !aligned(s.param_sq_sum, 8))
        return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "param_sq_sum is not 8-byte aligned");
      if (hp->scale_parameter && hp->param_sq_sum_valid && s.param_sq_sum == nullptr)
        return fail(ADAF_ERR_INVALID_ARGUMENT,
                    std::string(pre) + "param_sq_sum_valid is set but param_sq_sum is NULL");
      d.psq = s.param_sq_sum;
    }
    int64_t ntiles, nunits;
    if (t.ndim >= 2) {
      const int64_t H = t.shape[t.ndim - 2], W = t.shape[t.ndim - 1];
      const int64_t B = numel / (H * W);
      if (B > INT32_MAX) return fail(ADAF_ERR_UNSUPPORTED, std::string(pre) + "too many leading slices");
      d.H = H;
      d.W = W;
      d.B = static_cast<int32_t>(B);
      d.rb = static_cast<int32_t>(ceil_div(H, meo::kTileRows));
      d.cb = static_cast<int32_t>(ceil_div(W, meo::kTileCols));
      d.ncc = static_cast<int32_t>(ceil_div(W, meo::kColChunk));
      d.qg = ceil_div(W, meo::kQ8Group);
      ntiles = B * d.rb * d.cb;
      // Path: vector (16-byte aligned rows) or element-wise; a vector tensor
      // with bf16 gradients and kMinRowsW <= W <= kMaxWideW takes the fused
      // row-chunk pass 1 (fp32 gradients keep the tiled passes).
      const bool vec_shape = (W % 8 == 0);
      const bool rows_shape = vec_shape && W >= meo::kMinRowsW && W <= meo::kMaxWideW &&
                              H <= INT32_MAX && t.grad_dtype == ADAF_BFLOAT16;
      // Rows that fit one tile: the fused flat pass 1 (whole rows per tile)
      // and the bulk-copy flat apply, when g, p and exp_avg start on 16-byte
      // boundaries and so does every slice (16-byte pieces of the flat range).
      const bool flat_shape = W <= meo::kTileCols && !rows_shape;
      bool vec = vec_shape;
      if (full) {
        vec = vec_shape && aligned(t.param, 16) && aligned(t.grad, 16) &&
              (!hp->has_beta1 || (hp->exp_avg_int8 ? aligned(d.mq, 16) : aligned(d.m1, 16)));
        const size_t ge = t.grad_dtype == ADAF_BFLOAT16 ? 2 : 4;
        const bool flat = flat_shape && aligned(t.grad, 16) && aligned(t.param, 16) &&
                          (!hp->has_beta1 || hp->exp_avg_int8 || aligned(d.m1, 16)) &&
                          (B == 1 || (H * W) % static_cast<int64_t>(16 / ge) == 0);
        d.kind = (vec && rows_shape) ? meo::kFactoredRows
                                     : (flat ? meo::kFactoredFlat : (vec ? meo::kFactoredVec : meo::kFactoredScalar));
      } else {
        d.kind = rows_shape ? meo::kFactoredRows : (flat_shape ? meo::kFactoredFlat : meo::kFactoredScalar);
      }
      // Row-panel geometry (also reserved in the size query for rows_shape).
      int32_t prb_rows = 0;
      if (rows_shape) {
        d.pr = panel_rows(W);
        prb_rows = static_cast<int32_t>(ceil_div(H, d.pr));
      }
      const bool fused = meo::is_fused(d.kind);
      // The layout reserves room for every path the tensor may take (which
      // one depends on pointer alignment), so the workspace size does not
      // depend on the pointers.  Fused flat tensors take the row tiles as
      // their chunks.
      const bool need_tiled = true;
      const bool need_rows = rows_shape || flat_shape;
      if (flat_shape) {
        d.pr = flat_rows(W);
        prb_rows = static_cast<int32_t>(ceil_div(H, d.pr));
      }
      d.nrc = fused ? prb_rows : static_cast<int32_t>(ceil_div(H, meo::kRowChunk));
      d.prb = fused ? prb_rows : d.rb;
      nunits = fused ? B * prb_rows : ntiles;
      // pass-1 units of either path (the sum(p^2) partials are per unit)
      p1bound += std::max<int64_t>(ntiles, need_rows ? B * prb_rows : 0);
      items += B * (fused ? d.ncc : (d.nrc + d.ncc));
      d.mslot = nmrow;
      nmrow += B;
      d.rowchunk = nrowchunk;
      const int64_t nrc_max = std::max<int64_t>(d.nrc, need_tiled ? ceil_div(H, meo::kRowChunk) : 0);
      nrowchunk += B * std::max<int64_t>(nrc_max, need_rows ? prb_rows : 0);
      d.rowpart = nrowpart;
      if (need_tiled) nrowpart += align_up(static_cast<int64_t>(d.cb) * B * H, 4);
      d.colpart = ncolpart;  // multiple of 4 floats: 16-byte aligned column quads
      ncolpart += align_up(B * std::max<int64_t>(need_tiled ? d.rb : 0, need_rows ? prb_rows : 0) * W, 4);
      d.dpart = ndpart;
      if (need_rows) ndpart += align_up(B * prb_rows * W, 4);
      d.dsum = ndsum;
      if (need_rows) ndsum += B * d.ncc;
      plan->any_factored = true;
    } else {
      d.H = 1;
      d.W = numel;
      d.B = 1;
      ntiles = ceil_div(numel, meo::kTile1D);
      nunits = ntiles;
      d.rb = 1;
      d.cb = static_cast<int32_t>(ntiles > INT32_MAX ? INT32_MAX : ntiles);
      d.kind = meo::kUnfactored;
      d.qg = ceil_div(numel, meo::kQ8Group);
      p1bound += ntiles;
    }
    // Normalisation over the whole tensor, and the exchange layout of a row
    // shard (identical on every shard: it depends on B and W only).
    const int64_t local_rows = d.kind == meo::kUnfactored ? numel : d.H;
    d.hg = local_rows;
    d.ng = numel;
    if (shards != nullptr) {
      const int64_t gr = shards[k].global_rows;
      if (gr < local_rows)
        return fail(ADAF_ERR_INVALID_ARGUMENT, std::string(pre) + "global_rows is smaller than the shard's rows");
      d.hg = gr;
      d.ng = d.kind == meo::kUnfactored ? gr : static_cast<int64_t>(d.B) * gr * d.W;
      if (d.kind != meo::kUnfactored) {
        d.x1c = nx1col;
        nx1col += static_cast<int64_t>(d.B) * d.W;
        d.x1r = nx1row;  // relative until the column block's size is known
        nx1row += d.B;
      }
      if (d.pr > 0 || (d.W <= meo::kTileCols && d.kind != meo::kUnfactored)) {
        // may take a fused pass 1 (reserved whatever the pointers' alignment)
        d.dloc = ndloc;
        ndloc += align_up(static_cast<int64_t>(d.B) * d.W, 4);
      }
    }
    d.ntiles = ntiles;
    d.tile0 = tiles;
    tiles += ntiles;
    d.p1_0 = p1units;
    d.p1_n = nunits;
    p1units += nunits;
    if (tiles > INT32_MAX || items > INT32_MAX || p1units > INT32_MAX)
      return fail(ADAF_ERR_UNSUPPORTED, "the tensor list needs more than 2^31-1 work tiles");
    plan->dev.push_back(d);
  }
  const size_t nd = plan->dev.size();
  if (shards != nullptr) {
    // exchange round 1: [column sums of every factored tensor][sum_i row_i per slice][sum(p^2) per tensor]
    for (size_t k = 0; k < nd; ++k) {
      DevTensor& d = plan->dev[k];
      if (d.kind != meo::kUnfactored) d.x1r += nx1col;
      d.x1p = nx1col + nx1row + static_cast<int64_t>(k);
    }
    plan->round1_doubles = static_cast<size_t>(nx1col + nx1row) + nd;
    plan->round2_doubles = nd;
  }
  plan->pf_tiles.assign(nd + 1, 0);
  plan->pf_items.assign(nd + 1, 0);
  for (int c = 0; c < meo::kNumClasses; ++c) {
    plan->cls_idx[c].clear();
    for (int q = 0; q < 3; ++q) plan->cls_pf[q][c].assign(1, 0);
  }
  for (size_t k = 0; k < nd; ++k) {
    const DevTensor& d = plan->dev[k];
    plan->pf_tiles[k + 1] = plan->pf_tiles[k] + static_cast<int32_t>(d.ntiles);
    const int64_t per_slice = meo::is_fused(d.kind) ? d.ncc : (d.nrc + d.ncc);
    plan->pf_items[k + 1] =
        plan->pf_items[k] + (d.kind == meo::kUnfactored ? 0 : static_cast<int32_t>(int64_t(d.B) * per_slice));
    int c = meo::kClsUnfactored;
    const bool bf = d.gdt == meo::kGradBF16;
    if (d.kind == meo::kFactoredVec) c = bf ? meo::kClsVecBF16 : meo::kClsVecF32;
    if (d.kind == meo::kFactoredScalar) c = bf ? meo::kClsScalarBF16 : meo::kClsScalarF32;
    if (d.kind == meo::kFactoredRows) c = d.W <= meo::kMaxRowsW ? meo::kClsRowsBF16 : meo::kClsWideBF16;
    if (d.kind == meo::kFactoredFlat) c = bf ? meo::kClsFlatBF16 : meo::kClsFlatF32;
    plan->cls_idx[c].push_back(static_cast<int32_t>(k));
  }
  // Members of the tiled classes walked largest tiles first: the persistent
  // CTAs take the units round-robin, so ragged lists of small matrices end
  // on small tiles instead of on a few large ones (each tensor's results
  // land at its own offsets, so the order changes no value).
  for (int c : {meo::kClsVecBF16, meo::kClsVecF32, meo::kClsScalarBF16, meo::kClsScalarF32, meo::kClsFlatBF16,
                meo::kClsFlatF32}) {
    std::vector<int32_t>& m = plan->cls_idx[c];
    std::stable_sort(m.begin(), m.end(), [&](int32_t x, int32_t y) {
      const DevTensor& a = plan->dev[x];
      const DevTensor& b = plan->dev[y];
      return static_cast<double>(a.n) / static_cast<double>(a.ntiles) >
             static_cast<double>(b.n) / static_cast<double>(b.ntiles);  // values per tile, descending
    });
  }
  for (int c = 0; c < meo::kNumClasses; ++c) {
    for (int32_t k : plan->cls_idx[c]) {
      const DevTensor& d = plan->dev[k];
      const bool two_pass = d.kind == meo::kFactoredVec || d.kind == meo::kFactoredScalar;
      plan->cls_pf[0][c].push_back(plan->cls_pf[0][c].back() + static_cast<int32_t>(d.p1_n));
      plan->cls_pf[1][c].push_back(plan->cls_pf[1][c].back() + (two_pass ? static_cast<int32_t>(d.ntiles) : 0));
      plan->cls_pf[2][c].push_back(plan->cls_pf[2][c].back() + static_cast<int32_t>(d.ntiles));
    }
  }
  // Workspace layout: the header (uploaded each call: the device status word
  // at offset 0, the descriptor table at kTableOffset, the prefix arrays)
  // first, then scratch; every scratch region 256-byte aligned.
  size_t off = kTableOffset + align_up(nd * sizeof(DevTensor), 256);
  plan->off_pf_tiles = off;
  off += align_up((nd + 1) * sizeof(int32_t), 16);
  plan->off_pf_items = off;
  off += align_up((nd + 1) * sizeof(int32_t), 16);
  for (int c = 0; c < meo::kNumClasses; ++c) {
    for (int q = 0; q < 3; ++q) {
      plan->off_cls_pf[q][c] = off;
      off += align_up(plan->cls_pf[q][c].size() * sizeof(int32_t), 16);
    }
    plan->off_cls_idx[c] = off;
    off += align_up(plan->cls_idx[c].size() * sizeof(int32_t), 16);
  }
  plan->header_bytes = off;
  // Scratch starts after a bound on the header that depends on the tensor
  // count only: a tensor's class follows its pointers' alignment, and the
  // 16-byte rounding of the per-class arrays with it, so the size query
  // (without pointers) and the step must not use the header's exact size.
  // Per class: three prefix arrays of members + 1 entries and the index
  // array, each rounded up by at most 12 bytes; every tensor is in one class.
  const size_t header_bound = kTableOffset + align_up(nd * sizeof(DevTensor), 256) +
                              2 * align_up((nd + 1) * sizeof(int32_t), 16) +
                              (4 * nd + 3 * meo::kNumClasses) * sizeof(int32_t) + 4 * 12 * meo::kNumClasses;
  off = align_up(header_bound, 256);
  const int64_t nppart = std::max(tiles, std::max(p1units, p1bound));
  auto region = [&](size_t* where, size_t bytes) {
    *where = off;
    off = align_up(off + bytes, 256);
  };
  region(&plan->off_alpha, nd * sizeof(double));
  region(&plan->off_coef, nd * sizeof(double));
  region(&plan->off_ssum, nd * sizeof(double));
  region(&plan->off_mrow, nmrow * sizeof(double));
  region(&plan->off_rowchunk, nrowchunk * sizeof(double));
  region(&plan->off_dsum, ndsum * sizeof(double));
  region(&plan->off_spart, tiles * sizeof(double));
  region(&plan->off_ppart, nppart * sizeof(double));
  region(&plan->off_rowpart, nrowpart * sizeof(float));
  region(&plan->off_colpart, ncolpart * sizeof(float));
  region(&plan->off_dpart, ndpart * sizeof(float));
  if (shards != nullptr) region(&plan->off_dloc, ndloc * sizeof(float));
  plan->total_bytes = off;
  return ADAF_OK;
}

// ---- pinned staging of the descriptor table -------------------------------
// A small ring of pinned, device-mapped host buffers per device, read by the
// upload kernel (host_copy.cuh); a slot is reused only after the event
// recorded behind its previous upload has completed, so the host never
// overwrites bytes a pending upload still has to read.
constexpr int kSlots = 4;
struct Slot {
  void* host = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;
  bool pending = false;
};
struct DeviceCache {
  Slot slots[kSlots];
  int next = 0;
  std::vector<cudaEvent_t> free_events;
  meo::TableCache tables;              // device copies of the header (host_copy.cuh)
  std::vector<unsigned char> scratch;  // this call's header, built on the host
};

struct ProfRecord {
  int slot;
  int device;
  cudaEvent_t start, stop;
};

// Profiling slots: one per streaming kernel kind and tensor class, one per
// other kernel kind, in launch order.
constexpr int kNumSlots = 3 * meo::kNumClasses + 4;
const char* const kClassNames[meo::kNumClasses] = {"vec_bf16",  "vec_f32",   "elem_bf16", "elem_f32", "1d",
                                                   "rows_bf16", "wide_bf16", "flat_bf16", "flat_f32"};

int profile_slot(KernelId k, int cls) {
  const int C = meo::kNumClasses;
  switch (k) {
    case meo::kKPass1: return cls;
    case meo::kKStats: return C;
    case meo::kKScalars: return C + 1;
    case meo::kKPass2: return C + 2 + cls;
    case meo::kKClip: return 2 * C + 2;
    case meo::kKApply: return 2 * C + 3 + cls;
    case meo::kKPsq: return 3 * C + 3;
    default: return 0;
  }
}

const char* slot_name(int slot) {
  static std::string names[kNumSlots];
  static std::once_flag once;
  std::call_once(once, [] {
    const int C = meo::kNumClasses;
    for (int c = 0; c < C; ++c) {
      names[c] = std::string("k_pass1[") + kClassNames[c] + "]";
      names[C + 2 + c] = std::string("k_pass2[") + kClassNames[c] + "]";
      names[2 * C + 3 + c] = std::string("k_apply[") + kClassNames[c] + "]";
    }
    names[C] = "k_stats";
    names[C + 1] = "k_scalars";
    names[2 * C + 2] = "k_clip";
    names[3 * C + 3] = "k_psq";
  });
  return (slot >= 0 && slot < kNumSlots) ? names[slot].c_str() : "";
}

std::mutex g_mu;
std::atomic<int> g_stall_copies{0};
std::map<int, DeviceCache> g_cache;
bool g_profile = false;
std::vector<ProfRecord> g_prof;

cudaError_t get_event(DeviceCache& dc, cudaEvent_t* ev) {
  if (!dc.free_events.empty()) {
    *ev = dc.free_events.back();
    dc.free_events.pop_back();
    return cudaSuccess;
  }
  return cudaEventCreate(ev);
}

// Writes the uploaded header: status word 0, descriptor table, prefix arrays.
void fill_header(unsigned char* h, const Plan& plan) {
  const size_t nd = plan.dev.size();
  std::memset(h, 0, kTableOffset);  // status word := 0
  std::memcpy(h + kTableOffset, plan.dev.data(), nd * sizeof(DevTensor));
  std::memcpy(h + plan.off_pf_tiles, plan.pf_tiles.data(), (nd + 1) * sizeof(int32_t));
  std::memcpy(h + plan.off_pf_items, plan.pf_items.data(), (nd + 1) * sizeof(int32_t));
  for (int c = 0; c < meo::kNumClasses; ++c) {
    for (int q = 0; q < 3; ++q)
      std::memcpy(h + plan.off_cls_pf[q][c], plan.cls_pf[q][c].data(), plan.cls_pf[q][c].size() * sizeof(int32_t));
    if (!plan.cls_idx[c].empty())
      std::memcpy(h + plan.off_cls_idx[c], plan.cls_idx[c].data(), plan.cls_idx[c].size() * sizeof(int32_t));
  }
}

}  // namespace

namespace meo {

// The whole step (phase 0) or one call of a row-sharded step (phases 1-3:
// begin, middle, end): checks, plan, header upload, launch sequence.  Every
// argument check runs before the first CUDA call.
adaf_status step_core(const adaf_tensor* tensors, const adaf_state* states, const adaf_shard* shards, int32_t n,
                      int64_t step, const adaf_hparams* hp, void* workspace, size_t workspace_bytes,
                      int phase, double* round1, double* round2, void* stream, HeaderStaging staging) {
  adaf_status st = check_hparams(hp);
  if (st != ADAF_OK) return st;
  if (step < 1) return fail(ADAF_ERR_INVALID_ARGUMENT, "step must be >= 1");
  if (n > 0 && states == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "states is NULL");
  if (phase != 0 && n > 0 && shards == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "shards is NULL");
  if ((phase == 1 || phase == 2) && (round1 == nullptr || !aligned(round1, 8)))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "round1 is NULL or not 8-byte aligned");
  if ((phase == 2 || phase == 3) && (round2 == nullptr || !aligned(round2, 8)))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "round2 is NULL or not 8-byte aligned");
  Plan plan;
  st = make_plan(tensors, states, n, hp, true, &plan, phase != 0 ? shards : nullptr);
  if (st != ADAF_OK) return st;
  const size_t nd = plan.dev.size();
  if (nd == 0) return ADAF_OK;
  if (workspace == nullptr || !aligned(workspace, 256))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "workspace is NULL or not 256-byte aligned");
  if (workspace_bytes < plan.total_bytes) {
    char msg[128];
    std::snprintf(msg, sizeof(msg), "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                  plan.total_bytes);
    return fail(ADAF_ERR_WORKSPACE_TOO_SMALL, msg);
  }

  // Per-step scalars (Step 3 / Step 5 of the article), in double on the host.
  const double t = static_cast<double>(step);
  double rho = hp->lr;
  if (hp->relative_step) {
    const double cap = hp->warmup_init ? 1e-6 * t : 1e-2;
    const double inv = 1.0 / std::sqrt(t);
    rho = cap < inv ? cap : inv;
  }
  const double beta2 = 1.0 - std::pow(t, hp->decay_rate);
  bool any_psq = false;
  for (const DevTensor& d : plan.dev) any_psq = any_psq || d.psq != nullptr;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceCache& dc = g_cache[device];
  const unsigned char* hbase = ws;  // where the kernels read the header (descriptors, prefix arrays)
  RecordOnExit used_guard;
  if (staging == kStagePinned) {
    // The header is kept on the device per distinct content (TableCache): a
    // step whose header equals a kept one reads that copy; otherwise the
    // header is staged in a pinned ring slot and uploaded into a new device
    // copy.  The status word stays in the workspace and is cleared by a
    // one-thread kernel.
    dc.scratch.resize(plan.header_bytes);
    fill_header(dc.scratch.data(), plan);
    auto upload = [&](unsigned char* dst) -> cudaError_t {
      Slot& slot = dc.slots[dc.next];
      dc.next = (dc.next + 1) % kSlots;
      cudaError_t err = cudaSuccess;
      if (slot.pending) {
        err = cudaEventSynchronize(slot.done);
        if (err != cudaSuccess) return err;
        slot.pending = false;
      }
      if (slot.cap < plan.header_bytes) {
        if (slot.host != nullptr) cudaFreeHost(slot.host);
        slot.host = nullptr;
        slot.cap = 0;
        const size_t cap = align_up(plan.header_bytes, size_t(1) << 16);
        err = cudaHostAlloc(&slot.host, cap, cudaHostAllocPortable | cudaHostAllocMapped);
        if (err != cudaSuccess) return err;
        slot.cap = cap;
      }
      if (slot.done == nullptr && (err = cudaEventCreateWithFlags(&slot.done, cudaEventDisableTiming)) != cudaSuccess)
        return err;
      std::memcpy(slot.host, dc.scratch.data(), plan.header_bytes);
      if ((err = copy_from_host(dst, slot.host, plan.header_bytes, s)) != cudaSuccess) return err;  // no copy engine
      if ((err = cudaEventRecord(slot.done, s)) != cudaSuccess) return err;
      slot.pending = true;
      return cudaSuccess;
    };
    unsigned char* dev = nullptr;
    e = dc.tables.lookup(dc.scratch.data(), plan.header_bytes, s, upload, &dev, &used_guard.ev);
    if (e != cudaSuccess) return cuda_fail(e, "descriptor table upload");
    used_guard.s = s;
    hbase = dev;
    e = zero_word(reinterpret_cast<int32_t*>(ws), s);  // this step's status word
    if (e != cudaSuccess) return cuda_fail(e, "status word reset");
  } else {
    // Pageable staging: the runtime copies the host bytes out before the
    // call returns, so a local buffer suffices.
    std::vector<unsigned char> h(plan.header_bytes);
    fill_header(h.data(), plan);
    e = cudaMemcpyAsync(ws, h.data(), plan.header_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (descriptor table)");
  }
  const bool profile = g_profile && staging == kStagePinned;

  StepArgs a;
  std::memset(&a, 0, sizeof(a));
  a.tensors = reinterpret_cast<const DevTensor*>(hbase + kTableOffset);
  a.status = reinterpret_cast<int32_t*>(ws);
  a.pf_tiles = reinterpret_cast<const int32_t*>(hbase + plan.off_pf_tiles);
  a.pf_items = reinterpret_cast<const int32_t*>(hbase + plan.off_pf_items);
  a.alpha = reinterpret_cast<double*>(ws + plan.off_alpha);
  a.coef = reinterpret_cast<double*>(ws + plan.off_coef);
  a.mrow = reinterpret_cast<double*>(ws + plan.off_mrow);
  a.rowchunk = reinterpret_cast<double*>(ws + plan.off_rowchunk);
  a.ssum = reinterpret_cast<double*>(ws + plan.off_ssum);
  a.dsum = reinterpret_cast<double*>(ws + plan.off_dsum);
  a.dpart = reinterpret_cast<float*>(ws + plan.off_dpart);
  a.spart = reinterpret_cast<double*>(ws + plan.off_spart);
  a.ppart = reinterpret_cast<double*>(ws + plan.off_ppart);
  a.rowpart = reinterpret_cast<float*>(ws + plan.off_rowpart);
  a.colpart = reinterpret_cast<float*>(ws + plan.off_colpart);
  a.beta2 = beta2;
  a.rho = rho;
  a.eps1 = hp->eps1;
  a.eps2 = hp->eps2;
  a.clip = hp->clip_threshold;
  a.beta1 = hp->has_beta1 ? hp->beta1 : 0.0;
  a.wd = hp->weight_decay;
  a.scale_parameter = hp->scale_parameter ? 1 : 0;
  a.has_beta1 = hp->has_beta1 ? 1 : 0;
  a.psq_valid = (hp->scale_parameter && hp->param_sq_sum_valid) ? 1 : 0;
  a.want_psq_out = any_psq ? 1 : 0;
  a.stall_copies = g_stall_copies.load();
  a.phase = phase;
  a.q8 = (hp->has_beta1 && hp->exp_avg_int8) ? 1 : 0;
  a.round1 = round1;
  a.round2 = round2;
  a.dloc = phase != 0 ? reinterpret_cast<float*>(ws + plan.off_dloc) : nullptr;
  const int variant = meo::kernel_variant(a);
  int grid_limit[meo::kNumKernels][meo::kNumClasses];
  for (int k = 0; k < meo::kNumKernels; ++k) {
    for (int c = 0; c < meo::kNumClasses; ++c) {
      grid_limit[k][c] = meo::kernel_grid_limit(static_cast<KernelId>(k), static_cast<meo::TensorClass>(c),
                                                variant, device, &e);
      if (e != cudaSuccess) return cuda_fail(e, "kernel occupancy query");
    }
  }

  // One launch helper: optional profiling events around the launch.
  auto run = [&](KernelId k, int cls, auto&& launch) -> adaf_status {
    ProfRecord rec{profile_slot(k, cls), device, nullptr, nullptr};
    cudaError_t err;
    if (profile) {
      if ((err = get_event(dc, &rec.start)) != cudaSuccess) return cuda_fail(err, "cudaEventCreate (profile)");
      if ((err = get_event(dc, &rec.stop)) != cudaSuccess) return cuda_fail(err, "cudaEventCreate (profile)");
      if ((err = cudaEventRecord(rec.start, s)) != cudaSuccess) return cuda_fail(err, "cudaEventRecord (profile)");
    }
    err = launch();
    if (err != cudaSuccess) return cuda_fail(err, meo::kernel_name(k));
    if (profile) {
      if ((err = cudaEventRecord(rec.stop, s)) != cudaSuccess) return cuda_fail(err, "cudaEventRecord (profile)");
      g_prof.push_back(rec);
    }
    return ADAF_OK;
  };
  // A streaming kind over every class that has members, in groups of at most
  // kMaxGroup tensors (the kernels keep a group's prefix in shared memory).
  auto stream_all = [&](KernelId k, bool factored_only) -> adaf_status {
    for (int c = 0; c < meo::kNumClasses; ++c) {
      if (factored_only && c == meo::kClsUnfactored) continue;
      const int32_t m = static_cast<int32_t>(plan.cls_idx[c].size());
      const int q = stream_slot(k);
      const int32_t* pf_dev = reinterpret_cast<const int32_t*>(hbase + plan.off_cls_pf[q][c]);
      const int32_t* idx_dev = reinterpret_cast<const int32_t*>(hbase + plan.off_cls_idx[c]);
      for (int32_t g0 = 0; g0 < m; g0 += meo::kMaxGroup) {
        const int32_t g1 = g0 + meo::kMaxGroup < m ? g0 + meo::kMaxGroup : m;
        const int64_t units = plan.cls_pf[q][c][g1] - plan.cls_pf[q][c][g0];
        if (units == 0) continue;
        const int grid = static_cast<int>(units < grid_limit[k][c] ? units : grid_limit[k][c]);
        const meo::Range r{pf_dev, idx_dev, g0, g1};
        const meo::TensorClass tc = static_cast<meo::TensorClass>(c);
        adaf_status rs = run(k, c, [&] { return meo::launch_stream(k, tc, a, r, grid, s); });
        if (rs != ADAF_OK) return rs;
      }
    }
    return ADAF_OK;
  };
  const int nd_i = static_cast<int>(nd);
  // Phase 0: everything.  Row-sharded: 1 = pass 1, this shard's statistics
  // into exchange round 1; 2 = column statistics from exchange round 1, pass 2,
  // this shard's sum(u^2) into exchange round 2; 3 = clip from exchange round 2, apply.
  auto stats = [&]() -> adaf_status {
    if (!plan.any_factored) return ADAF_OK;
    const int32_t* pf_items_dev = reinterpret_cast<const int32_t*>(hbase + plan.off_pf_items);
    for (int32_t g0 = 0; g0 < nd_i; g0 += meo::kMaxGroup) {
      const int32_t g1 = g0 + meo::kMaxGroup < nd_i ? g0 + meo::kMaxGroup : nd_i;
      const int64_t units = plan.pf_items[g1] - plan.pf_items[g0];
      if (units == 0) continue;
      const int lim = grid_limit[meo::kKStats][0];
      const int grid = static_cast<int>(units < lim ? units : lim);
      const meo::Range r{pf_items_dev, nullptr, g0, g1};
      adaf_status rs = run(meo::kKStats, 0, [&] { return meo::launch_stats(a, r, grid, s); });
      if (rs != ADAF_OK) return rs;
    }
    return ADAF_OK;
  };
  auto per_tensor = [&](KernelId k) {
    return run(k, 0, [&] { return meo::launch_per_tensor(k, a, nd_i, s); });
  };
  if (phase == 1) {
    if ((st = stream_all(meo::kKPass1, false)) != ADAF_OK) return st;
    if ((st = stats()) != ADAF_OK) return st;
    return per_tensor(meo::kKScalars);
  }
  if (phase == 2) {
    if ((st = stats()) != ADAF_OK) return st;
    if ((st = per_tensor(meo::kKScalars)) != ADAF_OK) return st;
    if ((st = stream_all(meo::kKPass2, true)) != ADAF_OK) return st;
    return per_tensor(meo::kKClip);
  }
  if (phase == 3) {
    if ((st = per_tensor(meo::kKClip)) != ADAF_OK) return st;
    if ((st = stream_all(meo::kKApply, false)) != ADAF_OK) return st;
    return any_psq ? per_tensor(meo::kKPsq) : ADAF_OK;
  }
  if ((st = stream_all(meo::kKPass1, false)) != ADAF_OK) return st;
  if (plan.any_factored) {
    const int32_t* pf_items_dev = reinterpret_cast<const int32_t*>(hbase + plan.off_pf_items);
    for (int32_t g0 = 0; g0 < nd_i; g0 += meo::kMaxGroup) {
      const int32_t g1 = g0 + meo::kMaxGroup < nd_i ? g0 + meo::kMaxGroup : nd_i;
      const int64_t units = plan.pf_items[g1] - plan.pf_items[g0];
      if (units == 0) continue;
      const int lim = grid_limit[meo::kKStats][0];
      const int grid = static_cast<int>(units < lim ? units : lim);
      const meo::Range r{pf_items_dev, nullptr, g0, g1};
      st = run(meo::kKStats, 0, [&] { return meo::launch_stats(a, r, grid, s); });
      if (st != ADAF_OK) return st;
    }
  }
  st = run(meo::kKScalars, 0, [&] { return meo::launch_per_tensor(meo::kKScalars, a, nd_i, s); });
  if (st != ADAF_OK) return st;
  if ((st = stream_all(meo::kKPass2, true)) != ADAF_OK) return st;
  st = run(meo::kKClip, 0, [&] { return meo::launch_per_tensor(meo::kKClip, a, nd_i, s); });
  if (st != ADAF_OK) return st;
  if ((st = stream_all(meo::kKApply, false)) != ADAF_OK) return st;
  if (any_psq) {
    st = run(meo::kKPsq, 0, [&] { return meo::launch_per_tensor(meo::kKPsq, a, nd_i, s); });
    if (st != ADAF_OK) return st;
  }
  return ADAF_OK;
}

adaf_status step_impl(const adaf_tensor* tensors, const adaf_state* states, int32_t n, int64_t step,
                      const adaf_hparams* hp, void* workspace, size_t workspace_bytes, void* stream,
                      HeaderStaging staging) {
  return step_core(tensors, states, nullptr, n, step, hp, workspace, workspace_bytes, 0, nullptr, nullptr, stream,
                   staging);
}

adaf_status set_last_error(adaf_status st, const char* msg) { return fail(st, msg); }

}  // namespace meo

extern "C" {

void adafactor_default_hparams(adaf_hparams* hp) {
  if (hp == nullptr) return;
  std::memset(hp, 0, sizeof(*hp));
  hp->lr = 0.0;
  hp->has_lr = 0;
  hp->eps1 = 1e-30;
  hp->eps2 = 1e-3;
  hp->clip_threshold = 1.0;
  hp->decay_rate = -0.8;
  hp->beta1 = 0.0;
  hp->has_beta1 = 0;
  hp->weight_decay = 0.0;
  hp->scale_parameter = 1;
  hp->relative_step = 1;
  hp->warmup_init = 0;
  hp->param_sq_sum_valid = 0;
}

adaf_status adafactor_validate(const adaf_hparams* hp) { return check_hparams(hp); }

adaf_status adafactor_workspace_size(const adaf_tensor* tensors, int32_t n, size_t* bytes) {
  if (bytes == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "bytes is NULL");
  Plan plan;
  adaf_status st = make_plan(tensors, nullptr, n, nullptr, false, &plan);
  if (st != ADAF_OK) return st;
  *bytes = plan.total_bytes;
  return ADAF_OK;
}

adaf_status adafactor_step(const adaf_tensor* tensors, const adaf_state* states, int32_t n, int64_t step,
                           const adaf_hparams* hp, void* workspace, size_t workspace_bytes, void* stream) {
  return meo::step_impl(tensors, states, n, step, hp, workspace, workspace_bytes, stream, meo::kStagePinned);
}

adaf_status adafactor_shard_sizes(const adaf_tensor* tensors, const adaf_shard* shards, int32_t n,
                                  size_t* workspace_bytes, size_t* round1_bytes, size_t* round2_bytes) {
  if (workspace_bytes == nullptr || round1_bytes == nullptr || round2_bytes == nullptr)
    return fail(ADAF_ERR_INVALID_ARGUMENT, "an output pointer is NULL");
  if (n > 0 && shards == nullptr) return fail(ADAF_ERR_INVALID_ARGUMENT, "shards is NULL");
  Plan plan;
  adaf_status st = make_plan(tensors, nullptr, n, nullptr, false, &plan, shards);
  if (st != ADAF_OK) return st;
  *workspace_bytes = plan.total_bytes;
  *round1_bytes = plan.round1_doubles * sizeof(double);
  *round2_bytes = plan.round2_doubles * sizeof(double);
  return ADAF_OK;
}

adaf_status adafactor_shard_begin(const adaf_tensor* tensors, const adaf_state* states, const adaf_shard* shards,
                                  int32_t n, int64_t step, const adaf_hparams* hp, void* workspace,
                                  size_t workspace_bytes, double* round1, void* stream) {
  return meo::step_core(tensors, states, shards, n, step, hp, workspace, workspace_bytes, 1, round1, nullptr,
                        stream, meo::kStagePinned);
}

adaf_status adafactor_shard_middle(const adaf_tensor* tensors, const adaf_state* states, const adaf_shard* shards,
                                   int32_t n, int64_t step, const adaf_hparams* hp, void* workspace,
                                   size_t workspace_bytes, const double* round1, double* round2, void* stream) {
  return meo::step_core(tensors, states, shards, n, step, hp, workspace, workspace_bytes, 2,
                        const_cast<double*>(round1), round2, stream, meo::kStagePinned);
}

adaf_status adafactor_shard_end(const adaf_tensor* tensors, const adaf_state* states, const adaf_shard* shards,
                                int32_t n, int64_t step, const adaf_hparams* hp, void* workspace,
                                size_t workspace_bytes, const double* round2, void* stream) {
  return meo::step_core(tensors, states, shards, n, step, hp, workspace, workspace_bytes, 3, nullptr,
                        const_cast<double*>(round2), stream, meo::kStagePinned);
}

const char* adafactor_last_error(void) { return g_last_error.c_str(); }

void adafactor_debug_stall_copies(int32_t on) { g_stall_copies.store(on != 0 ? 1 : 0); }

adaf_status adafactor_device_status(const void* workspace, void* stream, int32_t* status) {
  if (workspace == nullptr || status == nullptr || !aligned(workspace, 256))
    return fail(ADAF_ERR_INVALID_ARGUMENT, "workspace or status is NULL, or workspace misaligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  *status = v;
  return ADAF_OK;
}

void adafactor_release_cache(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  const bool have_dev = cudaGetDevice(&cur) == cudaSuccess;
  for (auto& kv : g_cache) {
    if (cudaSetDevice(kv.first) != cudaSuccess) continue;
    for (Slot& sl : kv.second.slots) {
      if (sl.pending && sl.done) cudaEventSynchronize(sl.done);
      if (sl.done) cudaEventDestroy(sl.done);
      if (sl.host) cudaFreeHost(sl.host);
      sl = Slot();
    }
    for (cudaEvent_t ev : kv.second.free_events) cudaEventDestroy(ev);
    kv.second.free_events.clear();
    kv.second.tables.clear();
  }
  for (ProfRecord& r : g_prof) {
    if (cudaSetDevice(r.device) == cudaSuccess) {
      cudaEventDestroy(r.start);
      cudaEventDestroy(r.stop);
    }
  }
  g_prof.clear();
  g_cache.clear();
  meo::noalloc_forget_addresses();
  meo::lamb_forget_tables();
  meo::came_forget_tables();
  if (have_dev) cudaSetDevice(cur);
}

adaf_status adafactor_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profile = on != 0;
  return ADAF_OK;
}

adaf_status adafactor_profile_read(double* ms, int64_t* launches, int32_t nk) {
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
    DeviceCache& dc = g_cache[r.device];
    dc.free_events.push_back(r.start);
    dc.free_events.push_back(r.stop);
  }
  g_prof.clear();
  return st;
}

int32_t adafactor_num_kernels(void) { return kNumSlots; }

const char* adafactor_kernel_name(int32_t k) { return slot_name(k); }

}  // extern "C"
