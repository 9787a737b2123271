// Internal definitions shared by the host planner (adafactor_api.cpp) and the
// kernels (adafactor_kernels.cu).  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace meo {

// ---- tiling ---------------------------------------------------------------
// A factored tensor [B, H, W] is cut into tiles of kTileRows rows x kTileCols
// columns inside one slice b.  One CTA of kThreads threads streams a tile:
// warp w takes rows w, w + kWarps, ...; each lane owns kTileCols / 32 columns
// of the tile (8 consecutive ones per 256-column chunk on the vector path,
// one per 32-column chunk on the element-wise path).
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileRows = 256;
constexpr int kTileCols = 1024;
// A tensor with ndim < 2 is cut into flat tiles of kTile1D elements.
constexpr int kTile1D = 8192;
// Statistics kernel: a row item covers kRowChunk rows of one slice, a column
// item kColChunk columns of one slice.
constexpr int kRowChunk = 1024;
constexpr int kColChunk = 256;
// Tensors handled by one launch sequence (prefix arrays live in shared memory).
constexpr int kMaxGroup = 4096;

enum TensorKind : int32_t {
  kFactoredVec = 0,   // ndim >= 2, W % 8 == 0, 16-byte aligned pointers (tiled passes 1 and 2)
  kFactoredScalar = 1,// ndim >= 2, anything else
  kUnfactored = 2,    // ndim < 2
  kFactoredRows = 3,  // as kFactoredVec with kMinRowsW <= W <= kMaxWideW, bf16 grads: fused pass 1
  kFactoredFlat = 4,  // W <= kTileCols (rows not of kFactoredRows), aligned tile starts: fused flat pass 1
};
// Tensors whose pass 1 also forms the row statistic and the weighted column
// partials D_j (no pass 2).
__host__ __device__ inline bool is_fused(int32_t kind) { return kind == kFactoredRows || kind == kFactoredFlat; }

// Fused pass 1 (kFactoredRows): a CTA takes chunks of d.pr full rows and
// keeps the column sums of the chunk in registers, 8 values x G column
// groups of 256 per lane.  Two configurations:
//   rows:  2048 <= W <= 4096,  8 warps x 2 groups, 256-row chunks;
//   wide:  4096 <  W <= 14336, 14 warps x 4 groups, 128-row chunks.
constexpr int kMinRowsW = 2048;   // narrower rows keep the tiled two-pass path
constexpr int kMaxRowsW = 4096;   // 8 warps x 2 groups x 256 columns
constexpr int kMaxWideW = 14336;  // 14 warps x 4 groups x 256 columns
constexpr int kRowsChunk = 256;   // rows per work unit (rows configuration)
constexpr int kQ8Group = 128;     // values per group of the 8-bit first moment
constexpr int kWideChunk = 128;   // rows per work unit (wide configuration)

enum GradType : int32_t { kGradF32 = 0, kGradBF16 = 1 };

// Device-side descriptor of one tensor (built on the host each call).
struct DevTensor {
  float* p;
  const void* g;
  float* row;     // [B*H]
  float* col;     // [B*W]
  float* v;       // [N]      unfactored
  float* m1;      // [N]      beta1
  double* psq;    // [1]      optional sum(p^2) carry
  int64_t n;      // numel
  int64_t H, W;   // factored: matrix dims; unfactored: 1, n
  int32_t B;      // leading slices
  int32_t kind;   // TensorKind
  int32_t gdt;    // GradType
  int32_t rb;     // row blocks per slice   (ceil(H / kTileRows)); unfactored: 1
  int32_t cb;     // column blocks          (ceil(W / kTileCols)); unfactored: tiles
  int32_t nrc;    // row-sum chunks per slice: ceil(H / kRowChunk), or panels / row tiles (fused kinds)
  int32_t ncc;    // column chunks per slice(ceil(W / kColChunk))
  int32_t prb;    // row blocks of the column partials: rb, or panels per slice (kFactoredRows)
  int32_t pr;     // rows per pass-1 unit (fused kinds: a panel chunk, or a flat chunk)
  int32_t seg;    // unused (0)
  int32_t lanes;  // unused (0)
  int64_t ntiles;     // apply tiles
  int64_t p1_0, p1_n; // pass-1 units: global base (Ppart slot) and count
  int64_t dpart;      // float offset of the weighted column partials [B][prb][W] (fused kinds)
  int64_t dsum;       // double offset of per-chunk sum_j D_j / col_j [B][ncc] (fused kinds)
  int64_t tile0;      // global index of the tensor's first tile (Spart/Ppart slot)
  int64_t rowpart;    // float offset of rowpart [cb][B*H]
  int64_t colpart;    // float offset of colpart [B][rb][W]
  int64_t rowchunk;   // double offset of row-chunk sums [B][nrc]
  int64_t mslot;      // double offset of mean(row) [B]
  // Normalisation: rows and elements of the whole tensor (H and n unless the
  // tensor is one row shard of a larger one).
  int64_t hg;         // factored: rows per slice of the whole tensor; ndim < 2: its numel
  int64_t ng;         // numel of the whole tensor
  // Row-sharded steps only (0 otherwise).
  int64_t x1c;        // double offset in exchange round 1 of the column sums of g^2 [B][W]
  int64_t x1r;        // double offset in exchange round 1 of sum_i row_i per slice [B]
  int64_t x1p;        // double offset in exchange round 1 of sum(p^2)
  int64_t dloc;       // float offset in the workspace of this shard's D_j [B][W] (fused)
  // 8-bit first moment (beta1 with exp_avg_int8): int8 codes [N] and fp32
  // scales, one per group of kQ8Group values along the last dim.
  int8_t* mq;
  float* ms;          // [rows * qg]
  int64_t qg;         // groups per row: ceil(W / kQ8Group), ceil(n / kQ8Group) for ndim < 2
};
static_assert(sizeof(DevTensor) % 8 == 0, "DevTensor must stay 8-byte packed");

// Tensor classes: every streaming kernel is compiled per class so that each
// instantiation gets its own register allocation, and one launch covers all
// tensors of a class.
enum TensorClass : int32_t {
  kClsVecBF16 = 0,     // factored, vector path, bf16 grads
  kClsVecF32 = 1,      // factored, vector path, fp32 grads
  kClsScalarBF16 = 2,  // factored, element-wise path, bf16 grads
  kClsScalarF32 = 3,   // factored, element-wise path, fp32 grads
  kClsUnfactored = 4,  // ndim < 2 (any grad dtype)
  kClsRowsBF16 = 5,    // fused pass 1, bf16 grads, 2048 <= W <= 4096
  kClsWideBF16 = 6,    // fused pass 1, bf16 grads, 4096 < W <= 14336
  kClsFlatBF16 = 7,    // fused flat pass 1 (kFactoredFlat), bf16 grads
  kClsFlatF32 = 8,     // fused flat pass 1 (kFactoredFlat), fp32 grads
  kNumClasses = 9
};

// Per-call scalars and workspace regions, passed by value to every kernel.
struct StepArgs {
  const DevTensor* tensors;
  const int32_t* pf_tiles;   // [n+1] prefix of tiles over all tensors (tile0)
  const int32_t* pf_items;   // [n+1] prefix of statistics items (K2)
  double* alpha;             // [n]   effective lr
  double* coef;              // [n]   alpha / max(1, RMS(u)/d)
  double* mrow;              // mean(row) per slice, via DevTensor::mslot
  double* rowchunk;          // row-chunk sums of the updated row vector
  double* spart;             // [tiles] partial sum(u^2)
  double* ppart;             // [max(tiles, pass-1 units)] partial sum(p^2)
  double* ssum;              // [n] sum(u^2) of fused tensors
  double* dsum;              // per-chunk sum_j D_j / col_j of fused tensors
  float* rowpart;
  float* colpart;
  float* dpart;              // fused: column partials of g^2 / row_i
  double beta2;
  double rho;
  double eps1, eps2, clip, beta1, wd;
  int32_t scale_parameter;
  int32_t has_beta1;
  int32_t psq_valid;         // use DevTensor::psq instead of re-reading p
  int32_t want_psq_out;      // apply writes ppart for the carry
  int32_t* status;           // device status word (bit 0: a bounded wait gave up)
  int32_t stall_copies;      // testing hook: bulk-copy producers issue nothing
  // Row-sharded step (phase 0 = the single-call step; 1, 2, 3 = the begin,
  // middle and end calls).  round1/round2: the exchange buffers (sums over
  // all shards in the phase after the one that packs them).
  int32_t phase;
  int32_t q8;                // beta1 moment as int8 codes + group scales (DevTensor::mq, ms)
  double* round1;
  double* round2;
  float* dloc;
};

// Device status bits (the word is reset by every step call).
constexpr int32_t kStatusWaitTimeout = 1;
// A bounded wait gives up after this many SM clock cycles (~1 s).
constexpr long long kWaitCycles = 2000000000LL;

// The tensors one launch covers: members idx[m_begin..m_end) of a tensor
// index list, with pf[m] the first unit (tile or item) of member m relative to
// pf[m_begin] (the kernel copies pf[m_begin..m_end] to shared memory).
struct Range {
  const int32_t* pf;
  const int32_t* idx;
  int32_t m_begin, m_end;
};

// Kernel kinds, in launch order (also the profiling slots).
enum KernelId : int {
  kKPass1 = 0,     // read g (and p if needed): row/col partials, 1D v update
  kKStats = 1,     // row/col EMA update from the partials
  kKScalars = 2,   // per tensor: alpha, mean(row)
  kKPass2 = 3,     // read g: partial sum(u^2)
  kKClip = 4,      // per tensor: clip factor -> coef
  kKApply = 5,     // read g, p (exp_avg): write p (exp_avg), partial sum(p^2)
  kKPsq = 6,       // per tensor: sum(p^2) carry
  kNumKernels = 7
};

// Launchers (adafactor_kernels.cu).  Streaming kinds (pass1, pass2, apply)
// take a class and a member range; stats takes a member range over all
// tensors; the per-tensor kinds take a tensor count as grid.  Each returns the
// launch's cudaError_t.
cudaError_t launch_stream(KernelId k, TensorClass c, const StepArgs& a, const Range& r, int grid,
                          cudaStream_t s);
cudaError_t launch_stats(const StepArgs& a, const Range& r, int grid, cudaStream_t s);
cudaError_t launch_per_tensor(KernelId k, const StepArgs& a, int ntensors, cudaStream_t s);
// Kernel variant of a step: RMS(p) recomputed in pass 1 (1), first moment
// none / fp32 / 8-bit (x 2), sum(p_new^2) carried out (6); 0..11.
int kernel_variant(const StepArgs& a);
// Resident-CTA limit (CTAs per SM x SMs) of the kernel that a kind, tensor
// class and variant launch on a device (class and variant are ignored for
// the non-streaming kinds).
int kernel_grid_limit(KernelId k, TensorClass c, int variant, int device, cudaError_t* err);
const char* kernel_name(int k);

// How adafactor-step host code uploads the per-call header to the workspace.
enum HeaderStaging : int {
  kStagePinned = 0,    // library-owned pinned ring (cudaHostAlloc once), async copy
  kStagePageable = 1,  // pageable host buffer; no allocation by the CUDA runtime API
};

}  // namespace meo

#include "adafactor.h"

namespace meo {
// The step behind adafactor_step() (adafactor_api.cpp).  Per-kernel event
// timing is recorded only with kStagePinned.
adaf_status step_impl(const adaf_tensor* tensors, const adaf_state* states, int32_t n, int64_t step,
                      const adaf_hparams* hp, void* workspace, size_t workspace_bytes, void* stream,
                      HeaderStaging staging);
// Records msg for adafactor_last_error() on this thread; returns st.
adaf_status set_last_error(adaf_status st, const char* msg);
// Forgets the per-device addresses of the no-alloc scratch array
// (adafactor_noalloc.cu); adafactor_release_cache() calls it.
void noalloc_forget_addresses();
// Drop the device copies of the LAMB and CAME descriptor tables (they wait
// for the steps that read them); adafactor_release_cache calls them.
void lamb_forget_tables();
void came_forget_tables();
}  // namespace meo
