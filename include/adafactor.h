/*
 * adafactor.h — C ABI of the GB300 Adafactor step library (libmeo_adafactor.so).
 *
 * One call, adafactor_step(), applies one Adafactor step to a whole list of
 * tensors at once, on the caller's CUDA stream, with a fixed handful of kernel
 * launches whatever the list length.  The method is the one described in the
 * Colossal-AI distributed-optimizer article ("Colossal-AI 分布式优化器全解析：
 * Adafactor、CAME、GaLore 与 LAMB 如何无缝对接 Tensor Parallel 与 ZeRO",
 * blog.gitcode.com):
 *   - optimizer table ("四种优化器：原理速览", Adafactor row): the [H, W] second
 *     moment is kept as a row vector [H] and a column vector [W];
 *   - Step 3: defaults, relative step size, the manual-lr error, warmup_init,
 *     optional beta1 first moment, factored (ndim >= 2) vs. full second moment;
 *   - Step 4: the RMS helper;
 *   - Step 5: beta2t = 1 - t^decay_rate, the RMS clip of the update, the
 *     relative-step lr scaled by max(eps[1], RMS(param)).
 *
 * Per tensor, with t the 1-based step and every RMS over the whole tensor:
 *   rho   = relative_step ? min(warmup_init ? 1e-6 t : 1e-2, 1/sqrt(t)) : lr
 *   alpha = scale_parameter ? rho * max(eps2, RMS(param before the step)) : rho
 *   beta2 = 1 - t^decay_rate
 *   ndim >= 2, viewed as [B, H, W] (B = product of the leading dims):
 *     row[b,i] <- beta2 row[b,i] + (1-beta2) mean_j (g^2 + eps1)
 *     col[b,j] <- beta2 col[b,j] + (1-beta2) mean_i (g^2 + eps1)
 *     u = g * (row[b,i] / mean_i row[b,i])^-1/2 * col[b,j]^-1/2
 *   ndim < 2:
 *     v <- beta2 v + (1-beta2) (g^2 + eps1);   u = g / sqrt(v)
 *   u <- alpha * u / max(1, RMS(u) / clip_threshold)
 *   beta1 set:  exp_avg <- beta1 exp_avg + (1-beta1) u;  u <- exp_avg
 *   param <- param - weight_decay * alpha * param - u
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     contiguous row-major.  The library never allocates device memory; the
 *     caller owns params, grads, states and the workspace.
 *   - Nothing is checked lazily: every argument check runs before the first
 *     CUDA call, so a call that returns an error has changed nothing.
 *   - No C++ exception crosses this interface.  A failing call returns a
 *     non-zero adaf_status and leaves a message for adafactor_last_error()
 *     (per host thread).
 */
#ifndef MEO_ADAFACTOR_H
#define MEO_ADAFACTOR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum adaf_status {
    ADAF_OK = 0,
    ADAF_ERR_INVALID_ARGUMENT = 1,   /* bad hyper-parameter, pointer, shape or dtype */
    ADAF_ERR_UNSUPPORTED = 2,        /* valid but outside what this build handles    */
    ADAF_ERR_WORKSPACE_TOO_SMALL = 3,
    ADAF_ERR_CUDA = 4                /* a CUDA runtime call or launch failed         */
} adaf_status;

typedef enum adaf_dtype {
    ADAF_FLOAT32 = 0,
    ADAF_BFLOAT16 = 1
} adaf_dtype;

#define ADAF_MAX_NDIM 8

/* One parameter tensor and its gradient.
 *   param      fp32 [N], updated in place; 4-byte aligned.
 *   grad       grad_dtype [N], read only; aligned to its element size.
 *   ndim       0..8.  ndim >= 2: factored over the last two dims
 *              (B = shape[0]*...*shape[ndim-3], H = shape[ndim-2],
 *              W = shape[ndim-1]).  ndim 0 or 1: full second moment.
 *   shape      the first ndim entries are used; each >= 0.
 * A tensor with N = 0 is skipped.  16-byte aligned param/grad/exp_avg with
 * W a multiple of 8 take the vectorised kernels; anything else takes the
 * element-wise kernels, with the same results. */
typedef struct adaf_tensor {
    float* param;
    const void* grad;
    int32_t grad_dtype;
    int32_t ndim;
    int64_t shape[ADAF_MAX_NDIM];
} adaf_tensor;

/* The optimizer state of one tensor (device pointers, fp32, zeroed by the
 * caller before step 1).  Unused members may be NULL.
 *   exp_avg_sq_row  [B*H]  factored tensors
 *   exp_avg_sq_col  [B*W]  factored tensors
 *   exp_avg_sq      [N]    tensors with ndim < 2
 *   exp_avg         [N]    required when has_beta1
 *   param_sq_sum    one double, optional.  When non-NULL the step writes
 *                  sum(param^2) of the parameter it leaves behind, so that the
 *                  next step can take RMS(param) without re-reading param
 *                  (see adaf_hparams.param_sq_sum_valid). */
typedef struct adaf_state {
    float* exp_avg_sq_row;
    float* exp_avg_sq_col;
    float* exp_avg_sq;
    float* exp_avg;
    double* param_sq_sum;
    /* 8-bit first moment (adaf_hparams.exp_avg_int8; exp_avg is then unused):
     *   exp_avg_codes   int8 [N], 4-byte aligned (16-byte for the vector path)
     *   exp_avg_scales  fp32 [R * ceil(L / 128)], L = the last dim (N for
     *                   ndim < 2), R = N / L: one scale per group of 128
     *                   values along the last dim.  Zeroed before step 1. */
    int8_t* exp_avg_codes;
    float* exp_avg_scales;
} adaf_state;

/* Hyper-parameters (Step 3 of the article).  adafactor_default_hparams()
 * fills the article's defaults: no lr, eps=(1e-30, 1e-3), clip_threshold 1.0,
 * decay_rate -0.8, no beta1, weight_decay 0, scale_parameter, relative_step,
 * no warmup_init.
 *   param_sq_sum_valid  1 = every state's param_sq_sum holds sum(param^2) of
 *                       the parameter as it is now (written by the previous
 *                       step and untouched since); the step then skips one
 *                       read of every parameter.  0 = recompute it.  Only read
 *                       when scale_parameter is set. */
typedef struct adaf_hparams {
    double lr;
    int32_t has_lr;
    double eps1;
    double eps2;
    double clip_threshold;
    double decay_rate;
    double beta1;
    int32_t has_beta1;
    double weight_decay;
    int32_t scale_parameter;
    int32_t relative_step;
    int32_t warmup_init;
    int32_t param_sq_sum_valid;
    /* 1 = keep the beta1 first moment as int8 codes with one fp32 scale per
     * group of 128 values along the last dim (the block quantisation of the
     * ms-swift article's Q-GaLore section: scale = absmax / 127, symmetric
     * codes).  Each step dequantises the old moment (code * scale), forms
     * beta1 * old + (1 - beta1) * u, uses it unquantised for the update and
     * stores it re-quantised: scale = amax / 127, code = rint(m * (127 / amax))
     * in fp32, amax the group's max |m| (code and scale 0 if amax = 0).
     * Requires has_beta1.  Default 0. */
    int32_t exp_avg_int8;
} adaf_hparams;

/* Fills *hp with the article's defaults (Step 3).  hp must not be NULL. */
void adafactor_default_hparams(adaf_hparams* hp);

/* Checks the hyper-parameters alone (no CUDA call).  Errors, all
 * ADAF_ERR_INVALID_ARGUMENT:
 *   has_lr && relative_step      "Cannot combine manual lr and relative_step=True options"
 *                                (the error quoted in Step 3)
 *   warmup_init && !relative_step  (Step 3: warmup_init forces relative_step)
 *   !has_lr && !relative_step    "relative_step=False requires a manual lr"
 *   clip_threshold not finite or <= 0; has_lr with lr not finite or < 0;
 *   eps1, eps2 or weight_decay not finite or < 0; decay_rate not finite;
 *   has_beta1 with beta1 not in [0, 1);
 *   exp_avg_int8 without has_beta1. */
adaf_status adafactor_validate(const adaf_hparams* hp);

/* Bytes of device workspace adafactor_step() needs for this tensor list
 * (256-byte aligned start required).  Pure host computation, no CUDA call.
 * Fails with ADAF_ERR_INVALID_ARGUMENT on a malformed list (n < 0, NULL
 * tensors with n > 0, bad ndim/shape/dtype) and ADAF_ERR_UNSUPPORTED when the
 * list needs more than 2^31-1 work tiles. */
adaf_status adafactor_workspace_size(const adaf_tensor* tensors, int32_t n, size_t* bytes);

/* One Adafactor step over tensors[0..n) with states[0..n), step t = `step`
 * (>= 1), enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 * stream).  The call only enqueues work and reads no device memory from the
 * host.  The per-call descriptor table (pointers, shapes, work lists) is
 * built on the host; the library keeps device copies of up to 8 distinct
 * tables per device, and a call whose table equals a kept one reads that copy
 * and uploads nothing (a one-thread kernel on `stream` clears the status
 * word).  A new table is staged in a ring of 4 pinned host buffers per device
 * and read from there by a small kernel on `stream`, into a new device copy
 * (no copy engine: host-to-device copies queued on other streams do not hold
 * it back); such a call waits on the host only when the upload of the call 4
 * uploads earlier has not yet run.  A step whose table is new on the device
 * allocates its copy with cudaMalloc.  Params and states
 * are updated in place; grads are read only.  The workspace (>= the size
 * reported by adafactor_workspace_size, 256-byte aligned) is scratch owned by
 * this call until the enqueued work completes: calls that may run
 * concurrently on the device need distinct workspaces.
 * Errors: ADAF_ERR_INVALID_ARGUMENT (hyper-parameters as in
 * adafactor_validate; step < 1; NULL or misaligned pointers; missing state
 * buffers for a tensor's path; has_beta1 without exp_avg or, with
 * exp_avg_int8, without exp_avg_codes / exp_avg_scales), ADAF_ERR_UNSUPPORTED,
 * ADAF_ERR_WORKSPACE_TOO_SMALL, ADAF_ERR_CUDA (a CUDA call or a kernel launch
 * failed; work enqueued before the failure may have run). */
adaf_status adafactor_step(const adaf_tensor* tensors, const adaf_state* states, int32_t n,
                           int64_t step, const adaf_hparams* hp, void* workspace,
                           size_t workspace_bytes, void* stream);

/* adafactor_step_noalloc — the same step as adafactor_step(), with no
 * workspace argument and no device, pinned-host or event allocation by the
 * library (no cudaMalloc/cudaFree, no cudaHostAlloc, no cudaEventCreate).  The
 * article has no counterpart: this entry point exists for callers that cannot
 * hand out device memory, e.g. code running while a memory pool owns all of
 * the device memory and forbids cudaMalloc, code where an allocation would
 * synchronise the device at a point where that is not allowed, or hosts that
 * link the library without an allocator of their own.  The host-side planner
 * still builds each call's descriptor table in ordinary heap memory.
 *   - Scratch: a fixed ADAF_NOALLOC_SCRATCH_BYTES (64 MiB) __device__ array
 *     inside the library.  Every GPU that loads the library holds it until the
 *     process exits.  A tensor list whose scratch need (adafactor_workspace_size)
 *     is larger is rejected with ADAF_ERR_WORKSPACE_TOO_SMALL and a message
 *     giving both sizes, before any CUDA call.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress, with that device current) and keeps it
 *     for later calls; make that first call before any stream capture on the
 *     device.  adafactor_release_cache() forgets the kept addresses: call it
 *     after a device reset (cudaDeviceReset) before the next call.
 *   - The descriptor table of each call is copied from a host buffer that
 *     lives only for the call.  While `stream` is capturing, the call returns
 *     ADAF_ERR_UNSUPPORTED and enqueues nothing.
 *   - Sharing: every call on a device uses the same array and finds the last
 *     call's contents there.  The step rewrites everything it reads (the
 *     status word is reset by each call), so nothing needs clearing by the
 *     caller, but calls whose work may overlap on the GPU (different streams
 *     without ordering, several host threads) race on the array: order them
 *     on one stream.
 *   - Per-kernel event timing (adafactor_profile_*) does not cover this entry
 *     point; adafactor_noalloc_device_status() reads its status word.
 * Arguments, errors and results are those of adafactor_step() without the
 * workspace, plus ADAF_ERR_UNSUPPORTED for a capturing stream. */
#define ADAF_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
adaf_status adafactor_step_noalloc(const adaf_tensor* tensors, const adaf_state* states, int32_t n,
                                   int64_t step, const adaf_hparams* hp, void* stream);

/* Device-side status of the most recent adafactor_step_noalloc() on the
 * current device (the status word at the start of its scratch array, as
 * adafactor_device_status() reads it from a workspace): waits on `stream`,
 * then stores the word in *status (0, or ADAF_DEVICE_WAIT_TIMEOUT when a
 * bounded wait inside a kernel gave up and that step's results are not
 * valid).  Allocates nothing; synchronises the host with `stream`.  The
 * article has no counterpart.  Errors: ADAF_ERR_INVALID_ARGUMENT (status
 * NULL), ADAF_ERR_CUDA. */
adaf_status adafactor_noalloc_device_status(void* stream, int32_t* status);

/* ---- Row-sharded step (tensor rows split over several ranks) ------------
 * Step 4 of the article runs Adafactor on parameters split over a tensor-
 * parallel / ZeRO group: the factored statistics and the RMS partial sums are
 * summed over the group (all-reduce) before the update.  These three calls
 * are that step for a rank that holds a contiguous block of rows of every
 * tensor (a row shard); the sums over the group are the caller's collective
 * (e.g. an NCCL or gloo all-reduce), made between the calls.  Everything that
 * needs only the rank's own rows stays local: the row statistics, the update
 * and the parameters.
 *
 * Per tensor k, the rank passes its shard as an ordinary adaf_tensor (shape
 * with the rank's rows: [..., h_k, W] for ndim >= 2, [n_k] for ndim < 2, at
 * least one row or element) and shards[k].global_rows = the rows per slice of
 * the whole tensor (ndim >= 2) or its numel (ndim < 2).  States: exp_avg_sq_row,
 * exp_avg, exp_avg_sq hold the rank's rows / elements; exp_avg_sq_col holds
 * the whole [B*W] column statistic on every rank (every rank updates it
 * identically); param_sq_sum carries the rank's own sum(param^2).  Every rank
 * passes the same tensor order, the same leading dims and W, step and
 * hyper-parameters.
 *
 *   adafactor_shard_begin   pass 1 over the rank's rows, then writes to
 *                           round1 the rank's column sums of g^2, its sum of
 *                           the updated row statistic per slice, and its
 *                           sum(param^2).
 *   caller                  round1 <- sum of round1 over the ranks (float64)
 *   adafactor_shard_middle  column statistics, mean(row) and RMS(param) from
 *                           the summed round1; writes to round2 the rank's
 *                           sum(u^2) per tensor.
 *   caller                  round2 <- sum of round2 over the ranks (float64)
 *   adafactor_shard_end     the RMS clip from the summed round2, the update.
 *
 * The three calls of one step take the same arguments and the same workspace
 * (which carries intermediate results from call to call: do not use it for
 * anything else in between), on the same stream or with the order kept by
 * the caller.  round1 / round2 are device buffers of float64 of the sizes
 * adafactor_shard_sizes() gives (the same on every rank); they are read only
 * after the caller's sum.  With one rank and no collective the three calls
 * compute what adafactor_step() computes (sums in another order).
 * Errors: those of adafactor_step(), plus ADAF_ERR_INVALID_ARGUMENT for NULL
 * shards or round buffers, global_rows smaller than the shard's rows, or a
 * shard with no row of some tensor. */
typedef struct adaf_shard {
    int64_t global_rows;
} adaf_shard;

/* Sizes for a row-sharded step over tensors[0..n) (host only, no CUDA call):
 * the workspace (256-byte aligned start) and the two exchange buffers. */
adaf_status adafactor_shard_sizes(const adaf_tensor* tensors, const adaf_shard* shards, int32_t n,
                                  size_t* workspace_bytes, size_t* round1_bytes, size_t* round2_bytes);
adaf_status adafactor_shard_begin(const adaf_tensor* tensors, const adaf_state* states,
                                  const adaf_shard* shards, int32_t n, int64_t step,
                                  const adaf_hparams* hp, void* workspace, size_t workspace_bytes,
                                  double* round1, void* stream);
adaf_status adafactor_shard_middle(const adaf_tensor* tensors, const adaf_state* states,
                                   const adaf_shard* shards, int32_t n, int64_t step,
                                   const adaf_hparams* hp, void* workspace, size_t workspace_bytes,
                                   const double* round1, double* round2, void* stream);
adaf_status adafactor_shard_end(const adaf_tensor* tensors, const adaf_state* states,
                                const adaf_shard* shards, int32_t n, int64_t step,
                                const adaf_hparams* hp, void* workspace, size_t workspace_bytes,
                                const double* round2, void* stream);

/* Device-side status of the most recent adafactor_step() that used this
 * workspace: waits on the stream, then stores the status word in *status.
 * 0 = no problem.  Bit 0 (ADAF_DEVICE_WAIT_TIMEOUT): a bounded wait inside a
 * kernel gave up (about one second without progress) and the kernel stopped
 * early, so that step's results are not valid.  The word is reset by every
 * adafactor_step() call.  Synchronises the host with `stream`.
 * Errors: ADAF_ERR_INVALID_ARGUMENT, ADAF_ERR_CUDA. */
#define ADAF_DEVICE_WAIT_TIMEOUT 1
adaf_status adafactor_device_status(const void* workspace, void* stream, int32_t* status);

/* Testing hook for the device-side failure detection.  With
 * adafactor_debug_stall_copies(1), the bulk-copy producers of every following
 * adafactor_step() on any thread issue no copies, so the consumers' bounded
 * waits run out (about a second each): the step then ends early with
 * ADAF_DEVICE_WAIT_TIMEOUT in the device status word and garbage results, and
 * the CUDA context stays usable.  adafactor_debug_stall_copies(0) restores
 * normal operation.  For tests only; no other effect. */
void adafactor_debug_stall_copies(int32_t on);

/* Message of the last failing call on this host thread ("" if none). */
const char* adafactor_last_error(void);

/* Frees the library's caches for every device: the pinned staging buffers
 * and events, and the device copies of descriptor tables that adafactor_step,
 * the row-sharded calls, lamb_step and came_step keep (up to 8 per device and
 * optimizer, each the size of one call's table: a step whose table bytes equal
 * a kept copy's reads that copy instead of uploading its table again).  Waits
 * for the steps that read those copies.  Call only when no step work is in
 * flight, and after a device reset before the next step. */
void adafactor_release_cache(void);

/* ---- Kernel timing (CUDA events on the launching stream) ----------------
 * adafactor_profile_enable(1) makes every following adafactor_step() record a
 * CUDA event pair around each of its kernel launches on the launch stream;
 * adafactor_profile_read() waits for the recorded events, adds the elapsed
 * time per slot into ms[k] and the launch count into launches[k] for
 * k < min(nk, adafactor_num_kernels()), and forgets the records.  A slot is
 * one kernel kind, or one kind and tensor class for the streaming kernels;
 * adafactor_kernel_name(k) names it ("k_apply[vec_bf16]", "k_stats", ...).
 * adafactor_profile_enable(0) stops recording.  Errors: ADAF_ERR_CUDA. */
adaf_status adafactor_profile_enable(int32_t on);
adaf_status adafactor_profile_read(double* ms, int64_t* launches, int32_t nk);
int32_t adafactor_num_kernels(void);
const char* adafactor_kernel_name(int32_t k);

#ifdef __cplusplus
}
#endif

#endif /* MEO_ADAFACTOR_H */
