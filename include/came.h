/*
 * came.h — C ABI of the multi-tensor CAME step on one GB300 GPU (sm_103a).
 *
 * Operation.  The Colossal-AI distributed-optimizer article ("Colossal-AI
 * 分布式优化器全解析：Adafactor、CAME、GaLore 与 LAMB ...") describes CAME in
 * its overview table (Adafactor's low-rank second moment plus a confidence
 * matrix and a three-beta momentum, arXiv:2307.02047) and, in
 * "其余优化器的关键参数速查" (DistributedCAME), its defaults: lr = None (no
 * default: it must be given), eps = (1e-30, 1e-16), clip_threshold = 1.0,
 * betas = (0.9, 0.999, 0.9999), weight_decay = 0; the three betas track the
 * update, the squared gradient and the instability.  The rule is the CAME
 * algorithm of the cited paper.  Per tensor viewed as [B, H, W] slices (a
 * tensor with ndim < 2 is one row: its factored statistics become full
 * per-element vectors) and step t:
 *     r = b2 r + (1-b2) mean_j(g^2 + eps1),   c = b2 c + (1-b2) mean_i(g^2 + eps1)
 *     u = g / sqrt(r_i c_j / mean(r)),        uh = u / max(1, RMS(u) / d)
 *     m = b1 m + (1-b1) uh,                   U = (uh - m)^2
 *     R = b3 R + (1-b3) mean_j(U + eps2),     C = b3 C + (1-b3) mean_i(U + eps2)
 *     p = p - wd lr p - lr m / sqrt(R_i C_j / mean(R))
 * RMS(u) is over the whole tensor; means of r and R are per slice.
 *
 * Status codes, dtypes and the error message slot are shared with the
 * Adafactor ABI (adafactor.h).
 */
#ifndef MEO_CAME_H
#define MEO_CAME_H

#include <stddef.h>
#include <stdint.h>

#include "adafactor.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One tensor.  Device pointers to contiguous buffers owned by the caller;
 * ndim 0..ADAF_MAX_NDIM (ndim 0 is one value).  Any element-aligned address
 * is accepted: matrices whose last dim is a multiple of 8 with 16-byte
 * aligned p, g and exp_avg take 16-byte loads, others single-value loads. */
typedef struct came_tensor {
    float* p;                        /* fp32 parameter, updated in place      */
    const void* g;                   /* gradient, grad_dtype                  */
    int32_t grad_dtype;              /* ADAF_FLOAT32 or ADAF_BFLOAT16         */
    int32_t ndim;
    int64_t shape[ADAF_MAX_NDIM];
} came_tensor;

/* State of one tensor, fp32, zero before the first step.  ndim >= 2 (as
 * [B, H, W]): exp_avg_sq_row / exp_avg_res_row hold B*H values,
 * exp_avg_sq_col / exp_avg_res_col B*W; exp_avg_sq and exp_avg_res are
 * unused (may be NULL).  ndim < 2: exp_avg_sq and exp_avg_res hold numel
 * values, the row/col pointers are unused.  exp_avg always holds numel. */
typedef struct came_state {
    float* exp_avg;
    float* exp_avg_sq_row;
    float* exp_avg_sq_col;
    float* exp_avg_res_row;
    float* exp_avg_res_col;
    float* exp_avg_sq;
    float* exp_avg_res;
} came_state;

typedef struct came_hparams {
    double lr;                     /* required, >= 0                         */
    double eps1, eps2;             /* >= 0: added to g^2 and to U            */
    double clip_threshold;         /* d > 0                                  */
    double beta1, beta2, beta3;    /* in [0, 1)                              */
    double weight_decay;           /* >= 0, decoupled: p -= wd lr p          */
} came_hparams;

/* Article defaults with lr = 0 (a learning rate must be set by the caller). */
void came_default_hparams(came_hparams* hp);

/* Host-only check: all finite, lr >= 0, eps >= 0, clip_threshold > 0,
 * 0 <= beta < 1, weight_decay >= 0.  ADAF_ERR_INVALID_ARGUMENT otherwise. */
adaf_status came_validate(const came_hparams* hp);

/* Workspace bytes came_step() needs (host only, sizes only).  Errors:
 * ADAF_ERR_INVALID_ARGUMENT (malformed list), ADAF_ERR_UNSUPPORTED (more than
 * 2^31 tiles, a dim above 2^31, more than 2^40 values in a tensor). */
adaf_status came_workspace_size(const came_tensor* tensors, int32_t n, size_t* bytes);

/* One CAME step over the list, enqueued on `stream` (cudaStream_t; NULL is
 * the legacy default stream).  workspace: >= came_workspace_size() bytes of
 * device memory, 256-byte aligned, not in use by another call in flight.
 * step >= 1.  All checks run before the first CUDA call.  The descriptor
 * table is read from a device copy the library keeps (up to 8 distinct tables
 * per device) when one holds the same bytes; a new table goes through a
 * pinned ring of 4 host buffers into a new device copy (cudaMalloc), and the
 * call waits on the host only when the upload of 4 uploads earlier has not
 * run.  adafactor_release_cache() frees the copies.  Errors: ADAF_ERR_INVALID_ARGUMENT,
 * ADAF_ERR_UNSUPPORTED, ADAF_ERR_WORKSPACE_TOO_SMALL, ADAF_ERR_CUDA. */
adaf_status came_step(const came_tensor* tensors, const came_state* states, int32_t n, int64_t step,
                      const came_hparams* hp, void* workspace, size_t workspace_bytes, void* stream);

/* Per-kernel timing with CUDA events (as for the Adafactor step): a slot is
 * one kernel kind; its time covers the launches of that kind in a call (one
 * per tensor class that has members), and launches[k] counts those kernel
 * launches. */
adaf_status came_profile_enable(int32_t on);
adaf_status came_profile_read(double* ms, int64_t* launches, int32_t nk);
int32_t came_num_kernels(void);
const char* came_kernel_name(int32_t k);

#ifdef __cplusplus
}
#endif

#endif /* MEO_CAME_H */
