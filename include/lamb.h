/*
 * lamb.h — C ABI of the multi-tensor LAMB step on one GB300 GPU (sm_103a).
 *
 * Operation.  The Colossal-AI distributed-optimizer article ("Colossal-AI
 * 分布式优化器全解析：Adafactor、CAME、GaLore 与 LAMB ...") lists LAMB in its
 * overview table (a layer-wise adaptive update for very large batches) and,
 * in "其余优化器的关键参数速查" (DistributedLAMB), its defaults: lr = 1e-3,
 * betas = (0.9, 0.999), eps = 1e-6, weight_decay = 0, bias_correction = true,
 * and its core: a per-layer trust ratio between the norm of the parameter and
 * the norm of the update.  The rule itself is the LAMB algorithm of the paper
 * the article cites (arXiv:1904.00962).  Per tensor ("layer") and step t:
 *     m  = beta1 m + (1 - beta1) g
 *     v  = beta2 v + (1 - beta2) g^2
 *     mh = m / (1 - beta1^t),  vh = v / (1 - beta2^t)   (bias_correction;
 *                                                        else mh = m, vh = v)
 *     r  = mh / (sqrt(vh) + eps) + weight_decay * p
 *     p  = p - lr * (||p|| / ||r||) * r    (trust ratio 1 where a norm is 0)
 * Norms are over the whole tensor, with p as it is at the start of the step.
 *
 * Status codes, dtypes and the error message slot are shared with the
 * Adafactor ABI (adafactor.h): every call returns an adaf_status and leaves a
 * message for adafactor_last_error() when it fails.
 */
#ifndef MEO_LAMB_H
#define MEO_LAMB_H

#include <stddef.h>
#include <stdint.h>

#include "adafactor.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One tensor of the list.  All pointers are device pointers to contiguous
 * buffers of numel values owned by the caller; the library keeps none of
 * them after the call returns (the launches use them in stream order).
 * Any alignment is accepted: 16-byte aligned tensors (8-byte for a bf16
 * gradient) take 4-value loads, others single-value loads. */
typedef struct lamb_tensor {
    float* p;            /* fp32 parameter, updated in place                  */
    const void* g;       /* gradient, grad_dtype                              */
    int32_t grad_dtype;  /* ADAF_FLOAT32 or ADAF_BFLOAT16                     */
    int64_t numel;       /* >= 0; 0 leaves the tensor untouched               */
    float* exp_avg;      /* m, fp32, zero before the first step               */
    float* exp_avg_sq;   /* v, fp32, zero before the first step               */
} lamb_tensor;

typedef struct lamb_hparams {
    double lr;               /* >= 0                                        */
    double beta1, beta2;     /* in [0, 1)                                   */
    double eps;              /* >= 0                                        */
    double weight_decay;     /* >= 0                                        */
    int32_t bias_correction; /* non-zero: divide m, v by 1 - beta^t         */
} lamb_hparams;

/* Checks the hyper-parameters (finite, lr >= 0, eps >= 0, 0 <= beta < 1,
 * weight_decay >= 0).  Host only.  ADAF_ERR_INVALID_ARGUMENT on a bad value. */
adaf_status lamb_validate(const lamb_hparams* hp);

/* Workspace bytes lamb_step() needs for this list (host only; depends on the
 * sizes, not on the pointers).  ADAF_ERR_INVALID_ARGUMENT on a malformed list
 * (n < 0, NULL tensors with n > 0, negative numel, unknown dtype);
 * ADAF_ERR_UNSUPPORTED when a tensor has more than 2^40 values or the list
 * more than 2^31 work units. */
adaf_status lamb_workspace_size(const lamb_tensor* tensors, int32_t n, size_t* bytes);

/* One LAMB step over the list, enqueued on `stream` (a cudaStream_t; NULL is
 * the legacy default stream).  workspace: device memory of at least
 * lamb_workspace_size() bytes, 256-byte aligned, not used by another call
 * that is in flight.  Three launches: moments + per-unit norm partials,
 * per-tensor trust ratios, update.  step >= 1.  All argument checks run
 * before the first CUDA call.  The per-call descriptor table is read from a
 * device copy the library keeps (up to 8 distinct tables per device) when one
 * holds the same bytes; a new table goes through a pinned ring of 4 host
 * buffers into a new device copy (cudaMalloc), and the call waits on the host
 * only when the upload of 4 uploads earlier has not run.  adafactor_release_cache()
 * frees the copies.  Errors: ADAF_ERR_INVALID_ARGUMENT,
 * ADAF_ERR_UNSUPPORTED, ADAF_ERR_WORKSPACE_TOO_SMALL, ADAF_ERR_CUDA. */
adaf_status lamb_step(const lamb_tensor* tensors, int32_t n, int64_t step, const lamb_hparams* hp,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Copies the n trust ratios of the last lamb_step() on this workspace into
 * host memory (float64, list order), after synchronising `stream`.
 * Errors: ADAF_ERR_INVALID_ARGUMENT (NULL pointers, n < 0), ADAF_ERR_CUDA. */
adaf_status lamb_trust_ratios(const void* workspace, int32_t n, double* out, void* stream);

/* Per-kernel timing with CUDA events on the launching stream, as for the
 * Adafactor step: enable, run steps, read the summed milliseconds and launch
 * counts per kernel (nk slots; lamb_num_kernels() names them). */
adaf_status lamb_profile_enable(int32_t on);
adaf_status lamb_profile_read(double* ms, int64_t* launches, int32_t nk);
int32_t lamb_num_kernels(void);
const char* lamb_kernel_name(int32_t k);

#ifdef __cplusplus
}
#endif

#endif /* MEO_LAMB_H */
