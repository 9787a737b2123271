/*
 * Adafactor step oracle: plain, slow, float64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or run this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library: it is written from the method's description alone.
 *
 * Source of the method: the Colossal-AI distributed-optimizer article
 * ("Colossal-AI 分布式优化器全解析：Adafactor、CAME、GaLore 与 LAMB ...",
 * blog.gitcode.com), sections
 *   - "四种优化器：原理速览" table, Adafactor row: the [H, W] second moment is
 *     approximated by a row vector times a column vector, O(H*W) -> O(H+W);
 *   - "Step 3" (初始化模型与分布式优化器): defaults lr=None, eps=(1e-30, 1e-3),
 *     clip_threshold=1.0, decay_rate=-0.8, beta1=None, weight_decay=0.0,
 *     scale_parameter=True, relative_step=True, warmup_init=False; relative
 *     step size min(1e-2, 1/sqrt(step)) (warmup_init: 1e-6*step in place of
 *     1e-2); manual lr with relative_step is an error; warmup_init needs
 *     relative_step; beta1 set => exp_avg kept; ndim >= 2 => factored
 *     exp_avg_sq_row [H] / exp_avg_sq_col [W], otherwise a full exp_avg_sq;
 *   - "Step 4" (初始化 plugin 与 booster): the _rms helper (root mean square);
 *   - "Step 5" (训练循环): beta2t = 1 - step^decay_rate; the update is divided
 *     by max(1, RMS(update)/clip_threshold), then scaled by the relative-step
 *     lr; with scale_parameter the lr is multiplied by max(eps[1], RMS(param)).
 *
 * Readings where the article is silent (each one is also listed in the
 * design notes):
 *   - the factored statistics are EMAs of the row and column means of
 *     g*g + eps[0]; the update is g * (row_i / mean(row))^-1/2 * col_j^-1/2,
 *     with mean(row) taken over the freshly updated row vector;
 *   - tensors with ndim > 2 are viewed as [B, H, W] and factored over the last
 *     two dims, each leading index b with its own row/col vectors; RMS(update)
 *     and RMS(param) are taken over the whole tensor;
 *   - RMS(param) uses the parameter as it is at the start of the step;
 *   - exp_avg accumulates the clipped, lr-scaled update;
 *   - weight decay is decoupled: p <- p - weight_decay * lr * p, applied before
 *     the update is subtracted;
 *   - relative_step=False without a manual lr is an error;
 *   - a tensor with no elements is left untouched (nothing to update).
 *
 * Every quantity is float64; the step count t is 1-based.
 *
 * 8-bit first moment (oracle_adafactor_step_q8): the block quantisation of
 * the ms-swift GaLore / Q-GaLore article ("双重压缩：Q-Galore 的量化飞跃"
 * section) applied to exp_avg.  Its quantize_tensor listing takes groups of
 * 128 values, scale = (max |x| over the group) / 127, and code = the quotient
 * x / scale rounded (torch's round: half to even) and clamped to [-128, 127];
 * its dequantize_tensor is code * scale.  The surrounding QGaloreAdam listing
 * dequantises the stored moment before the update is formed from it
 * ("反投影前必须反量化": dequantise before projecting back).  Readings:
 *   - groups are 128 consecutive values along the last dim (a tensor with
 *     ndim < 2 is one row); the last group of a row may be shorter (the
 *     listing's flat reshape(-1, 128) is the same grouping whenever the last
 *     dim is a multiple of 128);
 *   - arithmetic of the quantiser in fp32, the listing's tensor precision:
 *     the new moment is rounded to fp32, amax = max |m|, scale = amax / 127,
 *     code = rint(m / scale) (two correctly rounded fp32 divisions, ties to
 *     even); a group whose scale is 0 (all zero, or amax / 127 below the
 *     smallest fp32 value) stores codes 0 (the listing would divide by 0);
 *   - one step: old moment = code * scale (fp32 product); new moment
 *     m = beta1 * old + (1 - beta1) * u in float64; m is quantised; the
 *     update applied to the parameter is the dequantised new moment
 *     code * scale (fp32 product), the value the stored state holds.
 * The three parts are exported separately (oracle_q8_moment,
 * oracle_q8_quantize, oracle_q8_apply) so that a caller can inspect the
 * codes between them; oracle_adafactor_step_q8 runs them in order.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    double lr;
    int32_t has_lr;
    double eps1;            /* eps[0]: added to g*g */
    double eps2;            /* eps[1]: floor of RMS(param) */
    double clip_threshold;  /* d */
    double decay_rate;
    double beta1;
    int32_t has_beta1;
    double weight_decay;
    int32_t scale_parameter;
    int32_t relative_step;
    int32_t warmup_init;
} oracle_hparams;

enum { ORACLE_OK = 0, ORACLE_INVALID = 1, ORACLE_NOMEM = 2 };

static void set_err(char* err, int errlen, const char* msg) {
    if (err && errlen > 0) {
        strncpy(err, msg, (size_t)errlen - 1);
        err[errlen - 1] = '\0';
    }
}

/* Argument rules of Step 3: manual lr and relative_step exclude each other;
 * warmup_init forces relative_step.  Reading: without relative_step a manual
 * lr is required.  The remaining range checks are plain sanity. */
int oracle_check_hparams(const oracle_hparams* hp, char* err, int errlen) {
    if (hp->has_lr && hp->relative_step) {
        set_err(err, errlen, "Cannot combine manual lr and relative_step=True options");
        return ORACLE_INVALID;
    }
    if (hp->warmup_init && !hp->relative_step) {
        set_err(err, errlen, "warmup_init=True requires relative_step=True");
        return ORACLE_INVALID;
    }
    if (!hp->has_lr && !hp->relative_step) {
        set_err(err, errlen, "relative_step=False requires a manual lr");
        return ORACLE_INVALID;
    }
    if (!(hp->clip_threshold > 0.0)) {
        set_err(err, errlen, "clip_threshold must be > 0");
        return ORACLE_INVALID;
    }
    return ORACLE_OK;
}

/* Step 3: relative step size min(1e-2, 1/sqrt(t)); with warmup_init the 1e-2
 * is replaced by 1e-6 * t.  Without relative_step the manual lr is used. */
double oracle_rho(const oracle_hparams* hp, int64_t t) {
    if (!hp->relative_step) return hp->lr;
    double cap = hp->warmup_init ? 1e-6 * (double)t : 1e-2;
    double inv_sqrt_t = 1.0 / sqrt((double)t);
    return cap < inv_sqrt_t ? cap : inv_sqrt_t;
}

/* Step 5: beta2t = 1 - t^decay_rate. */
double oracle_beta2(const oracle_hparams* hp, int64_t t) {
    return 1.0 - pow((double)t, hp->decay_rate);
}

/* Step 4's _rms: square root of the mean of squares. */
static double rms(const double* x, int64_t n) {
    double s = 0.0;
    for (int64_t k = 0; k < n; ++k) s += x[k] * x[k];
    return sqrt(s / (double)n);
}

/*
 * One Adafactor step on one tensor, in place.
 *   p        [N]      parameter (updated)
 *   g        [N]      gradient
 *   shape    [ndim]   row-major shape; ndim >= 2 => factored
 *   row      [B*H]    exp_avg_sq_row (factored only; else ignored)
 *   col      [B*W]    exp_avg_sq_col (factored only; else ignored)
 *   v        [N]      exp_avg_sq     (ndim < 2 only; else ignored)
 *   exp_avg  [N]      first moment   (has_beta1 only; else ignored)
 *   t        1-based step number
 * Returns ORACLE_OK, or ORACLE_INVALID with a message in err.
 */
/* The clipped, lr-scaled update u [N] of one step (before the first moment),
 * updating the second-moment state in place; *alpha_out = the step's lr.
 * *u_out is malloc'ed (NULL for an empty tensor). */
static int compute_update(const double* p, const double* g, int32_t ndim, const int64_t* shape,
                          double* row, double* col, double* v, int64_t t, const oracle_hparams* hp,
                          double** u_out, double* alpha_out, int64_t* n_out, char* err, int errlen) {
    *u_out = NULL;
    int rc = oracle_check_hparams(hp, err, errlen);
    if (rc != ORACLE_OK) return rc;
    if (t < 1) {
        set_err(err, errlen, "step must be >= 1");
        return ORACLE_INVALID;
    }
    if (ndim < 0 || ndim > 8) {
        set_err(err, errlen, "ndim must be in [0, 8]");
        return ORACLE_INVALID;
    }
    int64_t n = 1;
    for (int32_t k = 0; k < ndim; ++k) n *= shape[k];
    *n_out = n;
    if (n == 0) return ORACLE_OK;

    /* Step 3 / Step 5: lr = rho_t, times max(eps[1], RMS(p)) when
     * scale_parameter, with p as it is before this step touches it. */
    double rho = oracle_rho(hp, t);
    double alpha = rho;
    if (hp->scale_parameter) {
        double r = rms(p, n);
        alpha = rho * (hp->eps2 > r ? hp->eps2 : r);
    }
    double beta2 = oracle_beta2(hp, t);

    double* u = (double*)malloc((size_t)n * sizeof(double));
    if (!u) {
        set_err(err, errlen, "out of host memory");
        return ORACLE_NOMEM;
    }

    if (ndim >= 2) {
        /* Factored second moment over the last two dims. */
        int64_t H = shape[ndim - 2], W = shape[ndim - 1];
        int64_t B = n / (H * W);
        double* colsum = (double*)malloc((size_t)W * sizeof(double));
        if (!colsum) {
            free(u);
            set_err(err, errlen, "out of host memory");
            return ORACLE_NOMEM;
        }
        for (int64_t b = 0; b < B; ++b) {
            const double* gb = g + b * H * W;
            double* rb = row + b * H;
            double* cb = col + b * W;
            double* ub = u + b * H * W;
            /* row_i <- beta2 row_i + (1 - beta2) mean_j (g_ij^2 + eps1) */
            for (int64_t i = 0; i < H; ++i) {
                double s = 0.0;
                for (int64_t j = 0; j < W; ++j) s += gb[i * W + j] * gb[i * W + j] + hp->eps1;
                rb[i] = beta2 * rb[i] + (1.0 - beta2) * (s / (double)W);
            }
            /* col_j <- beta2 col_j + (1 - beta2) mean_i (g_ij^2 + eps1) */
            for (int64_t j = 0; j < W; ++j) colsum[j] = 0.0;
            for (int64_t i = 0; i < H; ++i)
                for (int64_t j = 0; j < W; ++j) colsum[j] += gb[i * W + j] * gb[i * W + j] + hp->eps1;
            for (int64_t j = 0; j < W; ++j)
                cb[j] = beta2 * cb[j] + (1.0 - beta2) * (colsum[j] / (double)H);
            /* mean of the updated row vector */
            double m = 0.0;
            for (int64_t i = 0; i < H; ++i) m += rb[i];
            m /= (double)H;
            /* u_ij = g_ij * (row_i / m)^-1/2 * col_j^-1/2 */
            for (int64_t i = 0; i < H; ++i) {
                double r_fac = 1.0 / sqrt(rb[i] / m);
                for (int64_t j = 0; j < W; ++j) {
                    double c_fac = 1.0 / sqrt(cb[j]);
                    ub[i * W + j] = gb[i * W + j] * r_fac * c_fac;
                }
            }
        }
        free(colsum);
    } else {
        /* Unfactored: full exp_avg_sq. */
        for (int64_t k = 0; k < n; ++k) {
            v[k] = beta2 * v[k] + (1.0 - beta2) * (g[k] * g[k] + hp->eps1);
            u[k] = g[k] / sqrt(v[k]);
        }
    }

    /* Step 5: u <- u / max(1, RMS(u) / clip_threshold), then u <- lr * u. */
    double clip_div = rms(u, n) / hp->clip_threshold;
    if (clip_div < 1.0) clip_div = 1.0;
    for (int64_t k = 0; k < n; ++k) u[k] = (u[k] / clip_div) * alpha;
    *u_out = u;
    *alpha_out = alpha;
    return ORACLE_OK;
}

/* Decoupled weight decay, then the update u (Step 3 / the readings above). */
static void apply_update(double* p, const double* u, int64_t n, double alpha, const oracle_hparams* hp) {
    if (hp->weight_decay != 0.0) {
        for (int64_t k = 0; k < n; ++k) p[k] = p[k] - hp->weight_decay * alpha * p[k];
    }
    for (int64_t k = 0; k < n; ++k) p[k] = p[k] - u[k];
}

int oracle_adafactor_step(double* p, const double* g, int32_t ndim, const int64_t* shape,
                          double* row, double* col, double* v, double* exp_avg, int64_t t,
                          const oracle_hparams* hp, char* err, int errlen) {
    double* u = NULL;
    double alpha = 0.0;
    int64_t n = 0;
    int rc = compute_update(p, g, ndim, shape, row, col, v, t, hp, &u, &alpha, &n, err, errlen);
    if (rc != ORACLE_OK || n == 0) return rc;

    /* Step 3: with beta1, exp_avg <- beta1 exp_avg + (1 - beta1) u; u <- exp_avg. */
    if (hp->has_beta1) {
        for (int64_t k = 0; k < n; ++k) {
            exp_avg[k] = hp->beta1 * exp_avg[k] + (1.0 - hp->beta1) * u[k];
            u[k] = exp_avg[k];
        }
    }
    apply_update(p, u, n, alpha, hp);
    free(u);
    return ORACLE_OK;
}

/* Groups of the 8-bit first moment: 128 values along the last dim. */
enum { ORACLE_Q8_GROUP = 128 };

/* Rows and groups per row of the 8-bit moment of a tensor of n values. */
static void q8_layout(int32_t ndim, const int64_t* shape, int64_t n, int64_t* last, int64_t* rows,
                      int64_t* groups) {
    *last = ndim >= 2 ? shape[ndim - 1] : n;
    *rows = *last > 0 ? n / *last : 0;
    *groups = (*last + ORACLE_Q8_GROUP - 1) / ORACLE_Q8_GROUP;
}

/* Dequantised value of one stored code: code * scale in fp32. */
static double q8_dequant(int8_t code, float scale) {
    const float x = (float)code * scale;
    return (double)x;
}

/* Part 1 of the 8-bit step: the clipped, lr-scaled update u of this step
 * (second-moment state updated in place), then the new first moment
 * m = beta1 * old + (1 - beta1) * u with old the dequantised stored moment.
 * moment_out [N] receives m (float64); *alpha_out the step's lr. */
int oracle_q8_moment(const double* p, const double* g, int32_t ndim, const int64_t* shape, double* row,
                     double* col, double* v, const int8_t* codes, const float* scales, double* moment_out,
                     double* alpha_out, int64_t t, const oracle_hparams* hp, char* err, int errlen) {
    if (!hp->has_beta1) {
        set_err(err, errlen, "the 8-bit first moment needs beta1");
        return ORACLE_INVALID;
    }
    double* u = NULL;
    int64_t n = 0;
    *alpha_out = 0.0;
    int rc = compute_update(p, g, ndim, shape, row, col, v, t, hp, &u, alpha_out, &n, err, errlen);
    if (rc != ORACLE_OK || n == 0) return rc;
    int64_t last, rows, groups;
    q8_layout(ndim, shape, n, &last, &rows, &groups);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < last; ++j) {
            const int64_t e = r * last + j;
            const double old = q8_dequant(codes[e], scales[r * groups + j / ORACLE_Q8_GROUP]);
            moment_out[e] = hp->beta1 * old + (1.0 - hp->beta1) * u[e];
        }
    }
    free(u);
    return ORACLE_OK;
}

/* Part 2: the quantize_tensor listing on each group of the new moment, in
 * fp32: m rounded to fp32, amax = max |m|, scale = amax / 127, code =
 * rint(m / scale) clamped to [-128, 127]; codes 0 where the scale is 0 (an
 * all-zero group, or one whose amax / 127 underflows). */
void oracle_q8_quantize(const double* moment, int32_t ndim, const int64_t* shape, int8_t* codes,
                        float* scales) {
    int64_t n = 1;
    for (int32_t k = 0; k < ndim; ++k) n *= shape[k];
    int64_t last, rows, groups;
    q8_layout(ndim, shape, n, &last, &rows, &groups);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < groups; ++k) {
            const int64_t j0 = k * ORACLE_Q8_GROUP;
            const int64_t j1 = j0 + ORACLE_Q8_GROUP < last ? j0 + ORACLE_Q8_GROUP : last;
            float amax = 0.0f;
            for (int64_t j = j0; j < j1; ++j) {
                const float a = fabsf((float)moment[r * last + j]);
                if (a > amax) amax = a;
            }
            const float scale = amax / 127.0f;
            scales[r * groups + k] = scale;
            for (int64_t j = j0; j < j1; ++j) {
                float q = 0.0f;
                if (scale > 0.0f) {
                    const float x = (float)moment[r * last + j] / scale;
                    q = rintf(x);
                    if (q < -128.0f) q = -128.0f;
                    if (q > 127.0f) q = 127.0f;
                }
                codes[r * last + j] = (int8_t)q;
            }
        }
    }
}

/* Part 3: decoupled weight decay, then the dequantised new moment
 * code * scale as the update. */
void oracle_q8_apply(double* p, int32_t ndim, const int64_t* shape, const int8_t* codes, const float* scales,
                     double alpha, const oracle_hparams* hp) {
    int64_t n = 1;
    for (int32_t k = 0; k < ndim; ++k) n *= shape[k];
    if (n == 0) return;
    int64_t last, rows, groups;
    q8_layout(ndim, shape, n, &last, &rows, &groups);
    double* u = (double*)malloc((size_t)n * sizeof(double));
    if (!u) return;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < last; ++j)
            u[r * last + j] = q8_dequant(codes[r * last + j], scales[r * groups + j / ORACLE_Q8_GROUP]);
    apply_update(p, u, n, alpha, hp);
    free(u);
}

/* One step with the first moment held as int8 codes [N] and fp32 scales
 * [rows * ceil(last_dim / 128)] (rows = N / last_dim; last_dim = N for
 * ndim < 2).  Requires beta1.  moment_out [N] (may be NULL) receives the
 * unquantised new moment.  Other arguments as oracle_adafactor_step. */
int oracle_adafactor_step_q8(double* p, const double* g, int32_t ndim, const int64_t* shape,
                             double* row, double* col, double* v, int8_t* codes, float* scales,
                             double* moment_out, int64_t t, const oracle_hparams* hp, char* err,
                             int errlen) {
    int64_t n = 1;
    for (int32_t k = 0; k < ndim && k < 8; ++k) n *= shape[k];
    double* m = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!m) {
        set_err(err, errlen, "out of host memory");
        return ORACLE_NOMEM;
    }
    double alpha = 0.0;
    int rc = oracle_q8_moment(p, g, ndim, shape, row, col, v, codes, scales, m, &alpha, t, hp, err, errlen);
    if (rc == ORACLE_OK && n > 0) {
        oracle_q8_quantize(m, ndim, shape, codes, scales);
        oracle_q8_apply(p, ndim, shape, codes, scales, alpha, hp);
        if (moment_out) memcpy(moment_out, m, (size_t)n * sizeof(double));
    }
    free(m);
    return rc;
}
