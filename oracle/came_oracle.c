/*
 * CAME step oracle: plain, slow, float64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or run this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Sources:
 *   - the Colossal-AI distributed-optimizer article ("Colossal-AI
 *     分布式优化器全解析：Adafactor、CAME、GaLore 与 LAMB ...",
 *     blog.gitcode.com): table "四种优化器：原理速览", CAME row (Adafactor's
 *     low-rank second moment plus a confidence matrix and momentum with three
 *     betas, arXiv:2307.02047; only a light confidence state is added), and
 *     section "其余优化器的关键参数速查", DistributedCAME: defaults lr=None,
 *     eps=(1e-30, 1e-16), clip_threshold=1.0, betas=(0.9, 0.999, 0.9999),
 *     weight_decay=0.0; the three betas track the update, the squared
 *     gradient and the instability (confidence) term.
 *   - The update rule is not printed on the article.  It is the CAME
 *     algorithm of the paper the article cites (Luo et al., "CAME:
 *     Confidence-guided Adaptive Memory Efficient Optimization",
 *     arXiv:2307.02047), for a matrix g of n rows and m columns:
 *       r = b2 r + (1 - b2) mean_j(g^2 + eps1)      (row statistic)
 *       c = b2 c + (1 - b2) mean_i(g^2 + eps1)      (column statistic)
 *       v_ij = r_i c_j / mean(r)
 *       u = g / sqrt(v);  uh = u / max(1, RMS(u) / d)
 *       m = b1 m + (1 - b1) uh
 *       U = (uh - m)^2                              (instability)
 *       R = b3 R + (1 - b3) mean_j(U + eps2),  C = b3 C + (1 - b3) mean_i(U + eps2)
 *       S_ij = R_i C_j / mean(R)
 *       p = p - lr m / sqrt(S)
 *     The paper writes row and column sums with v = r c / (1^T r); with means
 *     the same v results (the factors n and m cancel).
 *
 * Readings where the sources leave a step open (each one is also listed in
 * the design notes):
 *   - a tensor with ndim < 2 is a matrix of one row: its row statistics are
 *     scalars and v, S reduce to full per-element EMAs (v = EMA of g^2 + eps1,
 *     S = EMA of U + eps2); such tensors keep those full vectors;
 *   - ndim > 2 is viewed as [B, H, W], factored over the last two dims per
 *     leading index; RMS(u) is taken over the whole tensor;
 *   - lr has no default (the article's lr=None): a learning rate must be
 *     given; lr >= 0, eps >= 0, 0 <= beta < 1, clip_threshold > 0,
 *     weight_decay >= 0, all finite;
 *   - weight decay is decoupled: p <- p - weight_decay * lr * p, applied
 *     before the update is subtracted (both from the step's starting p);
 *   - a tensor with no elements is left untouched.
 *
 * Every quantity is float64; the step count t is 1-based (it does not enter
 * the rule: the betas are constants).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

typedef struct {
    double lr;
    double eps1;            /* eps[0]: added to g*g           */
    double eps2;            /* eps[1]: added to the instability */
    double clip_threshold;  /* d */
    double beta1, beta2, beta3;
    double weight_decay;
} oracle_came_hparams;

enum { CAME_OK = 0, CAME_INVALID = 1, CAME_NOMEM = 2 };

static int came_fail(char* err, int errlen, int code, const char* msg) {
    if (err && errlen > 0) snprintf(err, (size_t)errlen, "%s", msg);
    return code;
}

int oracle_came_check_hparams(const oracle_came_hparams* hp, char* err, int errlen) {
    if (!hp) return came_fail(err, errlen, CAME_INVALID, "hparams is NULL");
    if (!isfinite(hp->lr) || hp->lr < 0.0) return came_fail(err, errlen, CAME_INVALID, "invalid learning rate");
    if (!isfinite(hp->eps1) || hp->eps1 < 0.0 || !isfinite(hp->eps2) || hp->eps2 < 0.0)
        return came_fail(err, errlen, CAME_INVALID, "invalid eps");
    if (!isfinite(hp->clip_threshold) || hp->clip_threshold <= 0.0)
        return came_fail(err, errlen, CAME_INVALID, "invalid clip_threshold");
    const double b[3] = {hp->beta1, hp->beta2, hp->beta3};
    for (int k = 0; k < 3; ++k)
        if (!isfinite(b[k]) || b[k] < 0.0 || b[k] >= 1.0)
            return came_fail(err, errlen, CAME_INVALID, "invalid beta (needs 0 <= beta < 1)");
    if (!isfinite(hp->weight_decay) || hp->weight_decay < 0.0)
        return came_fail(err, errlen, CAME_INVALID, "invalid weight_decay");
    return CAME_OK;
}

static double rms(const double* x, int64_t n) {
    double s = 0.0;
    for (int64_t k = 0; k < n; ++k) s += x[k] * x[k];
    return sqrt(s / (double)n);
}

/*
 * Factored statistic of one [H, W] slice x (x already holds the values whose
 * row and column means are tracked, eps included): rb[i], cb[j] are updated
 * as EMAs with coefficient beta, and f[i*W+j] receives the reconstruction
 * rb_i cb_j / mean(rb).
 */
static void factored_ema(const double* x, int64_t H, int64_t W, double beta, double* rb, double* cb, double* f) {
    for (int64_t i = 0; i < H; ++i) {
        double s = 0.0;
        for (int64_t j = 0; j < W; ++j) s += x[i * W + j];
        rb[i] = beta * rb[i] + (1.0 - beta) * (s / (double)W);
    }
    for (int64_t j = 0; j < W; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < H; ++i) s += x[i * W + j];
        cb[j] = beta * cb[j] + (1.0 - beta) * (s / (double)H);
    }
    double mr = 0.0;
    for (int64_t i = 0; i < H; ++i) mr += rb[i];
    mr /= (double)H;
    for (int64_t i = 0; i < H; ++i)
        for (int64_t j = 0; j < W; ++j) f[i * W + j] = rb[i] * cb[j] / mr;
}

/*
 * One CAME step on one tensor.  Factored tensors (ndim >= 2) use row/col
 * (second moment, B*H and B*W values) and res_row/res_col (instability, the
 * same sizes); others use v and res (n values each).  exp_avg has n values.
 * Arrays not used by the tensor's kind may be NULL.
 */
int oracle_came_step(double* p, const double* g, int32_t ndim, const int64_t* shape, double* row, double* col,
                     double* v, double* exp_avg, double* res_row, double* res_col, double* res, int64_t t,
                     const oracle_came_hparams* hp, char* err, int errlen) {
    int rc = oracle_came_check_hparams(hp, err, errlen);
    if (rc != CAME_OK) return rc;
    if (t < 1) return came_fail(err, errlen, CAME_INVALID, "step must be >= 1");
    if (ndim < 0 || (ndim > 0 && !shape)) return came_fail(err, errlen, CAME_INVALID, "bad shape");
    int64_t n = 1;
    for (int32_t d = 0; d < ndim; ++d) {
        if (shape[d] < 0) return came_fail(err, errlen, CAME_INVALID, "negative dim");
        n *= shape[d];
    }
    if (n == 0) return CAME_OK;
    const int factored = ndim >= 2;
    int64_t B = 1, H = 1, W = n;
    if (factored) {
        H = shape[ndim - 2];
        W = shape[ndim - 1];
        B = n / (H * W);
        if (!row || !col || !res_row || !res_col) return came_fail(err, errlen, CAME_INVALID, "missing factored state");
    } else if (!v || !res) {
        return came_fail(err, errlen, CAME_INVALID, "missing unfactored state");
    }
    if (!exp_avg) return came_fail(err, errlen, CAME_INVALID, "missing exp_avg");

    double* x = (double*)malloc(sizeof(double) * (size_t)n);   /* g^2 + eps1, then U + eps2 */
    double* f = (double*)malloc(sizeof(double) * (size_t)n);   /* v, then S */
    double* u = (double*)malloc(sizeof(double) * (size_t)n);
    if (!x || !f || !u) {
        free(x); free(f); free(u);
        return came_fail(err, errlen, CAME_NOMEM, "out of memory");
    }

    /* second moment v */
    for (int64_t k = 0; k < n; ++k) x[k] = g[k] * g[k] + hp->eps1;
    if (factored) {
        for (int64_t b = 0; b < B; ++b)
            factored_ema(x + b * H * W, H, W, hp->beta2, row + b * H, col + b * W, f + b * H * W);
    } else {
        for (int64_t k = 0; k < n; ++k) {
            v[k] = hp->beta2 * v[k] + (1.0 - hp->beta2) * x[k];
            f[k] = v[k];
        }
    }
    /* u = g / sqrt(v), clipped by RMS */
    for (int64_t k = 0; k < n; ++k) u[k] = g[k] / sqrt(f[k]);
    double clip_div = rms(u, n) / hp->clip_threshold;
    if (clip_div < 1.0) clip_div = 1.0;
    for (int64_t k = 0; k < n; ++k) u[k] = u[k] / clip_div;
    /* momentum of the clipped update, and the instability against it */
    for (int64_t k = 0; k < n; ++k) {
        exp_avg[k] = hp->beta1 * exp_avg[k] + (1.0 - hp->beta1) * u[k];
        const double dlt = u[k] - exp_avg[k];
        x[k] = dlt * dlt + hp->eps2;
    }
    /* confidence S */
    if (factored) {
        for (int64_t b = 0; b < B; ++b)
            factored_ema(x + b * H * W, H, W, hp->beta3, res_row + b * H, res_col + b * W, f + b * H * W);
    } else {
        for (int64_t k = 0; k < n; ++k) {
            res[k] = hp->beta3 * res[k] + (1.0 - hp->beta3) * x[k];
            f[k] = res[k];
        }
    }
    /* decoupled weight decay, then the confidence-scaled momentum */
    for (int64_t k = 0; k < n; ++k) {
        p[k] = p[k] - hp->weight_decay * hp->lr * p[k];
        p[k] = p[k] - hp->lr * exp_avg[k] / sqrt(f[k]);
    }
    free(x); free(f); free(u);
    return CAME_OK;
}
