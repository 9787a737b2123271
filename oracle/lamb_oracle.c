/*
 * LAMB step oracle: plain, slow, float64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or run this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Sources:
 *   - the Colossal-AI distributed-optimizer article ("Colossal-AI
 *     分布式优化器全解析：Adafactor、CAME、GaLore 与 LAMB ...",
 *     blog.gitcode.com): table "四种优化器：原理速览", LAMB row (a layer-wise
 *     adaptive update for very large batches, arXiv:1904.00962), and section
 *     "其余优化器的关键参数速查", DistributedLAMB: defaults lr=1e-3,
 *     betas=(0.9, 0.999), eps=1e-6, weight_decay=0, bias_correction=True; the
 *     constructor checks lr, eps and betas; the core is a per-layer trust
 *     ratio between the norm of the update and the norm of the parameter.
 *   - The update rule itself is not printed on the article.  It is taken from
 *     the paper the article cites (You et al., "Large Batch Optimization for
 *     Deep Learning: Training BERT in 76 minutes", arXiv:1904.00962, the LAMB
 *     algorithm), read as follows:
 *       m = beta1 m + (1 - beta1) g
 *       v = beta2 v + (1 - beta2) g^2
 *       with bias correction: mh = m / (1 - beta1^t), vh = v / (1 - beta2^t);
 *       without: mh = m, vh = v
 *       r = mh / (sqrt(vh) + eps) + weight_decay * p
 *       trust = ||p|| / ||r||   (per layer)
 *       p = p - lr * trust * r
 *
 * Readings where the sources leave a step open (each one is also listed in
 * the design notes):
 *   - a "layer" is one tensor of the list; both norms are Euclidean norms
 *     over the whole tensor;
 *   - the scaling function of the trust ratio is the identity (no clamp);
 *   - where ||p|| = 0 or ||r|| = 0 the trust ratio is 1;
 *   - ||p|| and the weight-decay term use the parameter as it is at the start
 *     of the step;
 *   - the hyper-parameter checks: lr >= 0, eps >= 0, 0 <= beta < 1,
 *     weight_decay >= 0, all finite;
 *   - a tensor with no elements is left untouched.
 *
 * Every quantity is float64; the step count t is 1-based.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>

typedef struct {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    int32_t bias_correction;
} oracle_lamb_hparams;

enum { LAMB_OK = 0, LAMB_INVALID = 1 };

static int lamb_fail(char* err, int errlen, const char* msg) {
    if (err && errlen > 0) snprintf(err, (size_t)errlen, "%s", msg);
    return LAMB_INVALID;
}

int oracle_lamb_check_hparams(const oracle_lamb_hparams* hp, char* err, int errlen) {
    if (!hp) return lamb_fail(err, errlen, "hparams is NULL");
    if (!isfinite(hp->lr) || hp->lr < 0.0) return lamb_fail(err, errlen, "invalid learning rate");
    if (!isfinite(hp->eps) || hp->eps < 0.0) return lamb_fail(err, errlen, "invalid epsilon value");
    if (!isfinite(hp->beta1) || hp->beta1 < 0.0 || hp->beta1 >= 1.0)
        return lamb_fail(err, errlen, "invalid beta parameter at index 0");
    if (!isfinite(hp->beta2) || hp->beta2 < 0.0 || hp->beta2 >= 1.0)
        return lamb_fail(err, errlen, "invalid beta parameter at index 1");
    if (!isfinite(hp->weight_decay) || hp->weight_decay < 0.0)
        return lamb_fail(err, errlen, "invalid weight_decay value");
    return LAMB_OK;
}

/* The direction r of one element, from the updated moments and the old p. */
static double lamb_direction(double m, double v, double p, double bc1, double bc2, const oracle_lamb_hparams* hp) {
    const double mh = m / bc1;
    const double vh = v / bc2;
    return mh / (sqrt(vh) + hp->eps) + hp->weight_decay * p;
}

/*
 * One LAMB step on one tensor of n values.  p, m, v are updated in place;
 * trust_out (may be NULL) receives the trust ratio used.  The loops follow
 * the algorithm's order: moments, direction and both norms, trust ratio,
 * update.
 */
int oracle_lamb_step(double* p, const double* g, int64_t n, double* m, double* v, int64_t t,
                     const oracle_lamb_hparams* hp, double* trust_out, char* err, int errlen) {
    int rc = oracle_lamb_check_hparams(hp, err, errlen);
    if (rc != LAMB_OK) return rc;
    if (t < 1) return lamb_fail(err, errlen, "step must be >= 1");
    if (n < 0) return lamb_fail(err, errlen, "negative size");
    if (n == 0) {
        if (trust_out) *trust_out = 1.0;
        return LAMB_OK;
    }
    const double bc1 = hp->bias_correction ? 1.0 - pow(hp->beta1, (double)t) : 1.0;
    const double bc2 = hp->bias_correction ? 1.0 - pow(hp->beta2, (double)t) : 1.0;

    double psq = 0.0, rsq = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        m[i] = hp->beta1 * m[i] + (1.0 - hp->beta1) * g[i];
        v[i] = hp->beta2 * v[i] + (1.0 - hp->beta2) * g[i] * g[i];
        const double r = lamb_direction(m[i], v[i], p[i], bc1, bc2, hp);
        psq += p[i] * p[i];
        rsq += r * r;
    }
    const double pn = sqrt(psq), rn = sqrt(rsq);
    const double trust = (pn > 0.0 && rn > 0.0) ? pn / rn : 1.0;
    for (int64_t i = 0; i < n; ++i) {
        const double r = lamb_direction(m[i], v[i], p[i], bc1, bc2, hp);
        p[i] = p[i] - hp->lr * trust * r;
    }
    if (trust_out) *trust_out = trust;
    return LAMB_OK;
}
