"""Brute-force check of the oracle on tiny shapes at 50 significant digits.

The brute force is written in a different form from the oracle: it keeps the
factored statistics as running row and column *sums* R and C and rebuilds the
full second-moment estimate V_hat = R C^T / sum(R) (the rank-one
reconstruction in the Adafactor paper cited by the article's optimizer table),
then divides g by sqrt(V_hat) element by element.  The oracle keeps means and
uses the normalised factors (row_i / mean(row))^-1/2 col_j^-1/2.  The two agree
in exact arithmetic; a slip in either shows up as a mismatch far above 1e-13.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import HParams, State

mpmath = pytest.importorskip("mpmath")
mp = mpmath.mp


def brute_run(p0, grads, hp):
    mp.dps = 50
    shape = p0.shape
    n = int(np.prod(shape)) if shape else 1
    P = [mp.mpf(float(x)) for x in p0.reshape(-1)]
    e1, e2, d = mp.mpf(hp.eps[0]), mp.mpf(hp.eps[1]), mp.mpf(hp.clip_threshold)
    factored = len(shape) >= 2
    if factored:
        H, W = shape[-2], shape[-1]
        B = n // (H * W)
        R = [[mp.mpf(0)] * H for _ in range(B)]
        C = [[mp.mpf(0)] * W for _ in range(B)]
    else:
        V = [mp.mpf(0)] * n
    M = [mp.mpf(0)] * n
    for k, g in enumerate(grads):
        t = k + 1
        G = [mp.mpf(float(x)) for x in np.asarray(g, np.float64).reshape(-1)]
        if hp.relative_step:
            cap = mp.mpf("1e-6") * t if hp.warmup_init else mp.mpf("1e-2")
            rho = min(cap, 1 / mp.sqrt(t))
        else:
            rho = mp.mpf(hp.lr)
        rms_p = mp.sqrt(sum(x * x for x in P) / n)
        alpha = rho * max(e2, rms_p) if hp.scale_parameter else rho
        b2 = 1 - mp.power(t, mp.mpf(hp.decay_rate))
        U = [mp.mpf(0)] * n
        if factored:
            for b in range(B):
                base = b * H * W
                for i in range(H):
                    rs = sum(G[base + i * W + j] ** 2 + e1 for j in range(W))
                    R[b][i] = b2 * R[b][i] + (1 - b2) * rs
                for j in range(W):
                    cs = sum(G[base + i * W + j] ** 2 + e1 for i in range(H))
                    C[b][j] = b2 * C[b][j] + (1 - b2) * cs
                tot = sum(R[b])
                for i in range(H):
                    for j in range(W):
                        vhat = R[b][i] * C[b][j] / tot
                        U[base + i * W + j] = G[base + i * W + j] / mp.sqrt(vhat)
        else:
            for e in range(n):
                V[e] = b2 * V[e] + (1 - b2) * (G[e] ** 2 + e1)
                U[e] = G[e] / mp.sqrt(V[e])
        rms_u = mp.sqrt(sum(x * x for x in U) / n)
        div = max(mp.mpf(1), rms_u / d)
        U = [alpha * x / div for x in U]
        if hp.beta1 is not None:
            b1 = mp.mpf(hp.beta1)
            M = [b1 * m + (1 - b1) * u for m, u in zip(M, U)]
            U = list(M)
        if hp.weight_decay:
            wd = mp.mpf(hp.weight_decay)
            P = [x - wd * alpha * x for x in P]
        P = [x - u for x, u in zip(P, U)]
    out = {"p": np.array([float(x) for x in P])}
    if factored:
        out["row"] = np.array([float(x) / W for r in R for x in r])
        out["col"] = np.array([float(x) / H for c in C for x in c])
    else:
        out["v"] = np.array([float(x) for x in V])
    if hp.beta1 is not None:
        out["exp_avg"] = np.array([float(x) for x in M])
    return out


SHAPES = [(1, 1), (2, 3), (3, 2), (1, 5), (5, 1), (2, 2, 3), (4,)]
FLAGS = [
    dict(),
    dict(beta1=0.9),
    dict(weight_decay=0.1, beta1=0.5),
    dict(clip_threshold=0.3),
    dict(warmup_init=True),
    dict(scale_parameter=False, eps=(1e-3, 1e-2)),
    dict(lr=0.02, relative_step=False, scale_parameter=False, beta1=0.8, weight_decay=0.05),
    dict(lr=0.02, relative_step=False, decay_rate=-0.5),
]


@pytest.mark.parametrize("shape,flags", list(itertools.product(SHAPES, FLAGS)))
def test_oracle_matches_brute_force(shape, flags):
    hp = HParams(**flags)
    rng = np.random.default_rng(hash((shape, tuple(sorted(flags)))) % (2 ** 32))
    p0 = rng.normal(0, 0.5, size=shape)
    grads = [rng.standard_t(3, size=shape) for _ in range(10)]
    if len(shape) >= 2 and shape[-2] > 1:
        for g in grads[3:6]:
            g[..., 0, :] = 0.0  # a zero row for a few steps
    ref = brute_run(p0, grads, hp)
    p = p0.astype(np.float64).copy()
    st = State(shape, beta1=hp.beta1 is not None)
    for t, g in enumerate(grads, start=1):
        oracle.step(p, g, st, t, hp)
    np.testing.assert_allclose(p.reshape(-1), ref["p"], rtol=1e-13, atol=1e-15)
    if "row" in ref:
        np.testing.assert_allclose(st.row, ref["row"], rtol=1e-13)
        np.testing.assert_allclose(st.col, ref["col"], rtol=1e-13)
    else:
        np.testing.assert_allclose(st.v, ref["v"], rtol=1e-13)
    if "exp_avg" in ref:
        np.testing.assert_allclose(st.exp_avg, ref["exp_avg"], rtol=1e-12, atol=1e-16)
