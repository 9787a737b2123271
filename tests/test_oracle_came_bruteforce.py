"""Brute-force check of the CAME oracle on tiny shapes at 40 significant digits.

The brute force follows the CAME paper's own notation (arXiv:2307.02047,
the CAME algorithm), which differs from the oracle's: the factored statistics
are running row and column *sums* (r_t = b2 r + (1-b2)(g^2 + eps1) 1_m), and
the full matrices V = r c^T / (1^T r) and S = R C^T / (1^T R) are rebuilt
before use.  The oracle keeps means and forms r_i c_j / mean(r).  A vector is
handled here as a 1 x m matrix through the same factored code, while the
oracle keeps full per-element EMAs for it.  All of these agree in exact
arithmetic; a slip in either shows up far above the 1e-12 bar.
"""
import itertools

import numpy as np
import pytest

from oracle import came
from oracle.came import CameHParams, CameState

mpmath = pytest.importorskip("mpmath")
mp = mpmath.mp


def brute_run(p0, grads, hp):
    mp.dps = 40
    shape = p0.shape
    n = int(np.prod(shape)) if shape else 1
    if len(shape) >= 2:
        H, W = shape[-2], shape[-1]
    else:
        H, W = 1, n  # one row
    B = n // (H * W)
    e1, e2 = mp.mpf(hp.eps[0]), mp.mpf(hp.eps[1])
    d = mp.mpf(hp.clip_threshold)
    b1, b2, b3 = (mp.mpf(x) for x in hp.betas)
    lr, wd = mp.mpf(hp.lr), mp.mpf(hp.weight_decay)
    P = [mp.mpf(float(x)) for x in p0.reshape(-1)]
    M = [mp.mpf(0)] * n
    r = [[mp.mpf(0)] * H for _ in range(B)]
    c = [[mp.mpf(0)] * W for _ in range(B)]
    Rr = [[mp.mpf(0)] * H for _ in range(B)]
    Cc = [[mp.mpf(0)] * W for _ in range(B)]

    def factored(X, beta, rows, cols, b):
        # sums along rows / columns of slice b, EMAs, and the rebuilt matrix
        base = b * H * W
        for i in range(H):
            rows[b][i] = beta * rows[b][i] + (1 - beta) * sum(X[base + i * W + j] for j in range(W))
        for j in range(W):
            cols[b][j] = beta * cols[b][j] + (1 - beta) * sum(X[base + i * W + j] for i in range(H))
        tot = sum(rows[b])
        return {(i, j): rows[b][i] * cols[b][j] / tot for i in range(H) for j in range(W)}

    for g in grads:
        G = [mp.mpf(float(x)) for x in np.asarray(g, np.float64).reshape(-1)]
        X = [x * x + e1 for x in G]
        U = [mp.mpf(0)] * n
        for b in range(B):
            V = factored(X, b2, r, c, b)
            for (i, j), v in V.items():
                k = b * H * W + i * W + j
                U[k] = G[k] / mp.sqrt(v)
        rms = mp.sqrt(sum(u * u for u in U) / n)
        div = max(mp.mpf(1), rms / d)
        Uh = [u / div for u in U]
        Inst = [mp.mpf(0)] * n
        for k in range(n):
            M[k] = b1 * M[k] + (1 - b1) * Uh[k]
            Inst[k] = (Uh[k] - M[k]) ** 2 + e2
        for b in range(B):
            S = factored(Inst, b3, Rr, Cc, b)
            for (i, j), s in S.items():
                k = b * H * W + i * W + j
                P[k] = P[k] - wd * lr * P[k] - lr * M[k] / mp.sqrt(s)
    return np.array([float(x) for x in P]).reshape(shape), np.array([float(x) for x in M])


SHAPES = [(2, 3), (3, 2), (4,), (1, 5), (2, 2, 3), (5, 1)]
FLAGS = [
    dict(lr=1e-2),
    dict(lr=3e-3, clip_threshold=0.1, weight_decay=0.05),
    dict(lr=1e-3, betas=(0.5, 0.8, 0.7), eps=(1e-6, 1e-4)),
    dict(lr=2e-2, clip_threshold=50.0),
]


CASES = list(itertools.product(range(len(SHAPES)), range(len(FLAGS))))


@pytest.mark.parametrize("si,fi", CASES)
def test_oracle_matches_brute_force(si, fi):
    shape, flags = SHAPES[si], FLAGS[fi]
    came.build()
    rng = np.random.default_rng(1000 * si + fi)
    p0 = rng.standard_normal(shape) * 0.1
    # Student-t gradients with one exactly zero entry
    grads = [rng.standard_t(3, size=shape) * 1e-2 for _ in range(5)]
    for g in grads:
        g.reshape(-1)[0] = 0.0
    hp = CameHParams(**flags)
    p = p0.copy()
    st = CameState(shape)
    for t, g in enumerate(grads, 1):
        came.step(p, g, st, t, hp)
    pb, mb = brute_run(p0, grads, hp)
    np.testing.assert_allclose(p, pb, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(st.exp_avg, mb, rtol=1e-10, atol=1e-14)
