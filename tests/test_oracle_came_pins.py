"""Pins of the float64 CAME oracle against what the sources and the
mathematics fix.

Sources: the Colossal-AI distributed-optimizer article (CAME row of the
overview table; "其余优化器的关键参数速查", DistributedCAME defaults and the
roles of its three betas) and the CAME algorithm of the paper it cites
(arXiv:2307.02047).  Each test checks the oracle against a closed form, an
invariant or a special case that reduces to something simpler, so that a
plausible slip (the instability taken against the old momentum, a dropped
eps2, beta3 confused with beta2, a missing mean(R) normalisation, a column
mean over the wrong axis, the clip inverted, no square root of S, weight decay
without the lr, swapped momentum coefficients) fails at least one of them.
"""
import numpy as np
import pytest

from oracle import came
from oracle.came import CameHParams, CameState


@pytest.fixture(autouse=True, scope="module")
def _built():
    came.build()


def run(p0, grads, hp, shape=None):
    p = np.array(p0, dtype=np.float64, copy=True)
    st = CameState(p.shape if shape is None else shape)
    for t, g in enumerate(grads, 1):
        came.step(p, np.asarray(g, np.float64), st, t, hp)
    return p, st


def rank1(H, W, seed):
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.5, 2.0, H) * rng.choice([-1.0, 1.0], H)
    b = rng.uniform(0.5, 2.0, W) * rng.choice([-1.0, 1.0], W)
    return np.outer(a, b) * 1e-3


def test_article_defaults_and_checks():
    hp = CameHParams(lr=1e-3)
    assert (hp.eps, hp.clip_threshold, hp.betas, hp.weight_decay) == ((1e-30, 1e-16), 1.0, (0.9, 0.999, 0.9999), 0.0)
    came.check_hparams(hp)
    with pytest.raises(came.CameOracleError, match="learning rate"):
        came.check_hparams(CameHParams())
    for bad in (dict(lr=-1.0), dict(lr=1e-3, eps=(-1.0, 0.0)), dict(lr=1e-3, clip_threshold=0.0),
                dict(lr=1e-3, betas=(0.9, 1.0, 0.9)), dict(lr=1e-3, weight_decay=-1.0)):
        with pytest.raises(came.CameOracleError):
            came.check_hparams(CameHParams(**bad))


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_rank1_gradient_with_active_clip(wd):
    """g = a b^T makes the factored second moment exact: v = (1 - b2^t) g^2,
    so RMS(u) = (1 - b2^t)^-1/2 >= 1 and the clip leaves uh = sign(g).  Then
    m_t = (1 - b1^t) sign(g), the instability U + eps2 = b1^(2t) + eps2 is the
    same everywhere, R = C = S = rho_t with rho_t = b3 rho + (1 - b3)(b1^(2t) +
    eps2), and p_t = p (1 - wd lr) - lr (1 - b1^t) sign(g) / sqrt(rho_t)."""
    H, W = 6, 11
    g = rank1(H, W, 1)
    hp = CameHParams(lr=1e-2, eps=(0.0, 1e-3), betas=(0.8, 0.99, 0.95), weight_decay=wd)
    b1, b2, b3 = hp.betas
    p0 = np.random.default_rng(2).standard_normal((H, W)) * 0.02
    p = p0.copy()
    st = CameState((H, W))
    q, rho = p0.copy(), 0.0
    for t in range(1, 7):
        came.step(p, g, st, t, hp)
        rho = b3 * rho + (1 - b3) * (b1 ** (2 * t) + hp.eps[1])
        q = q * (1 - wd * hp.lr) - hp.lr * (1 - b1 ** t) * np.sign(g) / np.sqrt(rho)
        np.testing.assert_allclose(p, q, rtol=1e-12, atol=1e-17)
        np.testing.assert_allclose(st.exp_avg.reshape(H, W), (1 - b1 ** t) * np.sign(g), rtol=1e-12)


def test_rank1_gradient_with_inactive_clip():
    """With a clip threshold above RMS(u), uh = u = sign(g) / sqrt(1 - b2^t),
    the momentum is the scalar recurrence mu_t = b1 mu + (1 - b1) / sqrt(1 -
    b2^t) times sign(g), and U = (1/sqrt(1 - b2^t) - mu_t)^2 is uniform."""
    H, W = 5, 3
    g = rank1(H, W, 3)
    hp = CameHParams(lr=3e-3, eps=(0.0, 1e-6), clip_threshold=1e3, betas=(0.9, 0.999, 0.9999))
    b1, b2, b3 = hp.betas
    p0 = np.random.default_rng(4).standard_normal((H, W)) * 0.02
    p = p0.copy()
    st = CameState((H, W))
    q, mu, rho = p0.copy(), 0.0, 0.0
    for t in range(1, 6):
        came.step(p, g, st, t, hp)
        s = 1.0 / np.sqrt(1 - b2 ** t)
        mu = b1 * mu + (1 - b1) * s
        rho = b3 * rho + (1 - b3) * ((s - mu) ** 2 + hp.eps[1])
        q = q - hp.lr * mu * np.sign(g) / np.sqrt(rho)
        np.testing.assert_allclose(p, q, rtol=1e-11, atol=1e-17)


@pytest.mark.parametrize("shape2d", [(1, 37), (37, 1)])
def test_single_row_or_column_equals_the_vector_path(shape2d):
    """A 1 x m or n x 1 matrix makes both factored statistics exact per
    element, so it must match the full per-element (vector) path."""
    n = max(shape2d)
    rng = np.random.default_rng(5)
    p0 = rng.standard_normal(n) * 0.02
    grads = [rng.standard_normal(n) * 1e-3 for _ in range(6)]
    hp = CameHParams(lr=1e-2, eps=(1e-30, 1e-16), clip_threshold=0.5, weight_decay=0.05)
    p_vec, _ = run(p0, grads, hp)
    p_mat, _ = run(p0.reshape(shape2d), [g.reshape(shape2d) for g in grads], hp)
    np.testing.assert_allclose(p_mat.reshape(-1), p_vec, rtol=1e-12, atol=1e-18)


def test_row_and_column_means_agree():
    """Both second-moment factors are EMAs of the grand mean of g^2 + eps1,
    and both instability factors of the grand mean of U + eps2."""
    rng = np.random.default_rng(6)
    H, W = 9, 14
    p = rng.standard_normal((H, W)) * 0.02
    st = CameState((H, W))
    hp = CameHParams(lr=1e-3)
    for t in range(1, 8):
        came.step(p, rng.standard_normal((H, W)) * 1e-3, st, t, hp)
        assert st.row.mean() == pytest.approx(st.col.mean(), rel=1e-12)
        assert st.res_row.mean() == pytest.approx(st.res_col.mean(), rel=1e-12)


def test_gradient_scale_invariance():
    """With eps1 = 0, uh does not change when every gradient is scaled, so
    neither does anything downstream of it."""
    rng = np.random.default_rng(7)
    p0 = rng.standard_normal((8, 12)) * 0.02
    grads = [rng.standard_normal((8, 12)) * 1e-3 for _ in range(5)]
    hp = CameHParams(lr=1e-2, eps=(0.0, 1e-16), weight_decay=0.01)
    a, _ = run(p0, grads, hp)
    b, _ = run(p0, [37.0 * g for g in grads], hp)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-18)


@pytest.mark.parametrize("shape", [(6, 7), (40,)])
def test_zero_gradient_is_pure_decay(shape):
    """g = 0 gives u = 0, so m stays 0 and p only decays by (1 - wd lr)."""
    p0 = np.random.default_rng(8).standard_normal(shape)
    p, st = run(p0, [np.zeros(shape)] * 3, CameHParams(lr=0.1, weight_decay=0.2))
    np.testing.assert_allclose(p, p0 * (1 - 0.02) ** 3, rtol=1e-14)
    assert not st.exp_avg.any()


def test_clip_bounds_the_first_momentum():
    """m_1 = (1 - b1) uh and RMS(uh) = min(RMS(u), d): with a small threshold
    the clip is active and RMS(m_1) / (1 - b1) equals d."""
    rng = np.random.default_rng(9)
    hp = CameHParams(lr=1e-3, clip_threshold=0.3)
    _, st = run(rng.standard_normal((10, 20)), [rng.standard_normal((10, 20))], hp)
    assert np.sqrt(np.mean(st.exp_avg ** 2)) / (1 - hp.betas[0]) == pytest.approx(0.3, rel=1e-12)


def test_leading_dims_factor_per_slice():
    """[2, H, W] with an inactive clip equals the two [H, W] slices run alone."""
    rng = np.random.default_rng(10)
    H, W = 4, 6
    p0 = rng.standard_normal((2, H, W)) * 0.02
    grads = [rng.standard_normal((2, H, W)) * 1e-3 for _ in range(4)]
    hp = CameHParams(lr=1e-2, clip_threshold=1e6)
    p3, _ = run(p0, grads, hp)
    for b in range(2):
        pb, _ = run(p0[b], [g[b] for g in grads], hp)
        np.testing.assert_allclose(p3[b], pb, rtol=1e-13, atol=1e-18)


def test_empty_tensor_untouched():
    p = np.zeros((0, 5))
    came.step(p, np.zeros((0, 5)), CameState((0, 5)), 1, CameHParams(lr=1e-3))
