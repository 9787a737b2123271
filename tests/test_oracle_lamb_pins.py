"""Pins of the float64 LAMB oracle against what the sources and the
mathematics fix.

Sources: the Colossal-AI distributed-optimizer article (LAMB row of the
overview table; "其余优化器的关键参数速查", DistributedLAMB defaults and the
per-layer trust ratio) and the LAMB algorithm of the paper it cites
(arXiv:1904.00962).  Each test checks the oracle against a closed form, an
invariant, or a special case that reduces to a library routine (torch's Adam),
so that a plausible slip (a bias correction with the wrong power, a swapped
EMA, a missing square root, an inverted trust ratio, weight decay left out of
the direction, the lr dropped) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import lamb
from oracle.lamb import LambHParams, LambState


@pytest.fixture(autouse=True, scope="module")
def _built():
    lamb.build()


def _rng(seed):
    return np.random.default_rng(seed)


def test_article_defaults():
    hp = LambHParams()
    assert (hp.lr, hp.betas, hp.eps, hp.weight_decay, hp.bias_correction) == (1e-3, (0.9, 0.999), 1e-6, 0.0, True)
    lamb.check_hparams(hp)


@pytest.mark.parametrize("bad", [dict(lr=-1e-3), dict(eps=-1.0), dict(betas=(1.0, 0.999)), dict(betas=(0.9, -0.1)),
                                 dict(weight_decay=-0.1), dict(lr=float("nan"))])
def test_invalid_hparams_rejected(bad):
    with pytest.raises(lamb.LambOracleError):
        lamb.check_hparams(LambHParams(**bad))


@pytest.mark.parametrize("wd", [0.0, 0.3])
def test_first_step_from_zero_params_is_adam(wd):
    """||p|| = 0 gives a trust ratio of 1 and the weight-decay term vanishes,
    so the first step is exactly torch's Adam step (same bias correction and
    eps placement)."""
    g = _rng(1).standard_normal((37, 19)) * 1e-2
    hp = LambHParams(lr=3e-3, betas=(0.8, 0.95), eps=1e-5, weight_decay=wd)
    p = np.zeros_like(g)
    st = LambState(g.shape)
    trust = lamb.step(p, g, st, 1, hp)
    assert trust == 1.0
    tp = torch.zeros(g.shape, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.Adam([tp], lr=hp.lr, betas=hp.betas, eps=hp.eps)
    tp.grad = torch.from_numpy(g.copy())
    opt.step()
    np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-13, atol=1e-18)


@pytest.mark.parametrize("betas", [(0.9, 0.999), (0.5, 0.3), (0.0, 0.0)])
@pytest.mark.parametrize("wd", [0.0, 0.05])
def test_first_step_closed_form(betas, wd):
    """With bias correction the first step has mh = g and vh = g^2 whatever
    the betas, so r = g / (|g| + eps) + wd p."""
    rng = _rng(2)
    g = rng.standard_normal(500) * 1e-3
    p0 = rng.standard_normal(500) * 0.02
    hp = LambHParams(lr=1e-2, betas=betas, eps=1e-6, weight_decay=wd)
    p = p0.copy()
    trust = lamb.step(p, g, LambState(g.shape), 1, hp)
    r = g / (np.abs(g) + hp.eps) + wd * p0
    tr = np.linalg.norm(p0) / np.linalg.norm(r)
    assert trust == pytest.approx(tr, rel=1e-13)
    np.testing.assert_allclose(p, p0 - hp.lr * tr * r, rtol=1e-12, atol=1e-17)


def test_constant_gradient_with_bias_correction():
    """A constant gradient keeps mh = g and vh = g^2 at every step (the bias
    corrections undo 1 - beta^t exactly), so with wd = 0 the direction is the
    fixed s = g / (|g| + eps) and p follows p <- p - lr ||p|| s / ||s||."""
    rng = _rng(3)
    g = rng.standard_normal(300) * 1e-3
    p0 = rng.standard_normal(300) * 0.02
    hp = LambHParams(lr=0.05, betas=(0.9, 0.99), eps=1e-7)
    p = p0.copy()
    st = LambState(g.shape)
    s = g / (np.abs(g) + hp.eps)
    q = p0.copy()
    for t in range(1, 9):
        lamb.step(p, g, st, t, hp)
        q = q - hp.lr * np.linalg.norm(q) * s / np.linalg.norm(s)
        np.testing.assert_allclose(p, q, rtol=1e-11, atol=1e-16)


def test_constant_gradient_without_bias_correction():
    """Without bias correction and with a constant gradient, m_t = (1 - b1^t) g
    and v_t = (1 - b2^t) g^2, so r_t = (1 - b1^t) g / (sqrt(1 - b2^t) |g| + eps)."""
    rng = _rng(4)
    g = rng.standard_normal(200) * 1e-2
    p0 = rng.standard_normal(200) * 0.02
    hp = LambHParams(lr=0.02, betas=(0.7, 0.9), eps=1e-4, weight_decay=0.0, bias_correction=False)
    p = p0.copy()
    st = LambState(g.shape)
    q = p0.copy()
    for t in range(1, 7):
        trust = lamb.step(p, g, st, t, hp)
        r = (1 - hp.betas[0] ** t) * g / (math.sqrt(1 - hp.betas[1] ** t) * np.abs(g) + hp.eps)
        tr = np.linalg.norm(q) / np.linalg.norm(r)
        assert trust == pytest.approx(tr, rel=1e-12)
        q = q - hp.lr * tr * r
        np.testing.assert_allclose(p, q, rtol=1e-11, atol=1e-16)


def test_update_norm_is_lr_times_param_norm():
    """Whenever both norms are non-zero, ||p_new - p|| = lr * ||p|| exactly
    (the trust ratio rescales the direction to the parameter's norm)."""
    rng = _rng(5)
    hp = LambHParams(lr=7e-3, betas=(0.9, 0.999), eps=1e-6, weight_decay=0.01)
    p = rng.standard_normal((64, 33)) * 0.02
    st = LambState(p.shape)
    for t in range(1, 11):
        g = rng.standard_normal(p.shape) * 1e-3 * (1 + t)
        before = p.copy()
        lamb.step(p, g, st, t, hp)
        assert np.linalg.norm(p - before) == pytest.approx(hp.lr * np.linalg.norm(before), rel=1e-12)


def test_zero_gradient_is_pure_decay():
    """g = 0 leaves m = v = 0, so r = wd p, the trust ratio is 1 / wd and the
    step is p <- (1 - lr) p; with wd = 0 as well, r = 0 and p is unchanged."""
    rng = _rng(6)
    p0 = rng.standard_normal(100)
    g = np.zeros(100)
    p = p0.copy()
    trust = lamb.step(p, g, LambState(p.shape), 1, LambHParams(lr=0.1, weight_decay=0.25))
    assert trust == pytest.approx(4.0, rel=1e-14)
    np.testing.assert_allclose(p, 0.9 * p0, rtol=1e-14)
    p = p0.copy()
    trust = lamb.step(p, g, LambState(p.shape), 1, LambHParams(lr=0.1))
    assert trust == 1.0
    np.testing.assert_array_equal(p, p0)


def test_gradient_scale_invariance():
    """With eps = 0, r = mh / sqrt(vh) does not change when every gradient is
    scaled by the same factor."""
    rng = _rng(7)
    p0 = rng.standard_normal(120) * 0.02
    grads = [rng.standard_normal(120) * 1e-3 for _ in range(4)]
    hp = LambHParams(lr=1e-2, eps=0.0, weight_decay=0.02)
    out = []
    for c in (1.0, 37.0):
        p = p0.copy()
        st = LambState(p.shape)
        for t, g in enumerate(grads, 1):
            lamb.step(p, c * g, st, t, hp)
        out.append(p)
    np.testing.assert_allclose(out[0], out[1], rtol=1e-12, atol=1e-17)


def test_empty_tensor_untouched():
    p = np.zeros(0)
    assert lamb.step(p, np.zeros(0), LambState((0,)), 1, LambHParams()) == 1.0
