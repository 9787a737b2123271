"""Pins of the float64 oracle against what the article and the mathematics fix.

Each test checks the oracle against a closed form, an invariant or a special
case that reduces to something simpler, chosen so that a plausible slip in the
oracle (a dropped eps, a swapped row/col axis, a wrong beta2 exponent, a
missing mean normalisation, the clip applied after the lr, ...) fails at least
one of them.  Article passages: the Colossal-AI distributed-optimizer article,
"Step 3" (defaults, relative step, beta1, factored vs. full second moment),
"Step 4" (_rms) and "Step 5" (beta2t, RMS clip, lr scaling).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import HParams, State

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TWO_POW_M08 = 0.5743491774985175  # 2^-0.8 to 16 digits (exp(-0.8 ln 2))


def run(p0, grads, hp, beta1_state=None, t0=1):
    """Run the oracle over a list of gradients; returns (p, state)."""
    p = np.array(p0, dtype=np.float64, copy=True)
    st = State(p.shape, beta1=hp.beta1 is not None)
    for k, g in enumerate(grads):
        oracle.step(p, np.asarray(g, np.float64), st, t0 + k, hp)
    return p, st


def rms(x):
    x = np.asarray(x, np.float64)
    return float(np.sqrt(np.mean(x * x)))


@pytest.fixture(autouse=True, scope="module")
def _built():
    oracle.build()


def test_defaults_match_article():
    """The defaults printed in Step 3 (golden fixture with its citation)."""
    with open(os.path.join(GOLDEN, "adafactor_defaults.json")) as f:
        gold = json.load(f)["defaults"]
    hp = HParams()
    assert hp.lr is gold["lr"] is None
    assert list(hp.eps) == gold["eps"]
    assert hp.clip_threshold == gold["clip_threshold"]
    assert hp.decay_rate == gold["decay_rate"]
    assert hp.beta1 is gold["beta1"] is None
    assert hp.weight_decay == gold["weight_decay"]
    assert hp.scale_parameter is gold["scale_parameter"] is True
    assert hp.relative_step is gold["relative_step"] is True
    assert hp.warmup_init is gold["warmup_init"] is False


def test_step1_discards_initial_state_and_takes_means():
    """beta2_1 = 1 - 1^-0.8 = 0: after step 1 the row/col vectors are exactly the
    row/col means of g^2 + eps1, whatever the state held before."""
    rng = np.random.default_rng(1)
    g = rng.normal(size=(5, 7))
    hp = HParams(eps=(0.3, 1e-3))
    p = rng.normal(size=(5, 7))
    st = State((5, 7), beta1=False)
    st.row[:] = rng.uniform(1, 9, size=5)
    st.col[:] = rng.uniform(1, 9, size=7)
    oracle.step(p, g, st, 1, hp)
    q = g * g + 0.3
    np.testing.assert_allclose(st.row, q.mean(axis=1), rtol=1e-14)
    np.testing.assert_allclose(st.col, q.mean(axis=0), rtol=1e-14)


def test_beta2_second_step_closed_form():
    """g = 1 then g = 2 everywhere, eps1 = 0: row_2 = col_2 = 4 - 3 beta2_2 with
    beta2_2 = 1 - 2^-0.8, i.e. 1 + 3 * 2^-0.8."""
    hp = HParams(eps=(0.0, 1e-3))
    _, st = run(np.full((3, 4), 0.1), [np.ones((3, 4)), 2 * np.ones((3, 4))], hp)
    expect = 1.0 + 3.0 * TWO_POW_M08
    np.testing.assert_allclose(st.row, expect, rtol=1e-15)
    np.testing.assert_allclose(st.col, expect, rtol=1e-15)
    # a different decay rate: beta2_2 = 1 - 2^-0.5
    hp = HParams(eps=(0.0, 1e-3), decay_rate=-0.5)
    _, st = run(np.full((3, 4), 0.1), [np.ones((3, 4)), 2 * np.ones((3, 4))], hp)
    np.testing.assert_allclose(st.row, 1.0 + 3.0 / math.sqrt(2.0), rtol=1e-15)


def rank1(h, w, seed):
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.2, 2.0, h) * rng.choice([-1, 1], h)
    b = rng.uniform(0.2, 2.0, w) * rng.choice([-1, 1], w)
    return np.outer(a, b)


def test_rank1_gradient_gives_sign_update_every_step():
    """g = a (x) b makes g^2 rank one, so the factored estimate is exact:
    row_i col_j / mean(row) = g_ij^2, u = sign(g), RMS(u) = 1 (no clip) and
    p_t = p_{t-1} - 1e-2 * max(1e-3, RMS(p_{t-1})) * sign(g)."""
    g = rank1(6, 9, 2)
    p0 = np.random.default_rng(3).normal(0, 0.02, size=(6, 9))
    hp = HParams()
    p = p0.copy()
    st = State(p.shape, beta1=False)
    expect = p0.copy()
    for t in range(1, 6):
        oracle.step(p, g, st, t, hp)
        expect = expect - 1e-2 * max(1e-3, rms(expect)) * np.sign(g)
        np.testing.assert_allclose(p, expect, rtol=1e-12, atol=1e-17)


def test_rank1_states_closed_form():
    """For g = a (x) b at step 1: row_i = a_i^2 mean(b^2) + eps1 and
    col_j = b_j^2 mean(a^2) + eps1 (axes must not be swapped, H != W)."""
    rng = np.random.default_rng(4)
    a, b = rng.uniform(0.5, 2, 4), rng.uniform(0.5, 2, 11)
    hp = HParams(eps=(0.125, 1e-3))
    _, st = run(np.zeros((4, 11)), [np.outer(a, b)], hp)
    np.testing.assert_allclose(st.row, a * a * np.mean(b * b) + 0.125, rtol=1e-14)
    np.testing.assert_allclose(st.col, b * b * np.mean(a * a) + 0.125, rtol=1e-14)


def test_marginal_means_agree():
    """mean_i row_i = mean_j col_j at every step: both are EMAs of the grand mean
    of g^2 + eps1 with the same beta2."""
    rng = np.random.default_rng(5)
    hp = HParams()
    p = rng.normal(0, 0.02, size=(7, 13))
    st = State(p.shape, beta1=False)
    for t in range(1, 11):
        oracle.step(p, rng.standard_t(3, size=(7, 13)) * 1e-3, st, t, hp)
        assert abs(st.row.mean() - st.col.mean()) <= 1e-13 * st.row.mean()


@pytest.mark.parametrize("shape2d", [(1, 7), (7, 1)])
def test_single_row_or_column_equals_unfactored(shape2d):
    """H = 1 or W = 1: the factored estimate equals the full second moment in
    exact arithmetic, so the factored and 1D paths must agree."""
    rng = np.random.default_rng(6)
    hp = HParams(beta1=0.9, weight_decay=0.1)
    p2 = rng.normal(0, 0.02, size=shape2d)
    p1 = p2.reshape(-1).copy()
    s2, s1 = State(shape2d, beta1=True), State((7,), beta1=True)
    for t in range(1, 11):
        g = rng.normal(0, 1e-2, size=7)
        oracle.step(p2, g.reshape(shape2d), s2, t, hp)
        oracle.step(p1, g, s1, t, hp)
    np.testing.assert_allclose(p2.reshape(-1), p1, rtol=1e-12)
    np.testing.assert_allclose(s2.exp_avg, s1.exp_avg, rtol=1e-10, atol=1e-20)
    if shape2d[0] == 1:
        np.testing.assert_allclose(s2.col, s1.v, rtol=1e-12)
    else:
        np.testing.assert_allclose(s2.row, s1.v, rtol=1e-12)


def test_unfactored_first_step():
    """1D, step 1: V = g^2 + eps1, u = g / sqrt(g^2 + eps1) has |u| < 1 so no
    clip, and p_1 = p_0 - 1e-2 * max(1e-3, RMS(p_0)) * u."""
    rng = np.random.default_rng(7)
    g = rng.normal(size=9)
    p0 = rng.normal(0, 0.5, size=9)
    hp = HParams(eps=(0.5, 1e-3))
    p, st = run(p0, [g], hp)
    np.testing.assert_allclose(st.v, g * g + 0.5, rtol=1e-15)
    np.testing.assert_allclose(p, p0 - 1e-2 * rms(p0) * g / np.sqrt(g * g + 0.5), rtol=1e-13)


def test_scalar_tensor_takes_unfactored_path():
    p, st = run(np.array(0.3), [np.array(2.0)], HParams(eps=(0.0, 1e-3)))
    assert st.row is None and st.v.shape == (1,)
    np.testing.assert_allclose(p, 0.3 - 1e-2 * 0.3 * 1.0, rtol=1e-15)


def test_clip_closed_form():
    """Rank-1 g gives u = sign(g) with RMS 1; clip_threshold 0.25 divides it by 4."""
    g = rank1(5, 8, 8)
    p0 = np.random.default_rng(9).normal(0, 0.02, size=(5, 8))
    p, _ = run(p0, [g], HParams(clip_threshold=0.25))
    np.testing.assert_allclose(p, p0 - 1e-2 * rms(p0) * 0.25 * np.sign(g), rtol=1e-12)


@pytest.mark.parametrize("d", [1.0, 0.5, 3.0])
def test_clip_bounds_update_rms(d):
    """RMS(p_{t-1} - p_t) <= lr_t * clip_threshold when beta1 is off and there is
    no weight decay, with equality whenever the clip is active."""
    rng = np.random.default_rng(10)
    hp = HParams(clip_threshold=d)
    p = rng.normal(0, 0.02, size=(16, 24))
    st = State(p.shape, beta1=False)
    for t in range(1, 11):
        prev = p.copy()
        alpha = 1e-2 * max(1e-3, rms(prev))
        g = rng.standard_t(3, size=p.shape)
        g[rng.integers(0, 16)] = 0.0
        oracle.step(p, g, st, t, hp)
        assert rms(prev - p) <= alpha * d * (1 + 1e-12)


def test_gradient_scale_invariance():
    """u depends on g only through g / sqrt(E[g^2]): scaling g by c > 0 changes
    nothing (up to eps1 = 1e-30)."""
    rng = np.random.default_rng(11)
    grads = [rng.normal(size=(6, 5)) for _ in range(6)]
    p0 = rng.normal(0, 0.02, size=(6, 5))
    pa, _ = run(p0, grads, HParams())
    pb, _ = run(p0, [7.5 * g for g in grads], HParams())
    np.testing.assert_allclose(pa, pb, rtol=1e-13)


def test_zero_gradient_and_decay_closed_form():
    """A rank-1 step fills exp_avg with (1 - beta1) lr sign(g); then zero
    gradients give u = 0 (no NaN: col = eps1), so exp_avg_t = beta1 exp_avg_{t-1}
    and p_t = p_{t-1} (1 - wd lr) - exp_avg_t."""
    lr, b1, wd = 0.05, 0.9, 0.01
    hp = HParams(lr=lr, relative_step=False, scale_parameter=False, beta1=b1, weight_decay=wd)
    g = rank1(4, 6, 12)
    p0 = np.random.default_rng(13).normal(0, 0.02, size=(4, 6))
    grads = [g] + [np.zeros((4, 6))] * 5
    p, st = run(p0, grads, hp)
    m = (1 - b1) * lr * np.sign(g)
    expect = p0 * (1 - wd * lr) - m
    for _ in range(5):
        m = b1 * m
        expect = expect * (1 - wd * lr) - m
    np.testing.assert_allclose(p, expect, rtol=1e-12)
    np.testing.assert_allclose(st.exp_avg, m.reshape(-1), rtol=1e-12)
    assert np.all(np.isfinite(st.row)) and np.all(st.col > 0)


def test_beta1_constant_update_closed_form():
    """Constant rank-1 g with a fixed lr: the pre-momentum update is lr sign(g)
    each step, so exp_avg_t = lr sign(g) (1 - beta1^t)."""
    lr, b1 = 0.05, 0.9
    hp = HParams(lr=lr, relative_step=False, scale_parameter=False, beta1=b1)
    g = rank1(3, 7, 14)
    p0 = np.zeros((3, 7))
    p, st = run(p0, [g] * 8, hp)
    total = sum(1 - b1 ** k for k in range(1, 9))
    np.testing.assert_allclose(p, -lr * np.sign(g) * total, rtol=1e-12)
    np.testing.assert_allclose(st.exp_avg, (lr * np.sign(g) * (1 - b1 ** 8)).reshape(-1), rtol=1e-12)


@pytest.mark.parametrize("t,warmup,rho", [
    (1, False, 1e-2), (100, False, 1e-2), (40000, False, 1.0 / 200.0),
    (1, True, 1e-6), (5000, True, 5e-3), (20000, True, 1.0 / math.sqrt(20000.0)),
])
def test_relative_step_schedule(t, warmup, rho):
    """Step 3: rho_t = min(1e-2, 1/sqrt(t)), or min(1e-6 t, 1/sqrt(t)) with
    warmup_init.  A rank-1 g from a zero state at step t gives u = sign(g) /
    sqrt(1 - beta2_t); for t > 1 that has RMS > 1, so the clip brings it back to
    sign(g) and p_1 = p_0 - rho_t * max(1e-3, RMS(p_0)) * sign(g)."""
    g = rank1(4, 5, 15)
    p0 = np.random.default_rng(16).normal(0, 0.02, size=(4, 5))
    p, _ = run(p0, [g], HParams(warmup_init=warmup), t0=t)
    np.testing.assert_allclose(p, p0 - rho * rms(p0) * np.sign(g), rtol=1e-11)


def test_scale_parameter_floor_and_off():
    g = rank1(3, 3, 17)
    p0 = np.full((3, 3), 1e-5)
    p, _ = run(p0, [g], HParams())  # RMS(p) = 1e-5 < eps2 = 1e-3
    np.testing.assert_allclose(p, p0 - 1e-2 * 1e-3 * np.sign(g), rtol=1e-12, atol=1e-19)
    p, _ = run(p0, [g], HParams(scale_parameter=False))
    np.testing.assert_allclose(p, p0 - 1e-2 * np.sign(g), rtol=1e-12)
    p, _ = run(p0, [g], HParams(lr=0.3, relative_step=False, scale_parameter=True))
    np.testing.assert_allclose(p, p0 - 0.3 * 1e-3 * np.sign(g), rtol=1e-12)


def test_leading_dims_factor_per_slice():
    """[B, H, W] is factored over the last two dims with one row/col pair per
    leading index; with the clip and parameter scale out of play every slice
    evolves exactly like a 2D tensor of its own."""
    rng = np.random.default_rng(18)
    hp = HParams(clip_threshold=1e9, scale_parameter=False)
    p3 = rng.normal(0, 0.02, size=(3, 4, 5))
    slices = [p3[b].copy() for b in range(3)]
    s3 = State(p3.shape, beta1=False)
    ss = [State((4, 5), beta1=False) for _ in range(3)]
    for t in range(1, 6):
        g = rng.normal(size=(3, 4, 5))
        oracle.step(p3, g, s3, t, hp)
        for b in range(3):
            oracle.step(slices[b], g[b], ss[b], t, hp)
    for b in range(3):
        np.testing.assert_allclose(p3[b], slices[b], rtol=1e-14)
        np.testing.assert_allclose(s3.row[b * 4:(b + 1) * 4], ss[b].row, rtol=1e-14)
        np.testing.assert_allclose(s3.col[b * 5:(b + 1) * 5], ss[b].col, rtol=1e-14)


def test_argument_errors():
    with pytest.raises(oracle.OracleError, match="Cannot combine manual lr and relative_step=True options"):
        oracle.check_hparams(HParams(lr=1e-3))
    with pytest.raises(oracle.OracleError, match="warmup_init"):
        oracle.check_hparams(HParams(lr=1e-3, relative_step=False, warmup_init=True))
    with pytest.raises(oracle.OracleError, match="manual lr"):
        oracle.check_hparams(HParams(relative_step=False))
    with pytest.raises(oracle.OracleError, match="step"):
        oracle.step(np.zeros(3), np.zeros(3), State((3,), False), 0, HParams())


def test_empty_tensor_is_untouched():
    p = np.zeros((0, 5))
    st = State((0, 5), beta1=False)
    st.col[:] = 7.0
    oracle.step(p, np.zeros((0, 5)), st, 1, HParams())
    assert np.all(st.col == 7.0)
