"""Pins of the oracle's 8-bit first moment (block quantisation of exp_avg).

The quantiser follows the ms-swift GaLore / Q-GaLore article ("Q-GaLore"
section): groups of 128 values, scale = absmax / 127, symmetric int8 codes.
Readings (also in the oracle's header): groups run along the last dim (a
tensor with ndim < 2 is one row); the step's update uses the unquantised new
moment; the codes are rint(m * (127 / amax)) in fp32.  Each pin is a closed
form or an invariant that a plausible slip breaks (flat groups across rows,
floor instead of rint, the wrong divisor, the quantised moment used for the
update, the scale not stored)."""
import numpy as np
import pytest

import oracle

HP = oracle.HParams(beta1=0.5)


def groups_of(shape):
    rows, g = oracle.q8_groups(shape)
    last = shape[-1] if len(shape) >= 2 else int(np.prod(shape))
    return rows, g, last


def step_pair(shape, g, t, hp, st, p):
    """One oracle step; returns the applied update (p before - p after)."""
    before = p.copy()
    oracle.step(p, g, st, t, hp)
    return before - p


def test_q8_needs_beta1():
    st = oracle.State((4, 4), beta1=False, q8=True)
    with pytest.raises(oracle.OracleError, match="beta1"):
        oracle.step(np.zeros((4, 4)), np.ones((4, 4)), st, 1, oracle.HParams())


def test_rank1_gradient_gives_full_codes_and_closed_form_updates():
    """g = a (x) b makes u = alpha * sign(g) exactly (factored estimate exact,
    RMS(u) = 1, no clip), so every |m| in a group is equal: the codes are
    +-127 with the sign of g, the scale is fl32(fl32(m)/127), and the update
    of step 2 uses the dequantised old moment fl32(127 * scale)."""
    a = np.array([0.3, -1.2, 0.7, 2.0])
    b = np.linspace(-1.0, 1.5, 260) + 0.013
    g = np.outer(a, b)
    shape = g.shape
    p = np.random.default_rng(3).normal(0, 0.05, shape)
    st = oracle.State(shape, beta1=True, q8=True)
    ref = oracle.State(shape, beta1=True)
    p_ref = p.copy()
    d1 = step_pair(shape, g, 1, HP, st, p)
    oracle.step(p_ref, g, ref, 1, HP)
    np.testing.assert_array_equal(p, p_ref)  # step 1: old moment 0, update = unquantised moment
    alpha1 = 1e-2 * max(1e-3, np.sqrt(np.mean((p + d1) ** 2)))
    m1 = 0.5 * alpha1
    np.testing.assert_allclose(np.abs(d1), m1, rtol=1e-12)
    codes = st.exp_avg_codes.reshape(shape)
    np.testing.assert_array_equal(codes, 127 * np.sign(g).astype(np.int8))
    s1 = np.float32(np.float32(m1) / np.float32(127))
    np.testing.assert_array_equal(st.exp_avg_scales, s1)
    # step 2, same gradient
    p1 = p.copy()
    alpha2 = min(1e-2, 1 / np.sqrt(2)) * max(1e-3, np.sqrt(np.mean(p1 ** 2)))
    d2 = step_pair(shape, g, 2, HP, st, p)
    old = np.float64(np.float32(127) * s1)
    m2 = 0.5 * old + 0.5 * alpha2
    np.testing.assert_allclose(d2, m2 * np.sign(g), rtol=1e-12)


@pytest.mark.parametrize("shape", [(5, 300), (2, 3, 130), (1000,), (7, 128), (3, 1)])
def test_codes_scales_invariants_per_row_groups(shape):
    """After a step: |code| <= 127; in every group of 128 along the last dim
    max |code| = 127 (scale > 0); scale = fl32(amax / 127) with amax the
    group's max |fl32(m)|; |code - m * 127 / amax| <= 1/2; the applied update
    is the unquantised m (weight decay 0)."""
    rng = np.random.default_rng(11)
    p = rng.normal(0, 0.1, shape)
    st = oracle.State(shape, beta1=True, q8=True)
    hp = oracle.HParams(beta1=0.8)
    for t in range(1, 4):
        g = rng.standard_t(3, shape) * 1e-2
        m = step_pair(shape, g, t, hp, st, p).reshape(-1)
    rows, ng, last = groups_of(shape)
    codes = st.exp_avg_codes.reshape(rows, last).astype(np.int64)
    scales = st.exp_avg_scales.reshape(rows, ng)
    mq = m.reshape(rows, last).astype(np.float32)
    assert np.all(np.abs(codes) <= 127)
    for r in range(rows):
        for k in range(ng):
            sl = slice(128 * k, min(128 * (k + 1), last))
            amax = np.float32(np.max(np.abs(mq[r, sl])))
            assert amax > 0
            assert np.max(np.abs(codes[r, sl])) == 127
            assert scales[r, k] == np.float32(amax / np.float32(127))
            x = mq[r, sl].astype(np.float64) * 127.0 / float(amax)
            assert np.all(np.abs(codes[r, sl] - x) <= 0.5 + 1e-4)


def test_zero_gradient_keeps_codes_and_decays_scales():
    """g = 0 gives u = 0, so m = beta1 * code * scale: the codes stay (up to a
    rounding far from any tie) and the scale becomes beta1 times the old one;
    an all-zero state stays all zero."""
    shape = (3, 200)
    rng = np.random.default_rng(5)
    p = rng.normal(0, 0.1, shape)
    st = oracle.State(shape, beta1=True, q8=True)
    hp = oracle.HParams(beta1=0.6)
    oracle.step(p, rng.normal(0, 1e-2, shape), st, 1, hp)
    codes0, scales0 = st.exp_avg_codes.copy(), st.exp_avg_scales.copy()
    p_before = p.copy()
    oracle.step(p, np.zeros(shape), st, 2, hp)
    np.testing.assert_array_equal(st.exp_avg_codes, codes0)
    np.testing.assert_allclose(st.exp_avg_scales, 0.6 * scales0, rtol=2e-7)
    dq = codes0.astype(np.float64) * np.repeat(scales0.reshape(3, 2), [128, 72], axis=1).reshape(-1)
    np.testing.assert_allclose((p_before - p).reshape(-1), 0.6 * dq, rtol=1e-6, atol=1e-20)
    z = oracle.State(shape, beta1=True, q8=True)
    pz = p.copy()
    oracle.step(pz, np.zeros(shape), z, 1, hp)
    assert not z.exp_avg_codes.any() and not z.exp_avg_scales.any()
    np.testing.assert_array_equal(pz, p)


def test_groups_do_not_span_rows():
    """A large gradient in row 1 of a W = 130 tensor leaves row 0's scales to
    row 0's own values (groups [0, 128) and [128, 130) of each row)."""
    shape = (2, 130)
    rng = np.random.default_rng(9)
    g = rng.normal(0, 1e-2, shape)
    g[1, :2] = 5.0  # would dominate a flat group spanning rows 0 and 1
    p = rng.normal(0, 0.1, shape)
    st = oracle.State(shape, beta1=True, q8=True)
    m = step_pair(shape, g, 1, HP, st, p).reshape(shape).astype(np.float32)
    scales = st.exp_avg_scales.reshape(2, 2)
    assert scales[0, 1] == np.float32(np.max(np.abs(m[0, 128:])) / np.float32(127))
    assert np.max(np.abs(st.exp_avg_codes.reshape(shape)[0, 128:])) == 127
