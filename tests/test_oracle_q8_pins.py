"""Pins of the oracle's 8-bit first moment (block quantisation of exp_avg).

The quantiser is the quantize_tensor listing of the ms-swift GaLore /
Q-GaLore article ("双重压缩：Q-Galore 的量化飞跃" section): groups of 128
values, scale = absmax / 127, code = (x / scale) rounded (torch's round, ties
to even) and clamped to [-128, 127]; dequantised value code * scale.  The
QGaloreAdam listing beside it dequantises the stored moment before the update
is formed from it.  Readings (also in the oracle's header): groups run along
the last dim (a tensor with ndim < 2 is one row); the quantiser works in fp32,
the listing's tensor precision; the update applied to the parameter is the
dequantised new moment.

Each pin is a closed form, an exact tie, or an invariant that a plausible slip
breaks: flat groups across rows, floor or half-away rounding, the code taken
as m * (127 / amax) instead of m / scale, the wrong divisor of the scale, the
unquantised moment used for the update, the old moment not dequantised."""
import numpy as np
import pytest

import oracle

HP = oracle.HParams(beta1=0.5)
f32 = np.float32


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


def test_exact_ties_round_half_to_even():
    """Groups whose absmax is 127 * s with s a small integer have scale = s
    exactly, so x / scale of a value (k + 1/2) s is exactly k + 1/2 and torch's
    round sends it to the even neighbour.  With s = 7 the product x * fl(127 /
    amax) lands just above the tie (6.5000005 for x = 45.5), so a quantiser
    that multiplies by the reciprocal instead of dividing rounds these up."""
    m = np.zeros(3 * 128)
    # group 0: scale 1
    m[0:7] = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5]
    # group 1: scale 7
    m[128:132] = [889.0, 45.5, 87.5, -101.5]
    # group 2: all zero -> code 0 and scale 0
    codes, scales = oracle.q8_quantize(m, (3 * 128,))
    np.testing.assert_array_equal(scales, [1.0, 7.0, 0.0])
    np.testing.assert_array_equal(codes[0:7], [127, 2, 4, -2, 0, 2, 0])
    np.testing.assert_array_equal(codes[128:132], [127, 6, 12, -14])
    assert not codes[7:128].any() and not codes[132:].any()


def test_scale_is_absmax_over_127():
    """absmax 1 gives scale fl32(1/127) (not 1/128), and the group's absmax
    value gets code +-127 exactly."""
    m = np.zeros(128)
    m[5] = -1.0
    m[6] = 0.25
    codes, scales = oracle.q8_quantize(m, (1, 128))
    assert scales[0] == f32(1.0) / f32(127.0)
    assert codes[5] == -127
    assert codes[6] == 32  # 0.25 / (1/127) = 31.75


def test_rank1_gradient_gives_full_codes_and_closed_form_updates():
    """g = a (x) b makes u = alpha * sign(g) exactly (factored estimate exact,
    RMS(u) = 1, no clip), so every |m| in a group is equal: the codes are
    +-127 with the sign of g and the scale is fl32(fl32(m) / 127).  The update
    applied is the dequantised moment fl32(127 * scale), and step 2 starts
    from that value as its old moment."""
    a = np.array([0.3, -1.2, 0.7, 2.0])
    b = np.linspace(-1.0, 1.5, 260) + 0.013
    g = np.outer(a, b)
    shape = g.shape
    p = np.random.default_rng(3).normal(0, 0.05, shape)
    st = oracle.State(shape, beta1=True, q8=True)
    alpha1 = 1e-2 * max(1e-3, np.sqrt(np.mean(p ** 2)))
    d1 = step_pair(shape, g, 1, HP, st, p)
    m1 = 0.5 * alpha1
    codes = st.exp_avg_codes.reshape(shape)
    np.testing.assert_array_equal(codes, 127 * np.sign(g).astype(np.int8))
    s1 = f32(f32(m1) / f32(127))
    np.testing.assert_array_equal(st.exp_avg_scales, s1)
    deq1 = np.float64(f32(127) * s1)
    assert abs(deq1 - m1) > 1e-13  # the pin tells the dequantised value from m itself
    np.testing.assert_allclose(d1, deq1 * np.sign(g), rtol=0, atol=1e-16)
    # step 2, same gradient: old moment = deq1
    alpha2 = min(1e-2, 1 / np.sqrt(2)) * max(1e-3, np.sqrt(np.mean(p ** 2)))
    d2 = step_pair(shape, g, 2, HP, st, p)
    m2 = 0.5 * deq1 + 0.5 * alpha2
    s2 = f32(f32(m2) / f32(127))
    np.testing.assert_allclose(st.exp_avg_scales, s2, rtol=1e-7)
    np.testing.assert_allclose(d2, np.float64(f32(127) * s2) * np.sign(g), rtol=1e-7)


@pytest.mark.parametrize("shape", [(5, 300), (2, 3, 130), (1000,), (7, 128), (3, 1)])
def test_codes_scales_invariants_per_row_groups(shape):
    """After a step: |code| <= 127; in every group of 128 along the last dim
    max |code| = 127 (scale > 0); scale = fl32(amax / 127) with amax the
    group's max |fl32(m)|; |code - m / scale| <= 1/2; and the update applied
    (weight decay 0) is exactly fl32(code * scale), not the moment m itself."""
    rng = np.random.default_rng(11)
    p = rng.normal(0, 0.1, shape)
    st = oracle.State(shape, beta1=True, q8=True)
    hp = oracle.HParams(beta1=0.8)
    for t in range(1, 4):
        g = rng.standard_t(3, shape) * 1e-2
        d = step_pair(shape, g, t, hp, st, p).reshape(-1)
    m = st.moment
    rows, ng, last = groups_of(shape)
    codes = st.exp_avg_codes.reshape(rows, last).astype(np.int64)
    scales = st.exp_avg_scales.reshape(rows, ng)
    mq = m.reshape(rows, last).astype(np.float32)
    assert np.all(np.abs(codes) <= 127)
    deq = np.zeros((rows, last))
    for r in range(rows):
        for k in range(ng):
            sl = slice(128 * k, min(128 * (k + 1), last))
            amax = np.float32(np.max(np.abs(mq[r, sl])))
            assert amax > 0
            assert np.max(np.abs(codes[r, sl])) == 127
            assert scales[r, k] == np.float32(amax / np.float32(127))
            x = mq[r, sl].astype(np.float64) / float(scales[r, k])
            assert np.all(np.abs(codes[r, sl] - x) <= 0.5 + 1e-5)
            deq[r, sl] = (codes[r, sl].astype(np.float32) * scales[r, k]).astype(np.float64)
    # (d is p_before - p_after in float64: exact up to one rounding of p)
    np.testing.assert_allclose(d, deq.reshape(-1), rtol=0, atol=1e-16)
    assert np.mean(np.abs(deq.reshape(-1) - m) > 1e-14) > 0.9  # the dequantised value, not m itself


def test_zero_gradient_keeps_codes_and_decays_scales():
    """g = 0 gives u = 0, so m = beta1 * code * scale: the codes stay (the
    quotients are within a few ulps of the old integer codes, far from any
    tie), the scale becomes beta1 times the old one and the update is the new
    dequantised moment; an all-zero state stays all zero."""
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
    dq = codes0.astype(np.float64) * np.repeat(st.exp_avg_scales.reshape(3, 2).astype(np.float64),
                                               [128, 72], axis=1).reshape(-1)
    np.testing.assert_allclose((p_before - p).reshape(-1), dq, rtol=1e-7, atol=1e-20)
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
    step_pair(shape, g, 1, HP, st, p)
    m = st.moment.reshape(shape).astype(np.float32)
    scales = st.exp_avg_scales.reshape(2, 2)
    assert scales[0, 1] == np.float32(np.max(np.abs(m[0, 128:])) / np.float32(127))
    assert np.max(np.abs(st.exp_avg_codes.reshape(shape)[0, 128:])) == 127


def test_three_parts_make_the_step():
    """oracle.step on an 8-bit state equals q8_moment, q8_quantize and
    q8_apply run in order (the parts the GPU parity test reconciles
    between)."""
    shape = (6, 260)
    rng = np.random.default_rng(21)
    p0 = rng.normal(0, 0.1, shape)
    hp = oracle.HParams(beta1=0.9, weight_decay=0.01)
    a, b = oracle.State(shape, True, q8=True), oracle.State(shape, True, q8=True)
    pa, pb = p0.copy(), p0.copy()
    for t in range(1, 4):
        g = rng.normal(0, 1e-2, shape)
        oracle.step(pa, g, a, t, hp)
        m, alpha = oracle.q8_moment(pb, g, b, t, hp)
        b.exp_avg_codes[:], b.exp_avg_scales[:] = oracle.q8_quantize(m, shape)
        oracle.q8_apply(pb, b.exp_avg_codes, b.exp_avg_scales, shape, alpha, hp)
    np.testing.assert_array_equal(pa, pb)
    np.testing.assert_array_equal(a.exp_avg_codes, b.exp_avg_codes)
    np.testing.assert_array_equal(a.row, b.row)
