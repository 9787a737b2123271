"""8-bit first moment (exp_avg_int8) against the float64 oracle's quantised mode.

The oracle quantises as the ms-swift Q-GaLore quantize_tensor listing does
(scale = amax / 127, code = round-half-even(m / scale), in fp32) and applies
the dequantised moment; the kernels must give the same codes.  A code is an
integer decided by rounding the quotient m / scale, and the GPU's m carries
the fp32 rounding of the whole step upstream (the statistics, u, the clip),
while the oracle's m is float64 rounded once.  Where the quotient lies within
TIE_BAND of a half-integer, both roundings are correct answers for the same
moment; nowhere else may the codes differ.

TIE_BAND = 1e-3: the quotient is 127 m / amax, so a relative error e of m
(and of amax) moves it by at most 2 * 127 * e; 1e-3 covers e up to 3.9e-6,
about 33 fp32 ulps, several times the measured deviation of the fp32 step
(the parameter and statistics checks below hold it to the 2e-5 bar).

The oracle keeps its own state throughout (its own codes and scales from
step 1 on).  At a tie-band flip it adopts the GPU's code for that element
before applying the step, so that both sides continue from the same valid
state; every other element of the state evolves independently.  Checked
after each step: parameters and second moments within the 2e-5 bar, scales
at relative 2e-5 with an absolute slack of 1e-6 of the tensor's largest
scale (check_scales), codes equal outside the tie band, and fewer than 1e-3
of the codes flipped at ties."""
import numpy as np
import pytest
import torch

import oracle
from memory_efficient_optimizer_gb300 import synth
from memory_efficient_optimizer_gb300.optim import AdafactorStep, init_state, q8_scale_count
from parity_util import check, oracle_hp, to64

SHAPES = [(300, 2056), (131, 4104), (1000, 1032), (64, 1024), (257, 1025), (2, 3, 130), (9000,), (600,), (3, 1)]
FLAGS = [
    dict(beta1=0.9, weight_decay=0.01, exp_avg_int8=True),
    dict(lr=1e-3, relative_step=False, scale_parameter=False, beta1=0.9, weight_decay=0.01, exp_avg_int8=True),
]
TIE_BAND = 1e-3


def tie_distance(m, scales, shape):
    """Distance of each quotient fl32(m) / scale from the nearest half-integer
    (inf where the group's scale is 0)."""
    rows, groups = oracle.q8_groups(shape)
    last = shape[-1] if len(shape) >= 2 else int(np.prod(shape))
    m32 = np.asarray(m, np.float32).reshape(rows, last).astype(np.float64)
    sc = np.repeat(np.asarray(scales, np.float64).reshape(rows, groups), 128, axis=1)[:, :last]
    with np.errstate(divide="ignore", invalid="ignore"):
        x = np.where(sc > 0, m32 / np.where(sc > 0, sc, 1.0), np.nan)
    d = np.abs((x - np.floor(x)) - 0.5)
    return np.where(np.isnan(d), np.inf, d).reshape(-1)


def compare_codes(name, gpu_codes, ref_codes, m, ref_scales, shape):
    """Codes equal except by one at tie-band quotients; returns the flip mask."""
    got = np.asarray(gpu_codes).astype(np.int64).reshape(-1)
    ref = np.asarray(ref_codes).astype(np.int64).reshape(-1)
    bad = got != ref
    if bad.any():
        assert np.all(np.abs(got - ref)[bad] == 1), f"{name}: a code differs by more than one"
        dist = tie_distance(m, ref_scales, shape)
        worst = float(np.max(dist[bad]))
        assert worst < TIE_BAND, f"{name}: a code differs {worst:.3g} away from a rounding tie"
    return bad


def check_scales(name, gpu, ref):
    """Scales at relative 2e-5, with an absolute slack of 1e-6 of the
    tensor's largest scale.  A scale is amax / 127 of the new moment
    m = beta1 * old + (1 - beta1) * u; where old and u nearly cancel over a
    whole group (a group of one value at the end of a row, say), m keeps the
    fp32 rounding of its terms, which are bounded by the tensor's largest
    moments, not by m itself: the same bar the fp32 exp_avg takes."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    top = float(np.max(np.abs(ref))) if ref.size else 0.0
    check(name, gpu, ref, atol=max(1e-6 * top, 1e-30))


def gpu_state(states, k, n_sc):
    codes = states[k]["exp_avg_codes"].cpu().numpy().reshape(-1)
    scales = states[k]["exp_avg_scales"].cpu().numpy()[:n_sc]
    return codes, scales


def check_second_moment(nm, states, k, rs):
    if rs.row is not None:
        check(nm + ".row", to64(states[k]["exp_avg_sq_row"]), rs.row, atol=1e-30)
        check(nm + ".col", to64(states[k]["exp_avg_sq_col"]), rs.col, atol=1e-30)
    else:
        check(nm + ".exp_avg_sq", to64(states[k]["exp_avg_sq"]), rs.v, atol=1e-30)


def setup(flags, grad_dtype):
    hp = dict(flags)
    ohp = oracle_hp({k: v for k, v in hp.items() if k != "exp_avg_int8"})
    params = [synth.make_param(s, k, std=0.3).cuda() for k, s in enumerate(SHAPES)]
    ref_p = [to64(p) for p in params]
    ref_st = [oracle.State(s, beta1=True, q8=True) for s in SHAPES]
    grads = [torch.empty(s, dtype=grad_dtype, device="cuda") for s in SHAPES]
    states = init_state(params, beta1=hp["beta1"], exp_avg_int8=True)
    for k, s in enumerate(SHAPES):
        assert states[k]["exp_avg_scales"].numel() == max(1, q8_scale_count(s))
    return hp, ohp, params, ref_p, ref_st, grads, states


@pytest.mark.gpu
@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("flags", FLAGS)
def test_int8_step1_unforced(flags, grad_dtype):
    """Step 1 from the all-zero state, the oracle's plain step with no input
    from the GPU: codes equal outside the tie band; parameters within the bar,
    where a tie flipped once the oracle's parameter is moved by the one code
    step (the scale) that the other rounding applies."""
    hp, ohp, params, ref_p, ref_st, grads, states = setup(flags, grad_dtype)
    step = AdafactorStep(params, grads, states, **hp)
    for k, s in enumerate(SHAPES):
        g = synth.make_grad(s, k, 1, std=0.01, dtype=grad_dtype, kind="student_t_zero_rows")
        grads[k].copy_(g)
        oracle.step(ref_p[k], to64(g), ref_st[k], 1, ohp)
    step(1)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    flips = 0
    for k, s in enumerate(SHAPES):
        nm = f"q8-step1[{k}]{s}"
        rs = ref_st[k]
        codes, scales = gpu_state(states, k, rs.exp_avg_scales.size)
        check_scales(nm + ".scales", scales, rs.exp_avg_scales)
        bad = compare_codes(nm, codes, rs.exp_avg_codes, rs.moment, rs.exp_avg_scales, s)
        flips += int(bad.sum())
        p_gpu = to64(params[k]).reshape(-1)
        p_ref = ref_p[k].reshape(-1).copy()
        if bad.any():  # the oracle's parameter as if it had taken the GPU's code at the flips
            rows, groups = oracle.q8_groups(s)
            last = s[-1] if len(s) >= 2 else int(np.prod(s))
            sc = np.repeat(rs.exp_avg_scales.reshape(rows, groups).astype(np.float64), 128, axis=1)[:, :last]
            dc = rs.exp_avg_codes.astype(np.float64) - codes.astype(np.float64)
            p_ref[bad] += (dc * sc.reshape(-1))[bad]
        check(nm + ".param", p_gpu, p_ref)
        check_second_moment(nm, states, k, rs)
    total = sum(int(np.prod(s)) for s in SHAPES)
    assert flips <= 1e-3 * total, f"{flips} tie flips out of {total} codes"


@pytest.mark.gpu
@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("flags", FLAGS)
def test_int8_first_moment_matches_oracle(flags, grad_dtype):
    steps = 6
    hp, ohp, params, ref_p, ref_st, grads, states = setup(flags, grad_dtype)
    step = AdafactorStep(params, grads, states, **hp)
    flips = 0
    for t in range(1, steps + 1):
        host_g = []
        for k, s in enumerate(SHAPES):
            g = synth.make_grad(s, k, t, std=0.01, dtype=grad_dtype, kind="student_t_zero_rows")
            grads[k].copy_(g)
            host_g.append(to64(g))
        step(t)
        torch.cuda.synchronize()
        assert step.device_status() == 0
        for k, s in enumerate(SHAPES):
            nm = f"q8[{k}]{s} t={t}"
            rs = ref_st[k]
            m, alpha = oracle.q8_moment(ref_p[k], host_g[k], rs, t, ohp)
            codes_o, scales_o = oracle.q8_quantize(m, s)
            codes_g, scales_g = gpu_state(states, k, scales_o.size)
            check_scales(nm + ".scales", scales_g, scales_o)
            bad = compare_codes(nm, codes_g, codes_o, m, scales_o, s)
            flips += int(bad.sum())
            codes_o[bad] = codes_g[bad]  # both roundings of a tie are valid: continue from the GPU's
            rs.exp_avg_codes[:], rs.exp_avg_scales[:] = codes_o, scales_o
            oracle.q8_apply(ref_p[k], rs.exp_avg_codes, rs.exp_avg_scales, s, alpha, ohp)
            check(nm + ".param", to64(params[k]), ref_p[k])
            check_second_moment(nm, states, k, rs)
    total = sum(int(np.prod(s)) for s in SHAPES) * steps
    assert flips <= 1e-3 * total, f"{flips} tie flips out of {total} codes"


@pytest.mark.gpu
def test_int8_state_is_a_quarter_of_fp32():
    """The 8-bit state of a Llama-sized matrix: 1 byte per value plus one
    fp32 scale per 128 values (1.03 bytes), against 4 for fp32 exp_avg."""
    p = torch.zeros(4096, 4096, device="cuda")
    st = init_state([p], beta1=0.9, exp_avg_int8=True)[0]
    nbytes = st["exp_avg_codes"].numel() + 4 * st["exp_avg_scales"].numel()
    assert nbytes == 4096 * 4096 + 4 * 4096 * 32
