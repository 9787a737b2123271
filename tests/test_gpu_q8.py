"""8-bit first moment (exp_avg_int8) against the float64 oracle's quantised mode.

The codes are integers decided by rounding, so a value that falls within a
few fp32 ulps of a rounding tie may round either way depending on fp32 vs
float64 arithmetic upstream.  The test therefore teacher-forces the first-
moment state: before every step the oracle takes the GPU's codes and scales,
so both sides start each step from identical moments; parameters and second
moments evolve independently on both sides over all the steps.  After each
step: parameters and second moments within the 2e-5 bar, scales within 2e-5,
and every code equal to the oracle's except, by at most one, where the
oracle's m * 127 / amax lies within 1e-3 of a half-integer tie."""
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


def check_codes(name, gpu_codes, ref, moment):
    ref_codes = ref.exp_avg_codes.astype(np.int64)
    got = gpu_codes.astype(np.int64)
    bad = got != ref_codes
    if not bad.any():
        return 0
    assert np.all(np.abs(got - ref_codes)[bad] == 1), f"{name}: a code differs by more than one"
    rows, groups = oracle.q8_groups(ref.shape)
    last = ref.shape[-1] if len(ref.shape) >= 2 else int(np.prod(ref.shape))
    m32 = moment.astype(np.float32).reshape(rows, last)
    amax = np.zeros((rows, groups), np.float32)
    for k in range(groups):
        amax[:, k] = np.max(np.abs(m32[:, 128 * k:128 * (k + 1)]), axis=1)
    inv = np.where(amax > 0, np.float32(127) / np.where(amax > 0, amax, 1), 0).astype(np.float32)
    x = (m32 * np.repeat(inv, 128, axis=1)[:, :last]).reshape(-1).astype(np.float64)
    tie = np.abs(np.abs(x - np.floor(x)) - 0.5)
    assert np.all(tie[bad] < 1e-3), f"{name}: a code differs away from a rounding tie"
    return int(bad.sum())


@pytest.mark.gpu
@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("flags", FLAGS)
def test_int8_first_moment_matches_oracle(flags, grad_dtype):
    steps = 6
    hp = dict(flags)
    ohp = oracle_hp({k: v for k, v in hp.items() if k != "exp_avg_int8"})
    params = [synth.make_param(s, k, std=0.3).cuda() for k, s in enumerate(SHAPES)]
    ref_p = [to64(p) for p in params]
    ref_st = [oracle.State(s, beta1=True, q8=True) for s in SHAPES]
    grads = [torch.empty(s, dtype=grad_dtype, device="cuda") for s in SHAPES]
    states = init_state(params, beta1=hp["beta1"], exp_avg_int8=True)
    for k, s in enumerate(SHAPES):
        assert states[k]["exp_avg_scales"].numel() == max(1, q8_scale_count(s))
    step = AdafactorStep(params, grads, states, **hp)
    flips = 0
    for t in range(1, steps + 1):
        for k, s in enumerate(SHAPES):
            g = synth.make_grad(s, k, t, std=0.01, dtype=grad_dtype, kind="student_t_zero_rows")
            grads[k].copy_(g)
            # teacher forcing of the first moment: start from the GPU's codes and scales
            ref_st[k].exp_avg_codes[:] = states[k]["exp_avg_codes"].cpu().numpy().reshape(-1)
            n_sc = ref_st[k].exp_avg_scales.size
            ref_st[k].exp_avg_scales[:] = states[k]["exp_avg_scales"].cpu().numpy()[:n_sc]
            oracle.step(ref_p[k], to64(g), ref_st[k], t, ohp)
        step(t)
        torch.cuda.synchronize()
        assert step.device_status() == 0
        for k, s in enumerate(SHAPES):
            nm = f"q8[{k}]{s} t={t}"
            check(nm + ".param", to64(params[k]), ref_p[k])
            rs = ref_st[k]
            if rs.row is not None:
                check(nm + ".row", to64(states[k]["exp_avg_sq_row"]), rs.row, atol=1e-30)
                check(nm + ".col", to64(states[k]["exp_avg_sq_col"]), rs.col, atol=1e-30)
            else:
                check(nm + ".exp_avg_sq", to64(states[k]["exp_avg_sq"]), rs.v, atol=1e-30)
            sc = states[k]["exp_avg_scales"].cpu().numpy()[:rs.exp_avg_scales.size].astype(np.float64)
            check(nm + ".scales", sc, rs.exp_avg_scales.astype(np.float64), atol=1e-30)
            flips += check_codes(nm, states[k]["exp_avg_codes"].cpu().numpy().reshape(-1), rs, rs.moment)
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
