"""GPU parity of the CAME step (include/came.h) against the float64 CAME
oracle, element by element on the same seeded inputs.

Bar (per element, after the steps): |gpu - ref| <= 1e-7 + 2e-5 |ref| on the
parameters, plus each parameter's accumulated change to 2e-5 of the sum of
its per-step updates; every statistic (second moment and instability,
factored or full: sums of positive terms) at relative 2e-5.

The momentum m_t = b1 m_{t-1} + (1 - b1) uh_t is an EMA of signed clipped
updates, so an element can cancel to near zero while its terms are of order
one.  Its bar follows from the one the update takes: each uh_t may carry
2e-5 of its own size (the update bar), and each step rounds m to fp32 (at
most 2^-24 of the EMA of |uh|).  Then
    |m_gpu - m_ref| <= (2e-5 + T 2^-24) E_T,   E_t = b1 E_{t-1} + (1 - b1) |uh_t|,
the envelope E being the same EMA taken of |uh|.  The test rebuilds uh_t from
the oracle's consecutive momenta (uh_t = (m_t - b1 m_{t-1}) / (1 - b1)) and
reports the worst |dm| / bound beside RMS(m).
"""
import numpy as np
import pytest
import torch

from memory_efficient_optimizer_gb300 import synth
from memory_efficient_optimizer_gb300.came import Came, CameStep, came_step, init_came_state
from parity_util import RTOL, check, check_update, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from memory_efficient_optimizer_gb300 import build
    from oracle import came as came_oracle
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    came_oracle.build()


def oracle_hp(hp):
    from oracle.came import CameHParams
    return CameHParams(**hp)


# vector-class matrices (W % 8 == 0), scalar-class ones (odd W), several row
# and column tiles with ragged ends, 3-D and 4-D views, 1-row / 1-column
# matrices, 1-D tensors around the 8192-value units, an empty tensor; with
# bf16 gradients the row-panel pass takes (4, 4096), (3, 2056) and (300, 2048)
# (256-row chunks, a ragged last chunk), (2, 70, 4104) (128-row chunks, two
# slices, a ragged column group) and (1, 14336); (1, 16384) stays on the tiled passes
SHAPES = [(1,), (5,), (8193,), (0,), (7, 13), (1, 37), (37, 1), (64, 64), (300, 1030), (257, 1032),
          (2, 3, 520, 264), (2, 5, 9), (1000, 40), (4, 4096), (3, 2056), (300, 2048), (2, 70, 4104), (1, 14336),
          (1, 16384)]
HPARAMS = [
    dict(lr=1e-3),
    dict(lr=1e-3, weight_decay=0.1, clip_threshold=0.05),
    dict(lr=1e-3, betas=(0.5, 0.9, 0.95), eps=(1e-20, 1e-10)),
    dict(lr=1e-4, clip_threshold=100.0),
]
# Learning rates at which CAME's confidence-scaled steps move p by a large
# fraction of its size every step: p then cancels towards 0 and its
# element-wise relative bar measures the cancellation, not the step, so
# these runs take the per-step update bar (check_update) instead.
LARGE_LR = [
    dict(lr=1e-2, weight_decay=0.1, clip_threshold=0.05),
    dict(lr=3e-3, clip_threshold=100.0),
]
STATE_NAMES = ("exp_avg_sq_row", "exp_avg_sq_col", "exp_avg_res_row", "exp_avg_res_col")


def momentum_bound(env, steps):
    """Per-element bar of the momentum from the envelope E of |uh|."""
    return (RTOL + steps * 2.0 ** -24) * env + 1e-30


def check_momentum(name, gpu, ref, env, steps):
    """|dm| <= (2e-5 + T 2^-24) E elementwise; returns (worst |dm| / bound,
    worst |dm|, RMS(m))."""
    gpu = np.asarray(gpu, np.float64).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    bound = momentum_bound(np.asarray(env).reshape(-1), steps)
    err = np.abs(gpu - ref)
    if err.size == 0:
        return 0.0, 0.0, 0.0
    ratio = err / bound
    k = int(np.argmax(ratio))
    assert np.all(np.isfinite(gpu)) and ratio[k] <= 1.0, (
        f"{name}: |dm| = {err[k]:.3g} at {k} above (2e-5 + T 2^-24) E = {bound[k]:.3g} "
        f"(gpu={gpu[k]!r} ref={ref[k]!r})")
    return float(ratio[k]), float(err.max()), float(np.sqrt(np.mean(np.square(ref))))


MOMENTUM_REPORT = []


def run_came(shapes, hp, grad_dtype, steps, params=None, grad_std=1e-3, zero_grad_tensor=None):
    from oracle import came as came_oracle
    dev = "cuda"
    if params is None:
        params = [synth.make_param(s, k).to(dev) for k, s in enumerate(shapes)]
    ref_p = [to64(p) for p in params]
    p0 = [x.copy() for x in ref_p]
    abs_upd = [np.zeros(x.size) for x in ref_p]
    ref_st = [came_oracle.CameState(s) for s in shapes]
    env = [np.zeros(x.size) for x in ref_p]  # EMA of |uh| (the momentum's envelope)
    b1 = float(oracle_hp(hp).betas[0])
    grads = [torch.empty(s, dtype=grad_dtype, device=dev) for s in shapes]
    states = init_came_state(params)
    step = CameStep(params, grads, states, **hp)
    for t in range(1, steps + 1):
        for k, s in enumerate(shapes):
            g = synth.make_grad(s, k, t, std=grad_std, dtype=grad_dtype, kind="student_t_zero_rows")
            if zero_grad_tensor == k:
                g.zero_()
            grads[k].copy_(g)
            before = ref_p[k].copy()
            m_before = ref_st[k].exp_avg.copy()
            came_oracle.step(ref_p[k], to64(g), ref_st[k], t, oracle_hp(hp))
            abs_upd[k] += np.abs(ref_p[k] - before).reshape(-1)
            uh = (ref_st[k].exp_avg - b1 * m_before) / (1.0 - b1)
            env[k] = b1 * env[k] + (1.0 - b1) * np.abs(uh)
        step(t)
    torch.cuda.synchronize()
    return params, states, ref_p, ref_st, (p0, abs_upd, steps, env)


def compare(params, states, ref_p, ref_st, upd, tag="", p_bar=True):
    p0, abs_upd, steps, env = upd
    worst = (0.0, 0.0, 0.0)
    for k in range(len(params)):
        if p_bar:
            check(f"{tag}p[{k}]", to64(params[k]), ref_p[k])
        check_update(f"{tag}update[{k}]", to64(params[k]), ref_p[k], p0[k], steps, abs_upd[k])
        r = check_momentum(f"{tag}exp_avg[{k}]", to64(states[k]["exp_avg"]), ref_st[k].exp_avg, env[k], steps)
        worst = max(worst, r)
        if "exp_avg_sq_row" in states[k]:
            for name, ref in zip(STATE_NAMES, (ref_st[k].row, ref_st[k].col, ref_st[k].res_row, ref_st[k].res_col)):
                check(f"{tag}{name}[{k}]", to64(states[k][name]), ref, atol=1e-30)
        else:
            check(f"{tag}exp_avg_sq[{k}]", to64(states[k]["exp_avg_sq"]), ref_st[k].v, atol=1e-30)
            check(f"{tag}exp_avg_res[{k}]", to64(states[k]["exp_avg_res"]), ref_st[k].res, atol=1e-30)
    MOMENTUM_REPORT.append((tag, worst))
    print(f"momentum {tag or 'run'}: worst |dm|/bound {worst[0]:.3g}, worst |dm| {worst[1]:.3g}, "
          f"RMS(m) of that tensor {worst[2]:.3g}")


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("hp", HPARAMS)
def test_came_small_shapes(hp, grad_dtype):
    compare(*run_came(SHAPES, hp, grad_dtype, steps=6))


@pytest.mark.parametrize("hp", LARGE_LR)
def test_came_large_learning_rates_update_bar(hp):
    compare(*run_came(SHAPES, hp, torch.bfloat16, steps=6), p_bar=False)


def test_came_zero_gradient_tensors():
    """Tensors whose gradient is always 0 (u = 0: p only decays)."""
    shapes = [(300, 16), (513,), (64, 64)]
    compare(*run_came(shapes, dict(lr=0.01, weight_decay=0.05), torch.float32, steps=3, zero_grad_tensor=0))


def test_came_misaligned_views_take_the_scalar_path():
    shapes = [(64, 1024), (33, 520), (1000,)]
    bufs = [torch.zeros(int(np.prod(s)) + 1, device="cuda") for s in shapes]
    params = [b[1:].view(s) for b, s in zip(bufs, shapes)]
    for k, (p, s) in enumerate(zip(params, shapes)):
        p.copy_(synth.make_param(s, k))
    compare(*run_came(shapes, dict(lr=1e-3, weight_decay=0.01), torch.bfloat16, steps=4, params=params))


def test_came_bitwise_deterministic():
    shapes = [(257, 1032), (300, 1030), (8193,)]
    res = []
    for _ in range(2):
        params, states, *_rest = run_came(shapes, dict(lr=1e-3), torch.bfloat16, steps=3)
        res.append([p.clone() for p in params] + [st["exp_avg"].clone() for st in states])
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_came_optimizer_wrapper_matches_functional_step():
    shapes = [(64, 33), (129,), (16, 64)]
    p1 = [synth.make_param(s, k).cuda().requires_grad_() for k, s in enumerate(shapes)]
    p2 = [p.detach().clone() for p in p1]
    opt = Came(p1, lr=3e-3, weight_decay=0.02)
    st2 = init_came_state(p2)
    for t in range(1, 4):
        gs = [synth.make_grad(s, k, t, device="cuda") for k, s in enumerate(shapes)]
        for p, g in zip(p1, gs):
            p.grad = g.clone()
        opt.step()
        came_step(p2, gs, st2, t, lr=3e-3, weight_decay=0.02)
    torch.cuda.synchronize()
    for a, b in zip(p1, p2):
        assert torch.equal(a.detach(), b)


# one tensor of each distinct shape of the 8B list (a whole decoder layer:
# 4096-, 1024- and 14336-row matrices, the norm vectors) and the final norm
LLAMA_CAME_SAMPLE = [1, 2, 5, 7, 8, 289]


def test_llama3_8b_came_sampled():
    """The full Llama-3-8B list in the benchmark's launch configuration (one
    CameStep over all 291 tensors, bf16 gradients); the oracle recomputes the
    sampled tensors whole."""
    from oracle import came as came_oracle
    wl = synth.workload("llama3_8b_came")
    shapes = [s for _, s in wl.shapes]
    params = [synth.make_param(s, k, device="cuda") for k, s in enumerate(shapes)]
    ref_p = {k: to64(params[k]) for k in LLAMA_CAME_SAMPLE}
    ref_st = {k: came_oracle.CameState(shapes[k]) for k in LLAMA_CAME_SAMPLE}
    env = {k: np.zeros(ref_p[k].size) for k in LLAMA_CAME_SAMPLE}
    b1 = float(oracle_hp(wl.hparams).betas[0])
    grads = [torch.empty(s, dtype=wl.grad_dtype, device="cuda") for s in shapes]
    states = init_came_state(params)
    step = CameStep(params, grads, states, **wl.hparams)
    steps = 3
    for t in range(1, steps + 1):
        for k, s in enumerate(shapes):
            grads[k].copy_(synth.make_grad(s, k, t, device="cuda", std=wl.grad_std, dtype=wl.grad_dtype))
            if k in ref_p:
                m_before = ref_st[k].exp_avg.copy()
                came_oracle.step(ref_p[k], to64(grads[k]), ref_st[k], t, oracle_hp(wl.hparams))
                env[k] = b1 * env[k] + (1.0 - b1) * np.abs((ref_st[k].exp_avg - b1 * m_before) / (1.0 - b1))
        step(t)
    torch.cuda.synchronize()
    for k in LLAMA_CAME_SAMPLE:
        check(f"llama p[{k}]", to64(params[k]), ref_p[k])
        r = check_momentum(f"llama exp_avg[{k}]", to64(states[k]["exp_avg"]), ref_st[k].exp_avg, env[k], steps)
        print(f"momentum llama[{k}]: worst |dm|/bound {r[0]:.3g}, worst |dm| {r[1]:.3g}, RMS(m) {r[2]:.3g}")
    for k, p in enumerate(params):
        assert torch.isfinite(p).all(), k
