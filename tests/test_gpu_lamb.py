"""GPU parity of the LAMB step (include/lamb.h) against the float64 LAMB
oracle, element by element on the same seeded inputs.

Bar (per element, after the steps): |gpu - ref| <= 1e-7 + 2e-5 |ref| on the
parameters and both moments, and the trust ratios to relative 2e-5.  The GPU
keeps fp32 state and fp32 element arithmetic with float64 norms; the oracle is
float64 throughout.
"""
import numpy as np
import pytest
import torch

from memory_efficient_optimizer_gb300 import synth
from memory_efficient_optimizer_gb300.lamb import Lamb, LambStep, init_lamb_state, lamb_step
from parity_util import check, check_update, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from memory_efficient_optimizer_gb300 import build
    from oracle import lamb as lamb_oracle
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lamb_oracle.build()


def oracle_hp(hp):
    from oracle.lamb import LambHParams
    return LambHParams(**hp)


# flat sizes around the 4-value loads and the 8192-value work units, one
# empty tensor, 2-D / 3-D views (LAMB treats every tensor as one flat layer)
SHAPES = [(1,), (3,), (4,), (5,), (0,), (7, 13), (8192,), (8193,), (3, 8197), (100, 257), (2, 64, 64),
          (40000,), (1000, 130), (8191,), (16384 + 4,)]
HPARAMS = [
    dict(),
    dict(weight_decay=0.01),
    dict(lr=5e-3, bias_correction=False),
    dict(lr=0.02, betas=(0.5, 0.9), eps=1e-8, weight_decay=0.1),
]


def run_lamb(shapes, hp, grad_dtype, steps, params=None, grad_std=1e-3, zero_grad_tensor=None):
    """Runs the CUDA step and the oracle side by side; returns (gpu, ref) lists."""
    from oracle import lamb as lamb_oracle
    dev = "cuda"
    if params is None:
        params = [synth.make_param(s, k).to(dev) for k, s in enumerate(shapes)]
    ref_p = [to64(p) for p in params]
    p0 = [x.copy() for x in ref_p]
    abs_upd = [np.zeros(x.size) for x in ref_p]
    ref_st = [lamb_oracle.LambState(s) for s in shapes]
    grads = [torch.empty(s, dtype=grad_dtype, device=dev) for s in shapes]
    states = init_lamb_state(params)
    step = LambStep(params, grads, states, **hp)
    trust_ref = []
    for t in range(1, steps + 1):
        trust_ref = []
        for k, s in enumerate(shapes):
            g = synth.make_grad(s, k, t, std=grad_std, dtype=grad_dtype)
            if zero_grad_tensor == k:
                g.zero_()
            grads[k].copy_(g)
            before = ref_p[k].copy()
            trust_ref.append(lamb_oracle.step(ref_p[k], to64(g), ref_st[k], t, oracle_hp(hp)))
            abs_upd[k] += np.abs(ref_p[k] - before).reshape(-1)
        step(t)
    torch.cuda.synchronize()
    return params, states, ref_p, ref_st, step.trust_ratios(), trust_ref, (p0, abs_upd, steps)


def compare(params, states, ref_p, ref_st, trust, trust_ref, upd=None, tag=""):
    """The stated bar on p and both moments (exp_avg_sq relative only: it has
    no cancellation), the trust ratios, and each parameter's accumulated
    change to 2e-5 of the sum of its per-step updates."""
    for k in range(len(params)):
        check(f"{tag}p[{k}]", to64(params[k]), ref_p[k])
        check(f"{tag}exp_avg[{k}]", to64(states[k]["exp_avg"]), ref_st[k].exp_avg, atol=1e-10)
        check(f"{tag}exp_avg_sq[{k}]", to64(states[k]["exp_avg_sq"]), ref_st[k].exp_avg_sq, atol=1e-30)
        if upd is not None:
            p0, abs_upd, steps = upd
            check_update(f"{tag}update[{k}]", to64(params[k]), ref_p[k], p0[k], steps, abs_upd[k])
    np.testing.assert_allclose(trust, trust_ref, rtol=2e-5)


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("hp", HPARAMS)
def test_lamb_small_shapes(hp, grad_dtype):
    out = run_lamb(SHAPES, hp, grad_dtype, steps=8)
    compare(*out)


def test_lamb_zero_gradient_tensor_and_zero_param():
    """A tensor whose gradient is always 0 (r = wd p: pure decay) and one
    whose parameter is 0 (trust ratio 1)."""
    shapes = [(300, 7), (513,), (64, 64)]
    params = [synth.make_param(s, k).cuda() for k, s in enumerate(shapes)]
    params[1].zero_()
    out = run_lamb(shapes, dict(weight_decay=0.05, lr=0.01), torch.float32, steps=4, params=params,
                   zero_grad_tensor=0)
    compare(*out)


def test_lamb_misaligned_views_take_the_scalar_path():
    shapes = [(1000,), (37, 41), (9000,)]
    bufs = [torch.zeros(int(np.prod(s)) + 1, device="cuda") for s in shapes]
    params = [b[1:].view(s) for b, s in zip(bufs, shapes)]
    for k, (p, s) in enumerate(zip(params, shapes)):
        p.copy_(synth.make_param(s, k))
    out = run_lamb(shapes, dict(weight_decay=0.01), torch.bfloat16, steps=5, params=params)
    compare(*out)


def test_lamb_bitwise_deterministic():
    shapes = [(1000, 130), (40000,), (7, 13)]
    res = []
    for _ in range(2):
        params, states, *_rest = run_lamb(shapes, dict(weight_decay=0.01), torch.bfloat16, steps=3)
        res.append([p.clone() for p in params] + [st["exp_avg"].clone() for st in states])
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_lamb_optimizer_wrapper_matches_functional_step():
    shapes = [(64, 33), (129,)]
    p1 = [synth.make_param(s, k).cuda().requires_grad_() for k, s in enumerate(shapes)]
    p2 = [p.detach().clone() for p in p1]
    opt = Lamb(p1, lr=3e-3, weight_decay=0.02)
    st2 = init_lamb_state(p2)
    for t in range(1, 4):
        gs = [synth.make_grad(s, k, t, device="cuda") for k, s in enumerate(shapes)]
        for p, g in zip(p1, gs):
            p.grad = g.clone()
        opt.step()
        lamb_step(p2, gs, st2, t, lr=3e-3, weight_decay=0.02)
    torch.cuda.synchronize()
    for a, b in zip(p1, p2):
        assert torch.equal(a.detach(), b)


# the first tensors of the list (embedding and a whole decoder layer) and the
# final norm; lm_head (the same shape as the embedding) is left out for time
LLAMA_LAMB_SAMPLE = [0, 1, 2, 5, 7, 8, 289]


def test_llama3_8b_lamb_sampled():
    """The full Llama-3-8B list in the benchmark's launch configuration (one
    LambStep over all 291 tensors, bf16 gradients); the oracle recomputes the
    sampled tensors whole (LAMB norms are per tensor)."""
    from oracle import lamb as lamb_oracle
    wl = synth.workload("llama3_8b_lamb")
    shapes = [s for _, s in wl.shapes]
    params = [synth.make_param(s, k, device="cuda") for k, s in enumerate(shapes)]
    ref_p = {k: to64(params[k]) for k in LLAMA_LAMB_SAMPLE}
    ref_st = {k: lamb_oracle.LambState(shapes[k]) for k in LLAMA_LAMB_SAMPLE}
    grads = [torch.empty(s, dtype=wl.grad_dtype, device="cuda") for s in shapes]
    states = init_lamb_state(params)
    step = LambStep(params, grads, states, **wl.hparams)
    steps = 3
    for t in range(1, steps + 1):
        trust_ref = {}
        for k, s in enumerate(shapes):
            grads[k].copy_(synth.make_grad(s, k, t, device="cuda", std=wl.grad_std, dtype=wl.grad_dtype))
            if k in ref_p:
                trust_ref[k] = lamb_oracle.step(ref_p[k], to64(grads[k]), ref_st[k], t, oracle_hp(wl.hparams))
        step(t)
    torch.cuda.synchronize()
    trust = step.trust_ratios()
    for k in LLAMA_LAMB_SAMPLE:
        check(f"llama p[{k}]", to64(params[k]), ref_p[k])
        check(f"llama exp_avg[{k}]", to64(states[k]["exp_avg"]), ref_st[k].exp_avg, atol=1e-10)
        assert trust[k] == pytest.approx(trust_ref[k], rel=2e-5)
    assert all(np.isfinite(trust)) and all(x > 0 for x in trust)
