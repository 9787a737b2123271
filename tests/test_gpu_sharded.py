"""Row-sharded step (the distributed step of the Colossal-AI distributed-
optimizer article, Step 4) against the float64 oracle on the whole tensors.

Each tensor is split by rows into `nranks` contiguous blocks of uneven size
(elements for ndim < 2).  The ranks run one after another on one GPU; the
all-reduce between the library calls is emulated by summing the ranks'
exchange buffers on the device.  After the steps, the gathered parameters and
row states, and every rank's column state, must match the oracle run on the
unsharded tensors within the stated bar, and the column states must be
identical on all ranks."""
import numpy as np
import pytest
import torch

import oracle
from memory_efficient_optimizer_gb300 import synth
from memory_efficient_optimizer_gb300.optim import AdafactorShardStep, init_state
from parity_util import check, check_update, oracle_hp, to64

SHAPES = [(300, 2056), (131, 4104), (1000, 1032), (257, 1025), (2, 130, 4096), (3, 5, 7), (9000,), (600,)]
FLAGS = [
    dict(),
    dict(beta1=0.9, weight_decay=0.1),
    dict(lr=0.01, relative_step=False, scale_parameter=False, beta1=0.5),
]


def split(n, nranks):
    """Uneven contiguous blocks [b_r, b_{r+1}) of range(n), each non-empty."""
    cuts = [0] + [max(r, min(n - nranks + r, int(round(n * f)))) for r, f in
                  zip(range(1, nranks), np.linspace(0, 1, nranks + 1)[1:-1] ** 1.3)] + [n]
    assert all(b > a for a, b in zip(cuts, cuts[1:])), cuts
    return cuts


def shard(t, cuts, r):
    """Rank r's block of t: rows [cuts[r], cuts[r+1]) of every slice (elements for ndim < 2)."""
    if t.dim() >= 2:
        return t[..., cuts[r]:cuts[r + 1], :].contiguous()
    return t[cuts[r]:cuts[r + 1]].contiguous()


def gather(parts):
    return torch.cat(parts, dim=-2 if parts[0].dim() >= 2 else 0)


@pytest.mark.gpu
@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("nranks", [1, 3])
@pytest.mark.parametrize("flags", FLAGS)
def test_row_sharded_step_matches_oracle(flags, nranks, grad_dtype):
    steps = 6
    hp = dict(flags)
    ohp = oracle_hp(hp)
    beta1 = hp.get("beta1")
    rows = [s[-2] if len(s) >= 2 else s[0] for s in SHAPES]
    cuts = [split(h, nranks) for h in rows]
    full_p = [synth.make_param(s, k, std=0.3) for k, s in enumerate(SHAPES)]
    p0 = [to64(p) for p in full_p]
    ref_p = [x.copy() for x in p0]
    ref_st = [oracle.State(s, beta1=beta1 is not None) for s in SHAPES]
    abs_upd = [np.zeros_like(x) for x in p0]
    ranks = []
    for r in range(nranks):
        params = [shard(p, cuts[k], r).cuda() for k, p in enumerate(full_p)]
        grads = [torch.empty(p.shape, dtype=grad_dtype, device="cuda") for p in params]
        states = init_state(params, beta1=beta1)
        ranks.append(AdafactorShardStep(params, grads, states, rows, **hp))
    for t in range(1, steps + 1):
        full_g = [synth.make_grad(s, k, t, std=0.01, dtype=grad_dtype, kind="student_t_zero_rows")
                  for k, s in enumerate(SHAPES)]
        for r, st in enumerate(ranks):
            for k, g in enumerate(full_g):
                st.grads[k].copy_(shard(g, cuts[k], r))
        for k, g in enumerate(full_g):
            before = ref_p[k].copy()
            oracle.step(ref_p[k], to64(g), ref_st[k], t, ohp)
            abs_upd[k] += np.abs(ref_p[k] - before)
        # begin on every rank, sum exchange round 1, middle, sum exchange round 2, end
        for st in ranks:
            st.begin(t)
        tot = sum(st.round1 for st in ranks)
        for st in ranks:
            st.round1.copy_(tot)
        for st in ranks:
            st.middle(t)
        tot = sum(st.round2 for st in ranks)
        for st in ranks:
            st.round2.copy_(tot)
        for st in ranks:
            st.end(t)
    torch.cuda.synchronize()
    for st in ranks:
        assert st.device_status() == 0
    for k, s in enumerate(SHAPES):
        nm = f"shard{nranks}[{k}]{s}"
        got = to64(gather([st.params[k] for st in ranks]))
        check(nm + ".param", got, ref_p[k])
        check_update(nm + ".param-update", got, ref_p[k], p0[k], steps, abs_upd[k])
        rs = ref_st[k]
        if rs.row is not None:
            row = to64(torch.cat([st.states[k]["exp_avg_sq_row"] for st in ranks], dim=-1))  # [..., rows]
            check(nm + ".row", row, rs.row, atol=1e-30)
            col0 = ranks[0].states[k]["exp_avg_sq_col"]
            for st in ranks[1:]:
                assert torch.equal(st.states[k]["exp_avg_sq_col"], col0), nm + ": column states differ between ranks"
            check(nm + ".col", to64(col0), rs.col, atol=1e-30)
        else:
            v = to64(gather([st.states[k]["exp_avg_sq"] for st in ranks]))
            check(nm + ".exp_avg_sq", v, rs.v, atol=1e-30)
        if rs.exp_avg is not None:
            m = to64(gather([st.states[k]["exp_avg"] for st in ranks]))
            check(nm + ".exp_avg", m, rs.exp_avg)


@pytest.mark.gpu
def test_one_shard_equals_the_single_call_step():
    """With one rank and no collective the three calls compute what
    adafactor_step() computes (sums in another order: compared at the bar)."""
    from memory_efficient_optimizer_gb300.optim import AdafactorStep
    shapes = [(300, 2056), (1000, 1032), (9000,)]
    params_a = [synth.make_param(s, k).cuda() for k, s in enumerate(shapes)]
    params_b = [p.clone() for p in params_a]
    grads = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in shapes]
    sa, sb = init_state(params_a), init_state(params_b)
    one = AdafactorStep(params_a, grads, sa)
    sh = AdafactorShardStep(params_b, grads, sb, [s[-2] if len(s) >= 2 else s[0] for s in shapes])
    for t in range(1, 6):
        for k, s in enumerate(shapes):
            grads[k].copy_(synth.make_grad(s, k, t, dtype=torch.bfloat16))
        one(t)
        sh(t)
    torch.cuda.synchronize()
    for k in range(len(shapes)):
        check(f"one-shard[{k}]", to64(params_b[k]), to64(params_a[k]))
