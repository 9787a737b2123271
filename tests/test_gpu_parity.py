"""GPU parity: the CUDA step against the float64 oracle on the same seeded
inputs, element by element (tolerances in parity_util).

Workloads (memory_efficient_optimizer_gb300.synth): the 256x512 + 512 case,
one Llama-3-8B decoder layer, the edge-shape sweep with 2,000 small matrices,
and the full Llama-3-8B list in both hyper-parameter settings, where the GPU
steps all 291 tensors in the benchmark's launch configuration and the oracle
recomputes a sample of them (one tensor of each shape, the first and last
tensors of the list included).
"""
import numpy as np
import pytest
import torch

from memory_efficient_optimizer_gb300 import synth
from memory_efficient_optimizer_gb300.optim import AdafactorStep, init_state
from parity_util import Run, check, run_parity, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import oracle
    from memory_efficient_optimizer_gb300 import build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    oracle.build()


def test_tiny_workload_10_steps():
    run_parity(synth.workload("tiny"))


def test_llama_layer_10_steps():
    run_parity(synth.workload("llama_layer"), gen_device="cuda")


def test_edge_sweep_10_steps():
    run_parity(synth.workload("edge"), gen_device="cuda")


# one tensor of every distinct shape of the 8B list, plus the first and last
LLAMA_SAMPLE = [0, 1, 2, 5, 7, 8, 289, 290]


def _invariants(run):
    # mean(row) = mean(col) per factored tensor (both EMAs of the grand mean)
    for k, st in enumerate(run.states):
        if "exp_avg_sq_row" in st:
            r = st["exp_avg_sq_row"].double().mean().item()
            c = st["exp_avg_sq_col"].double().mean().item()
            assert abs(r - c) <= 1e-5 * abs(r), (k, r, c)
        assert torch.isfinite(run.params[k]).all()


def test_llama3_8b_defaults_sampled():
    run_parity(synth.workload("llama3_8b"), sample=[1, 2, 5, 7, 8, 289, 290], gen_device="cuda",
               extra_checks=_invariants)


def test_llama3_8b_beta1_student_t_sampled():
    run_parity(synth.workload("llama3_8b_beta1"), sample=[1, 2, 5, 7, 8, 289, 290], gen_device="cuda",
               extra_checks=_invariants)


SMALL_SHAPES = [(1, 1), (2, 3), (3, 2), (1, 5), (5, 1), (2, 2, 3), (4,), (), (600, 2100), (257, 1025),
                (3, 4097), (1000, 1032), (2, 3, 520, 264), (7, 1, 9), (1, 65536), (9000,),
                # flat walk over whole rows (W <= 1024, not a multiple of 8): several
                # staged chunks per tile and a ragged last chunk, 1..8-lane row segments
                (700, 33), (300, 1023), (513, 7), (260, 1), (1030, 3),
                # 2, 4, 8 and 16 columns per lane in registers (W <= 512), and the
                # staged form just above
                (130, 100), (91, 200), (50, 512), (40, 513), (33, 32), (17, 16),
                # bf16: fused row-chunk pass, 8-warp configuration (2048 <= W <= 4096): a
                # one-lane last column group, two chunks with a ragged one, B = 2 slices
                (300, 2056), (2, 130, 4096),
                # bf16: 14-warp configuration (4096 < W <= 14336): ragged chunks and
                # sub-panels, the widest row, chunks of one sub-panel; W = 16384, 16392
                # and 2040 stay tiled
                (131, 4104), (67, 14336), (3, 16384), (5, 16392), (9, 2040), (7, 9000), (129, 5000),
                (1, 8192)]
FLAGS = [
    dict(),
    dict(beta1=0.9, weight_decay=0.1),
    dict(warmup_init=True),
    dict(clip_threshold=0.05),
    dict(scale_parameter=False, eps=(1e-3, 1e-2)),
    dict(lr=0.02, relative_step=False, scale_parameter=False, beta1=0.5, weight_decay=0.01),
    dict(lr=0.01, relative_step=False, decay_rate=-0.5),
]


@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("flags", FLAGS)
def test_small_shapes_all_flags(flags, grad_dtype):
    wl = synth.Workload("small", [(f"t{k}", s) for k, s in enumerate(SMALL_SHAPES)], grad_dtype, 0.5,
                        flags, 10, grad_kind="student_t_zero_rows", param_std=0.3)
    run_parity(wl)


@pytest.mark.parametrize("carry,offset", [(True, "both"), (False, "both"), (False, "params"), (True, "grads")])
def test_misaligned_views_take_the_elementwise_path(carry, offset):
    """Params and/or grads offset by one element from a 16-byte boundary
    cannot use the vector kernels or the 4-value loads of the flat walk;
    results must not change."""
    shapes = [(64, 1024), (33, 520), (100,), (20, 2048), (9, 4104), (300, 77)]
    hp = dict(beta1=0.9)
    import oracle
    from parity_util import oracle_hp
    po = 1 if offset in ("both", "params") else 0
    go = 1 if offset in ("both", "grads") else 0
    bufs_p = [torch.zeros(int(np.prod(s)) + 1, device="cuda") for s in shapes]
    params = [b[po:po + int(np.prod(s))].view(s) for b, s in zip(bufs_p, shapes)]
    for k, (p, s) in enumerate(zip(params, shapes)):
        p.copy_(synth.make_param(s, k))
    p0 = [to64(p) for p in params]
    refs = [x.copy() for x in p0]
    rst = [oracle.State(s, True) for s in shapes]
    gbufs = [torch.zeros(int(np.prod(s)) + 1, device="cuda", dtype=torch.bfloat16) for s in shapes]
    grads = [b[go:go + int(np.prod(s))].view(s) for b, s in zip(gbufs, shapes)]
    states = init_state(params, beta1=0.9, param_sq_sum=carry)
    step = AdafactorStep(params, grads, states, **hp)
    for t in range(1, 6):
        for k, s in enumerate(shapes):
            grads[k].copy_(synth.make_grad(s, k, t, dtype=torch.bfloat16))
            oracle.step(refs[k], to64(grads[k]), rst[k], t, oracle_hp(hp))
        step(t)
    torch.cuda.synchronize()
    for k in range(len(shapes)):
        check(f"misaligned[{k}]", to64(params[k]), refs[k])


def _run_steps(shapes, hp, t0, t1, params, states, grad_dtype=torch.float32):
    grads = [torch.empty(s, device="cuda", dtype=grad_dtype) for s in shapes]
    step = AdafactorStep(params, grads, states, **hp)
    for t in range(t0, t1):
        for k, s in enumerate(shapes):
            grads[k].copy_(synth.make_grad(s, k, t, dtype=grad_dtype))
        step(t)
    torch.cuda.synchronize()


@pytest.mark.parametrize("shapes,grad_dtype", [
    ([(600, 2100), (300,), (8, 64, 40)], torch.float32),
    ([(300, 2056), (131, 4104), (1000, 1032), (300,)], torch.bfloat16),  # fused, fused wide, tiled
])
def test_bitwise_deterministic_and_resumable(shapes, grad_dtype):
    """Two runs are bit-identical (fixed-order reductions, no atomics), and 5
    steps + copying params/state out and back + 5 steps equals 10 steps."""
    hp = dict(beta1=0.9, weight_decay=0.01)

    def fresh():
        params = [synth.make_param(s, k).cuda() for k, s in enumerate(shapes)]
        return params, init_state(params, beta1=0.9, param_sq_sum=False)

    pa, sa = fresh()
    _run_steps(shapes, hp, 1, 11, pa, sa, grad_dtype)
    pb, sb = fresh()
    _run_steps(shapes, hp, 1, 11, pb, sb, grad_dtype)
    for x, y in zip(pa, pb):
        assert torch.equal(x, y)
    pc, sc = fresh()
    _run_steps(shapes, hp, 1, 6, pc, sc, grad_dtype)
    saved_p = [p.cpu().clone() for p in pc]
    saved_s = [{k: v.cpu().clone() for k, v in st.items()} for st in sc]
    pd = [p.cuda() for p in saved_p]
    sd = [{k: v.cuda() for k, v in st.items()} for st in saved_s]
    _run_steps(shapes, hp, 6, 11, pd, sd, grad_dtype)
    for x, y in zip(pa, pd):
        assert torch.equal(x, y)
    for x, y in zip(sa, sd):
        for k in x:
            assert torch.equal(x[k], y[k]), k


def test_guard_bands_untouched():
    """Every tensor lives inside a larger buffer filled with a sentinel; after
    10 steps the bytes around each tensor are unchanged."""
    shapes = [(517, 1029), (1024, 1032), (77,), (3, 5, 7), (130, 2056), (67, 4104)]
    pad = 4096
    hp = dict(beta1=0.9)

    def guarded(shape, dtype, fill):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), fill, device="cuda", dtype=dtype)
        return buf, buf[pad:pad + n].view(shape)

    pb = [guarded(s, torch.float32, 7.0) for s in shapes]
    gb = [guarded(s, torch.bfloat16, 3.0) for s in shapes]
    params = [v for _, v in pb]
    grads = [v for _, v in gb]
    for k, (p, s) in enumerate(zip(params, shapes)):
        p.copy_(synth.make_param(s, k))
    states = init_state(params, beta1=0.9)
    sbufs = []
    for st in states:
        for name in list(st):
            buf, view = guarded(tuple(st[name].shape), st[name].dtype, -5.0)
            view.zero_()
            st[name] = view
            sbufs.append(buf)
    step = AdafactorStep(params, grads, states, **hp)
    ws = step.workspace
    for t in range(1, 11):
        for k, s in enumerate(shapes):
            grads[k].copy_(synth.make_grad(s, k, t, dtype=torch.bfloat16))
        step(t)
    torch.cuda.synchronize()
    for buf, fill in [(b, 7.0) for b, _ in pb] + [(b, 3.0) for b, _ in gb] + [(b, -5.0) for b in sbufs]:
        assert torch.all(buf[:pad] == fill) and torch.all(buf[-pad:] == fill)
    assert ws is step.workspace


def test_optimizer_wrapper_matches_functional_step():
    import memory_efficient_optimizer_gb300 as meo
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(64, 128), torch.nn.ReLU(), torch.nn.Linear(128, 8)).cuda()
    ref = [p.detach().clone() for p in model.parameters()]
    ref_states = init_state(ref, beta1=0.9, param_sq_sum=False)
    opt = meo.Adafactor(model.parameters(), beta1=0.9)
    for t in range(1, 6):
        x = torch.randn(32, 64, device="cuda")
        loss = model(x).square().mean()
        opt.zero_grad()
        loss.backward()
        grads = [p.grad.detach().clone() for p in model.parameters()]
        opt.step()
        meo.adafactor_step(ref, grads, ref_states, t, beta1=0.9)
    torch.cuda.synchronize()
    for p, r in zip(model.parameters(), ref):
        check("wrapper", to64(p), to64(r), rtol=1e-6, atol=1e-9)


def test_native_library_is_loaded():
    import os
    from memory_efficient_optimizer_gb300 import binding
    lib = binding.load()
    maps = open("/proc/self/maps").read()
    assert os.path.realpath(binding.library_path()) in maps
    assert lib is not None


def test_more_tensors_than_one_launch_group():
    """4,500 tensors: more than one launch group (4,096 tensors share one
    launch's prefix array), in every class (vector, element-wise, fused, 1D),
    against the oracle."""
    rng = np.random.default_rng(4500)
    kinds = [(3, 5), (16, 24), (2, 2056), (7,), (9, 1)]
    shapes = [kinds[k % len(kinds)] if k % 7 else (int(rng.integers(1, 9)), int(rng.integers(1, 40)))
              for k in range(4500)]
    wl = synth.Workload("groups", [(f"t{k}", s) for k, s in enumerate(shapes)], torch.bfloat16, 1e-2,
                        dict(beta1=0.9, weight_decay=0.01), 3)
    run_parity(wl)


def test_two_step_objects_alternating_share_kept_tables():
    """Two AdafactorStep objects over the same params and states, each with its
    own gradient buffers, called in turn (the double-buffered upload pattern
    of a training loop): every call after the first two reads a descriptor
    table kept on the device.  Results must equal the oracle's, and a third
    object over a different list in between must not disturb them."""
    import oracle
    from parity_util import oracle_hp
    shapes = [(300, 2056), (130, 100), (17, 16), (513,), (2, 40, 600)]
    hp = dict(beta1=0.9)
    params = [synth.make_param(s, k).cuda() for k, s in enumerate(shapes)]
    refs = [to64(p) for p in params]
    rst = [oracle.State(s, True) for s in shapes]
    states = init_state(params, beta1=0.9)
    bufs = [[torch.empty(s, device="cuda", dtype=torch.bfloat16) for s in shapes] for _ in range(2)]
    steps = [AdafactorStep(params, bufs[b], states, **hp) for b in range(2)]
    other_p = [synth.make_param((64, 64), 99).cuda()]
    other = AdafactorStep(other_p, [torch.zeros(64, 64, device="cuda")], init_state(other_p))
    for t in range(1, 7):
        b = t % 2
        for k, s in enumerate(shapes):
            bufs[b][k].copy_(synth.make_grad(s, k, t, dtype=torch.bfloat16))
            oracle.step(refs[k], to64(bufs[b][k]), rst[k], t, oracle_hp(hp))
        steps[b](t)
        if t == 3:
            other(1)
    torch.cuda.synchronize()
    assert steps[0].device_status() == 0 and steps[1].device_status() == 0
    for k in range(len(shapes)):
        check(f"alternating[{k}]", to64(params[k]), refs[k])


def test_wide_chunks_run_back_to_back_in_one_cta():
    """More wide-class chunks than one CTA per SM: 400 bf16 matrices of 3 or 5
    rows of 4104 or 9000 values (one chunk each, of 2 or 3 sub-panels), so
    most CTAs of the wide pass run two or three chunks in a row and carry the
    mbarrier phases and share buffers of the split form from one chunk to the
    next, against the oracle; with and without sum(p^2) recomputed in pass 1."""
    kinds = [(3, 4104), (5, 9000), (3, 9000), (5, 4104)]
    shapes = [kinds[k % len(kinds)] for k in range(400)]
    for hp in (dict(), dict(beta1=0.9, weight_decay=0.01)):
        wl = synth.Workload("wide_many", [(f"t{k}", s) for k, s in enumerate(shapes)], torch.bfloat16, 1e-2,
                            hp, 4)
        run_parity(wl)
