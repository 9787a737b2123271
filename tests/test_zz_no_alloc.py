"""adafactor_step_noalloc: the step for callers that cannot allocate.

Some callers cannot hand the library any device memory: code that runs while a
memory pool owns the whole device and forbids cudaMalloc, code where an
allocation would synchronise the device at the wrong moment, or hosts without
an allocator of their own.  adafactor_step_noalloc() serves them with a fixed
scratch array compiled into the library.  These tests check, through the C
ABI, that it gives exactly the results of adafactor_step() with a caller
workspace on two calls in a row (the same kernels in the same order on the
same inputs, so the results must be bit-identical: a tolerance would hide a
race on the shared scratch), that a list too large for its scratch is turned
away with a clear error, that a capturing stream is turned away, and that a
bounded wait that runs out inside a kernel shows in the status word that
adafactor_noalloc_device_status() reads.  This file is named to be collected
last.
"""
import ctypes
import time

import pytest
import torch

from memory_efficient_optimizer_gb300 import binding as B
from memory_efficient_optimizer_gb300 import synth
from memory_efficient_optimizer_gb300.optim import AdafactorStep, init_state, make_hparams

SHAPES = [(600, 2100), (33, 520), (77, 13), (300,), (2, 64, 40), (1, 4096)]
HP = dict(beta1=0.9, weight_decay=0.01)


def _setup(dev):
    p_ws = [synth.make_param(s, k).to(dev) for k, s in enumerate(SHAPES)]
    p_na = [p.clone() for p in p_ws]
    g = [torch.empty(s, device=dev, dtype=torch.bfloat16) for s in SHAPES]
    st_ws = init_state(p_ws, beta1=HP["beta1"])
    st_na = init_state(p_na, beta1=HP["beta1"])
    with_ws = AdafactorStep(p_ws, g, st_ws, **HP)
    marshal = AdafactorStep(p_na, g, st_na, **HP)  # only its descriptor arrays are used
    return p_ws, p_na, g, st_ws, st_na, with_ws, marshal


@pytest.mark.gpu
def test_noalloc_step_matches_workspace_step_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    p_ws, p_na, g, st_ws, st_na, with_ws, marshal = _setup(dev)
    stream = torch.cuda.current_stream(dev)
    for t in (1, 2):
        for k, s in enumerate(SHAPES):
            g[k].copy_(synth.make_grad(s, k, t, dtype=torch.bfloat16))
        with_ws(t)
        hp = make_hparams(**HP, param_sq_sum_valid=(t > 1))
        B.adafactor_step_noalloc(marshal._tensors, marshal._states, len(SHAPES), t, hp, int(stream.cuda_stream))
        assert B.adafactor_noalloc_device_status(int(stream.cuda_stream)) == 0
        torch.cuda.synchronize()
        for k in range(len(SHAPES)):
            assert torch.equal(p_na[k], p_ws[k]), (t, k)
            for name in st_ws[k]:
                assert torch.equal(st_na[k][name], st_ws[k][name]), (t, k, name)


@pytest.mark.gpu
def test_noalloc_turns_away_a_capturing_stream():
    """Its descriptor table comes from a host buffer that lives only for the
    call, so a capture would record a copy from freed memory: the call must
    return ADAF_ERR_UNSUPPORTED and enqueue nothing."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    p_ws, p_na, g, st_ws, st_na, with_ws, marshal = _setup(dev)
    for k, s in enumerate(SHAPES):
        g[k].copy_(synth.make_grad(s, k, 1, dtype=torch.bfloat16))
    before = [p.clone() for p in p_na]
    side = torch.cuda.Stream(dev)
    hp = make_hparams(**HP)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        rc = B.load().adafactor_step_noalloc(marshal._tensors, marshal._states, len(SHAPES), 1, ctypes.byref(hp),
                                             ctypes.c_void_p(side.cuda_stream))
    assert rc == B.ADAF_ERR_UNSUPPORTED
    assert "capturing" in B.adafactor_last_error()
    torch.cuda.synchronize()
    for k in range(len(SHAPES)):
        assert torch.equal(p_na[k], before[k])


@pytest.mark.gpu
def test_noalloc_status_word_reports_a_wait_that_ran_out():
    """With the copy producers stalled (the library's testing hook), the
    bulk-copy apply's bounded waits run out; the step ends by itself and the
    status word of the scratch array says so.  The next normal call resets it."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes = [(64, 4096), (300,)]
    params = [synth.make_param(s, k).to(dev) for k, s in enumerate(shapes)]
    grads = [synth.make_grad(s, k, 1, dtype=torch.bfloat16).to(dev) for k, s in enumerate(shapes)]
    states = init_state(params)
    marshal = AdafactorStep(params, grads, states)
    stream = int(torch.cuda.current_stream(dev).cuda_stream)
    hp = make_hparams()
    B.adafactor_debug_stall_copies(True)
    try:
        t0 = time.time()
        B.adafactor_step_noalloc(marshal._tensors, marshal._states, len(shapes), 1, hp, stream)
        status = B.adafactor_noalloc_device_status(stream)
        waited = time.time() - t0
    finally:
        B.adafactor_debug_stall_copies(False)
    assert status & B.ADAF_DEVICE_WAIT_TIMEOUT
    assert waited < 60.0
    B.adafactor_step_noalloc(marshal._tensors, marshal._states, len(shapes), 2, hp, stream)
    assert B.adafactor_noalloc_device_status(stream) == 0


def test_noalloc_rejects_a_list_beyond_its_scratch():
    """Llama-3-8B needs ~254 MB of scratch: more than the fixed area, so the
    call fails before touching CUDA, naming both sizes."""
    shapes = [s for _, s in synth.llama3_8b_shapes()]
    n = len(shapes)
    ts = (B.adaf_tensor * n)()
    ss = (B.adaf_state * n)()
    for k, s in enumerate(shapes):
        ts[k].param = ts[k].grad = 1 << 20
        ts[k].grad_dtype = B.ADAF_BFLOAT16
        ts[k].ndim = len(s)
        for d, v in enumerate(s):
            ts[k].shape[d] = v
    hp = B.adafactor_default_hparams()
    rc = B.load().adafactor_step_noalloc(ts, ss, n, 1, ctypes.byref(hp), None)
    assert rc == B.ADAF_ERR_WORKSPACE_TOO_SMALL
    msg = B.adafactor_last_error()
    need = B.adafactor_workspace_size(ts, n)
    assert str(need) in msg and str(64 << 20) in msg
