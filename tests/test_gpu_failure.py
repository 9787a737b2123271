"""Device-side failure detection without a GPU fault.

The bulk-copy kernels wait on mbarriers; every wait is bounded (about one
second).  The testing hook adafactor_debug_stall_copies(1) makes the copy
producers issue nothing, so the consumers' waits run out: the step must end
by itself, report ADAF_DEVICE_WAIT_TIMEOUT in the device status word, and
leave the CUDA context usable (the next, normal run matches the oracle)."""
import time

import pytest
import torch

from memory_efficient_optimizer_gb300 import binding, synth
from memory_efficient_optimizer_gb300.optim import AdafactorStep, init_state
from parity_util import run_parity

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    shapes = [(64, 4096), (96, 1024), (300,)]  # row-panel pass, tiled pass, 1D
    params = [synth.make_param(s, k).cuda() for k, s in enumerate(shapes)]
    grads = [synth.make_grad(s, k, 1, dtype=torch.bfloat16).cuda() for k, s in enumerate(shapes)]
    states = init_state(params)
    step = AdafactorStep(params, grads, states)
    binding.adafactor_debug_stall_copies(True)
    try:
        t0 = time.time()
        step(1)
        status = step.device_status()
        waited = time.time() - t0
    finally:
        binding.adafactor_debug_stall_copies(False)
    assert status & binding.ADAF_DEVICE_WAIT_TIMEOUT
    assert waited < 60.0
    # the next call of the same step (its descriptor table is kept on the
    # device, nothing uploaded) starts from a cleared status word
    step(2)
    assert step.device_status() == 0
    # the context is still usable: a normal run agrees with the oracle
    wl = synth.Workload("after_timeout", [(f"t{k}", s) for k, s in enumerate(shapes)], torch.bfloat16, 1e-2,
                        {}, 3)
    run, _ = run_parity(wl)
    assert run.step_fn.device_status() == 0
