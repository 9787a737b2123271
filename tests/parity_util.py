"""Shared helpers of the GPU parity tests: run the CUDA step and the float64
oracle on the same seeded inputs and compare element by element.

Tolerances (per element, after the configured number of steps):
  * the stated bar, on params and every state:  |gpu - ref| <= 1e-7 + 2e-5 |ref|;
  * a stricter check on what the steps changed:
      |(p_gpu - p0) - (p_ref - p0)| <= 2e-5 sum_t |p_ref,t - p_ref,t-1| + T ulp32(p_ref)
    (each step's update to 2e-5 of its own size, T fp32 roundings of the
    stored parameter, one per step), and the
    row/col/exp_avg_sq states at relative 2e-5 with no absolute slack beyond
    1e-30 (the eps1 scale).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from memory_efficient_optimizer_gb300 import synth
from memory_efficient_optimizer_gb300.optim import AdafactorStep, init_state

RTOL, ATOL = 2e-5, 1e-7


def oracle_hp(hparams: dict) -> oracle.HParams:
    kw = dict(hparams)
    return oracle.HParams(**kw)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def check(name, gpu, ref, rtol=RTOL, atol=ATOL):
    gpu = np.asarray(gpu, np.float64).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)) == np.all(np.isfinite(ref)), f"{name}: finiteness differs"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        k = int(np.argmax(np.where(bad, err / np.maximum(bound, 1e-300), 0)))
        raise AssertionError(f"{name}: {int(bad.sum())}/{gpu.size} outside |d| <= {atol:g} + {rtol:g}|ref|; "
                             f"worst at {k}: gpu={gpu[k]!r} ref={ref[k]!r}")
    return float(np.max(err / np.maximum(np.abs(ref), 1e-300))) if gpu.size else 0.0


def check_update(name, p_gpu, p_ref, p0, steps, abs_updates):
    d_gpu = np.asarray(p_gpu, np.float64).reshape(-1) - p0.reshape(-1)
    d_ref = np.asarray(p_ref, np.float64).reshape(-1) - p0.reshape(-1)
    ulp = np.spacing(np.abs(np.asarray(p_ref, np.float32).reshape(-1))).astype(np.float64)
    err = np.abs(d_gpu - d_ref)
    bound = RTOL * abs_updates.reshape(-1) + steps * ulp
    bad = ~(err <= bound)
    if bad.any():
        k = int(np.argmax(np.where(bad, err / np.maximum(bound, 1e-300), 0)))
        raise AssertionError(f"{name}: update differs at {int(bad.sum())} elements; worst at {k}: "
                             f"gpu delta={d_gpu[k]!r} ref delta={d_ref[k]!r}")


class Run:
    """The CUDA step over a tensor list, with persistent grad buffers (so one
    marshalled AdafactorStep serves every step, as in training)."""

    def __init__(self, shapes, hparams, grad_dtype, device="cuda", params=None, carry=True):
        self.shapes = [tuple(s) for s in shapes]
        self.hparams = dict(hparams)
        self.params = params
        self.grads = [torch.empty(s, dtype=grad_dtype, device=device) for s in self.shapes]
        self.states = init_state(self.params, beta1=self.hparams.get("beta1"), param_sq_sum=carry)
        self.step_fn = AdafactorStep(self.params, self.grads, self.states, **self.hparams)

    def step(self, t, grads):
        for buf, g in zip(self.grads, grads):
            buf.copy_(g, non_blocking=True)
        self.step_fn(t)


def run_parity(workload: synth.Workload, steps=None, sample=None, gen_device="cpu", extra_checks=None,
               carry=True):
    """Runs the CUDA step on the whole workload and the oracle on the tensors
    listed in `sample` (all when None); compares params and states."""
    steps = steps or workload.steps
    shapes = [s for _, s in workload.shapes]
    idxs = range(len(shapes)) if sample is None else sample
    hp = dict(workload.hparams)
    ohp = oracle_hp(hp)
    params = [synth.make_param(s, k, device=gen_device, std=workload.param_std).to("cuda") for k, s in
              enumerate(shapes)]
    p0 = {k: to64(params[k]) for k in idxs}
    ref_p = {k: p0[k].copy() for k in idxs}
    ref_st = {k: oracle.State(shapes[k], beta1=hp.get("beta1") is not None) for k in idxs}
    abs_upd = {k: np.zeros_like(p0[k]) for k in idxs}
    run = Run(shapes, hp, workload.grad_dtype, params=params, carry=carry)
    for t in range(1, steps + 1):
        grads = [synth.make_grad(s, k, t, device=gen_device, std=workload.grad_std, dtype=workload.grad_dtype,
                                 kind=workload.grad_kind) for k, s in enumerate(shapes)]
        host_g = {k: to64(grads[k]) for k in idxs}
        run.step(t, [g.to("cuda", non_blocking=True) for g in grads])
        del grads
        for k in idxs:
            before = ref_p[k].copy()
            oracle.step(ref_p[k], host_g[k], ref_st[k], t, ohp)
            abs_upd[k] += np.abs(ref_p[k] - before)
            del before
        del host_g
    torch.cuda.synchronize()
    assert run.step_fn.device_status() == 0, "a bounded wait inside a kernel gave up"
    report = {}
    for k in idxs:
        nm = f"{workload.name}[{k}]{shapes[k]}"
        report[k] = check(nm + ".param", to64(run.params[k]), ref_p[k])
        check_update(nm + ".param-update", to64(run.params[k]), ref_p[k], p0[k], steps, abs_upd[k])
        st, rs = run.states[k], ref_st[k]
        if rs.row is not None:
            check(nm + ".row", to64(st["exp_avg_sq_row"]), rs.row)
            check(nm + ".col", to64(st["exp_avg_sq_col"]), rs.col)
            check(nm + ".row(rel)", to64(st["exp_avg_sq_row"]), rs.row, atol=1e-30)
            check(nm + ".col(rel)", to64(st["exp_avg_sq_col"]), rs.col, atol=1e-30)
        else:
            check(nm + ".exp_avg_sq", to64(st["exp_avg_sq"]), rs.v)
            check(nm + ".exp_avg_sq(rel)", to64(st["exp_avg_sq"]), rs.v, atol=1e-30)
        if rs.exp_avg is not None:
            check(nm + ".exp_avg", to64(st["exp_avg"]), rs.exp_avg)
            scale = float(np.max(np.abs(rs.exp_avg))) if rs.exp_avg.size else 0.0
            check(nm + ".exp_avg(rel)", to64(st["exp_avg"]), rs.exp_avg, atol=1e-6 * scale)
    if extra_checks:
        extra_checks(run)
    return run, report
