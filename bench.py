#!/usr/bin/env python3
"""Benchmark of the GB300 Adafactor step on Llama-3-8B-shaped parameters.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3_8b|llama3_8b_beta1|llama_layer|edge|tiny]

One step = one full Adafactor step (all kernels of the launch sequence) over
the whole tensor list of the workload, with synthetic inputs resident in HBM
(48 GB for Llama-3-8B: fp32 params, bf16 grads; far larger than the 129 MB
L2, so no flush is needed between steps).  Rank 0 prints one JSON line.

The ``*_lamb`` and ``*_came`` workloads run the multi-tensor LAMB
(include/lamb.h) or CAME (include/came.h) step instead, with the same JSON
line (metrics LAMB_METRIC, CAME_METRIC).

--impl reference times the float64 CPU oracle (single thread) on a bounded
sample of the same workload per step.  With --gpus N > 1 every rank runs an
independent replica of the step on its own GPU (the step has no collective);
value = total params/s over all ranks with the slowest rank's time.  Started
without torchrun, ``--gpus N`` re-launches itself under
``python -m torch.distributed.run --nproc-per-node N`` (127.0.0.1, a free
port); under torchrun, WORLD_SIZE must equal N.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import mmap
import re
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from memory_efficient_optimizer_gb300 import binding, synth  # noqa: E402
from memory_efficient_optimizer_gb300.came import CameStep, init_came_state  # noqa: E402
from memory_efficient_optimizer_gb300.lamb import LambStep, init_lamb_state  # noqa: E402
from memory_efficient_optimizer_gb300.optim import AdafactorShardStep, AdafactorStep, init_state  # noqa: E402

METRIC = "Adafactor step params/sec and effective HBM GB/s (% of 8 TB/s), Llama-3-8B shapes"
LAMB_METRIC = "LAMB step params/sec and effective HBM GB/s, Llama-3-8B shapes"
CAME_METRIC = "CAME step params/sec and effective HBM GB/s, Llama-3-8B shapes"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
KERNEL_SRC = os.path.join(ROOT, "memory_efficient_optimizer_gb300", "csrc", "adafactor_kernels.cu")
KERNEL_HDR = os.path.join(ROOT, "memory_efficient_optimizer_gb300", "csrc", "adafactor_internal.h")
PANEL_HDR = os.path.join(ROOT, "memory_efficient_optimizer_gb300", "csrc", "row_panel.cuh")
LAMB_SRC = os.path.join(ROOT, "memory_efficient_optimizer_gb300", "csrc", "lamb.cu")
LAMB_HDR = os.path.join(ROOT, "include", "lamb.h")
CAME_SRC = os.path.join(ROOT, "memory_efficient_optimizer_gb300", "csrc", "came.cu")
CAME_HDR = os.path.join(ROOT, "include", "came.h")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return int(sk.getsockname()[1])


def torchrun_cmd(nproc: int, script: str, argv, port: int):
    """The single-node torch.distributed.run command that starts `script`
    once per rank (one rank per GPU)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={int(nproc)}",
            "--master-addr", "127.0.0.1", "--master-port", str(int(port)), script, *argv]


def launch_ranks(nproc: int, script: str, argv) -> int:
    """Runs `script` with `argv` as nproc ranks under torch.distributed.run;
    returns the launcher's exit status (non-zero if any rank failed)."""
    return subprocess.call(torchrun_cmd(nproc, script, list(argv), free_port()))


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (max) of a per-rank timing; identity at N = 1."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(n_params: int, world: int, ms_per_step: float) -> float:
    """Whole-job params/s: every rank steps its own full replica."""
    return world * n_params / (ms_per_step / 1e3)


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        for key in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if key in peaks and peaks[key]:
                return float(peaks[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# Classes whose pass 1 also forms sum(u^2) (g read twice per step, not three
# times): the row-panel pass and the fused flat pass.
FUSED_CLASSES = ("rows_bf16", "wide_bf16", "flat_bf16", "flat_f32")


def tensor_class(shape, grad_bytes):
    """The library's tensor class of a contiguous, 256-byte aligned tensor."""
    if len(shape) < 2:
        return "1d"
    w = int(shape[-1])
    if w <= 1024:  # whole rows per tile (every tile start 4-value aligned here)
        return "flat_" + ("bf16" if grad_bytes == 2 else "f32")
    if w % 8:
        return "elem_" + ("bf16" if grad_bytes == 2 else "f32")
    if grad_bytes == 2 and 2048 <= w <= 4096:
        return "rows_bf16"
    if grad_bytes == 2 and 4096 < w <= 14336:
        return "wide_bf16"
    return "vec_" + ("bf16" if grad_bytes == 2 else "f32")


def first_moment_bytes(n, beta1, q8, group_scales=0):
    """Read + write bytes of the first moment of n values: fp32 exp_avg, or
    int8 codes plus one fp32 scale per group."""
    if not beta1:
        return 0
    return 2 * (n + 4 * group_scales) if q8 else 8 * n


def algorithmic_bytes(shapes, grad_bytes, beta1, q8=False):
    """Minimum bytes per step as the roofline of the method counts them (three
    reads of g: the statistics pass, the sum(u^2) pass and the update; p read +
    write; exp_avg read + write with beta1; the second-moment state read +
    write), the minimum of this implementation (the fused pass folds the
    sum(u^2) pass into the statistics pass for "rows" tensors, so g is read
    twice there), and the minimum per streaming launch slot ("k_apply[rows_bf16]",
    ...).  Returns (per step as defined, per step of this implementation, slots)."""
    step = impl = 0
    slots = {}
    for _, s in shapes:
        n = 1
        for d in s:
            n *= int(d)
        cls = tensor_class(s, grad_bytes)
        if len(s) >= 2:
            lead = n // (int(s[-2]) * int(s[-1]))
            state_rw = 2 * 4 * lead * (int(s[-2]) + int(s[-1]))
            state_read = state_rw // 2
            p1 = grad_bytes * n + (2 * 4 * lead * int(s[-2]) if cls in FUSED_CLASSES else 0)
        else:
            state_rw = 2 * 4 * n
            state_read = 4 * n
            p1 = grad_bytes * n + state_rw
        last = int(s[-1]) if len(s) >= 2 else n
        m1 = first_moment_bytes(n, beta1, q8, (n // last if last else 0) * ((last + 127) // 128))
        step += 3 * grad_bytes * n + 8 * n + m1 + state_rw
        impl += (2 if cls in FUSED_CLASSES or cls == "1d" else 3) * grad_bytes * n + 8 * n + m1 + state_rw
        slots[f"k_pass1[{cls}]"] = slots.get(f"k_pass1[{cls}]", 0) + p1
        if cls.startswith(("vec", "elem")):
            slots[f"k_pass2[{cls}]"] = slots.get(f"k_pass2[{cls}]", 0) + grad_bytes * n
        slots[f"k_apply[{cls}]"] = slots.get(f"k_apply[{cls}]", 0) + grad_bytes * n + 8 * n + m1 + state_read
    return step, impl, slots


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi (every 50 ms)
    while the benchmark runs; summary() keeps the samples taken inside the
    timed window (host wall clock), or the whole sampling span when the window
    caught fewer than 3."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.out = ""
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    @staticmethod
    def _ts(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        rows = []
        for r in csv.reader(io.StringIO(self.out or "")):
            r = [x.strip() for x in r]
            if len(r) < 10 or (self.uuid and self.uuid not in r[1]):
                continue
            rows.append(r)
        scope = "whole run"
        if self.window and rows:
            inside = [r for r in rows if (ts := self._ts(r[0])) is not None
                      and self.window[0] - 0.05 <= ts <= self.window[1] + 0.05]
            if len(inside) >= 3:
                rows, scope = inside, "timed region"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[2]) for r in rows) if v is not None]
        mx = [v for v in (num(r[3]) for r in rows) if v is not None]
        pw = [v for v in (num(r[4]) for r in rows) if v is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(rows), "scope": scope}


def device_uuid(dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# Sections of the kernel source (by their "// ---- <title>" banner) that hold
# a launch slot's code; the traffic record of the slot stays valid while
# these sections and the shared header are unchanged.
KERNEL_SECTIONS = {
    "k_apply": ("small helpers", "per-tile column factors", "apply: ", "vector path of apply", "apply (vector path)",
                "apply of the flat class"),
}


def kernel_source_digest(kernel):
    """sha256 of the source a launch slot's kernel is built from: the shared
    headers (adafactor_internal.h, row_panel.cuh) plus the slot's sections of
    the kernel file (the whole file for slots without a section list); for
    the LAMB and CAME kernels, their own source file and header with the
    shared headers they include."""
    for prefix, files in (("k_lamb", (LAMB_SRC, LAMB_HDR, KERNEL_HDR)),
                          ("k_came", (CAME_SRC, CAME_HDR, KERNEL_HDR, PANEL_HDR))):
        if kernel.startswith(prefix):
            text = "".join(open(f, encoding="utf-8").read() for f in files)
            return hashlib.sha256(text.encode()).hexdigest()
    text = open(KERNEL_SRC, encoding="utf-8").read()
    titles = KERNEL_SECTIONS.get(kernel.split("[")[0])
    if titles:
        parts = re.split(r"(?m)^// ---- ", text)[1:]
        text = "".join(p for p in parts if p.startswith(titles))
    header = "".join(open(f, encoding="utf-8").read() for f in (KERNEL_HDR, PANEL_HDR))
    return hashlib.sha256((header + text).encode()).hexdigest()


def traffic_record(kernel, workload):
    """dram bytes per full launch of `kernel` in `workload` from the committed
    ncu summary (records are keyed "workload/kernel": a launch slot moves
    different bytes in different workloads), or None when there is no record
    or the kernel's source changed since the counters were taken."""
    if workload is None:
        return None
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        sha = kernel_source_digest(kernel)
        entry = rec.get(f"{workload}/{kernel}")
        if entry and entry.get("kernel_source_sha256") == sha:
            return float(entry["dram_bytes_per_full_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# ---------------------------------------------------------------- our arm --
class HugePinned:
    """Page-locked host memory backed by transparent huge pages: anonymous
    memory advised MADV_HUGEPAGE, touched, then registered with
    cudaHostRegister.  The GPU's DMA then walks one translation per huge page
    (512 MB on the 64 KB-page Arm hosts) instead of one per base page.
    Measured on the GB300 host after a process that had used some 40 GB of
    host memory exited: the double-buffered e2e upload from a torch pinned
    buffer (base pages) took 152 ms per step while the device step ran
    beside it, from this buffer 79 ms (the plain copy alone: 76 ms in both).
    `tensor` is a uint8 tensor over the memory; close() unregisters it."""

    def __init__(self, nbytes):
        self.nbytes = max(int(nbytes), 1)
        self.mm = mmap.mmap(-1, self.nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        if hasattr(self.mm, "madvise") and hasattr(mmap, "MADV_HUGEPAGE"):
            self.mm.madvise(mmap.MADV_HUGEPAGE)
        self.tensor = torch.frombuffer(self.mm, dtype=torch.uint8)
        self.tensor.fill_(0)  # fault the pages in (huge pages where the kernel has them)
        rc = torch.cuda.cudart().cudaHostRegister(self.tensor.data_ptr(), self.nbytes, 0)
        self.registered = int(rc) == 0
        if not self.registered:
            raise RuntimeError(f"cudaHostRegister failed: {rc}")

    def close(self):
        if self.registered:
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaHostUnregister(self.tensor.data_ptr())
            self.registered = False


def flat_views(like, device, pin=False, huge=False):
    """One contiguous buffer holding a tensor of each shape/dtype of `like`
    (offsets rounded up to 256 bytes) and the views into it.  With huge=True
    (host only) the buffer is a HugePinned block; its owner is returned as a
    third value (None otherwise), to be closed when the views are done."""
    offs, total = [], 0
    for x in like:
        offs.append(total)
        total += (x.numel() * x.element_size() + 255) // 256 * 256
    owner = None
    if huge:
        owner = HugePinned(total)
        buf = owner.tensor
    else:
        buf = torch.empty(max(total, 1), dtype=torch.uint8, device=device, pin_memory=pin)
    views = [buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for o, x in zip(offs, like)]
    return (buf, views, owner) if huge else (buf, views)


def plain_h2d_rate(host_flat, dev_flat, dev, world, reps=2):
    """The box's plain host->device copy rate for the same bytes as one e2e
    step: one cudaMemcpyAsync of the flat pinned gradient buffer, nothing else
    running; best of `reps`, CUDA events."""
    nbytes = host_flat.numel()
    s = torch.cuda.current_stream(dev)
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(s)
        dev_flat.copy_(host_flat, non_blocking=True)
        e1.record(s)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        best = ms if best is None else min(best, ms)
    return {"h2d_gbs": nbytes / (best / 1e3) / 1e9, "bytes": nbytes, "ms": best,
            "how": "one cudaMemcpyAsync of the flat pinned gradient buffer, one stream, nothing else running, best "
                   f"of {reps}; frac_of_link = this copy time / the e2e step time"}


HOST_NUMA = None


def bind_to_gpu_numa_node(local: int):
    """Restricts this process to the host CPUs of the GPU's NUMA node (from
    sysfs), before any pinned buffer is allocated, so that pinned pages are
    first touched on the node nearest the GPU.  Records what it did in
    HOST_NUMA; leaves the affinity alone where sysfs gives no answer."""
    global HOST_NUMA
    info = {"gpu_numa_node": None, "cpus": None, "bound": False}
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(local), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout.strip()
        bus = out.lower()
        if bus.count(":") == 2 and len(bus.split(":")[0]) == 8:
            bus = bus[4:]  # nvidia-smi prints an 8-digit domain, sysfs a 4-digit one
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            node = int(f.read().strip())
        info["gpu_numa_node"] = node
        if node >= 0:
            with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
                cpus = set()
                for part in f.read().strip().split(","):
                    if "-" in part:
                        a, b = part.split("-")
                        cpus.update(range(int(a), int(b) + 1))
                    elif part:
                        cpus.add(int(part))
            allowed = os.sched_getaffinity(0) & cpus
            if allowed:
                os.sched_setaffinity(0, allowed)
                info["cpus"] = len(allowed)
                info["bound"] = True
    except (OSError, ValueError, subprocess.SubprocessError):
        pass
    HOST_NUMA = info
    return info


class numa_local:
    """Within the block, the process runs on the CPUs of the GPU's NUMA node
    (bind_to_gpu_numa_node); the previous affinity comes back afterwards.  The
    pinned buffers allocated inside keep their node-local pages."""

    def __init__(self, local: int):
        self.local = local
        self.saved = None

    def __enter__(self):
        self.saved = os.sched_getaffinity(0)
        bind_to_gpu_numa_node(self.local)
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.saved)
        return False


class E2EUploads:
    """Double-buffered gradient uploads of an end-to-end run.  The step's
    gradients live in one flat pinned host buffer (as a training loop's flat
    gradient buffer would; huge-page backed, HugePinned), and each step
    copies it with one cudaMemcpyAsync into one of two flat device buffers,
    on its own stream, while the previous step runs.  (291 separate pinned
    buffers, one copy each, measured erratic on the GB300 host: 77 to 294 ms
    for the same 16 GB, against a steady 76 ms for one flat buffer.)"""

    def __init__(self, grads, dev):
        self.host, hviews, self.owner = flat_views(grads, "cpu", huge=True)
        for hv, g in zip(hviews, grads):
            hv.copy_(g)
        self.dev_flat, self.views = [], []
        for _ in range(2):
            buf, views = flat_views(grads, dev)
            self.dev_flat.append(buf)
            self.views.append(views)
        self.nbytes = sum(g.numel() * g.element_size() for g in grads)
        self.s_in = torch.cuda.Stream(dev)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_step = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]

    def upload(self, k):
        b = k % 2
        if self.used[b]:
            self.s_in.wait_event(self.ev_step[b])  # the step that last read this buffer is done
        with torch.cuda.stream(self.s_in):
            self.dev_flat[b].copy_(self.host, non_blocking=True)
            self.ev_in[b].record(self.s_in)

    def before_step(self, k, s_comp):
        s_comp.wait_event(self.ev_in[k % 2])

    def after_step(self, k, s_comp):
        self.used[k % 2] = True
        self.ev_step[k % 2].record(s_comp)

    def timed(self, nsteps, compute, s_comp, world, dev):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        e0.record(s_comp)
        self.s_in.wait_event(e0)
        self.upload(0)
        for k in range(nsteps):
            if k + 1 < nsteps:
                self.upload(k + 1)
            self.before_step(k, s_comp)
            compute(k)
            self.after_step(k, s_comp)
        e1.record(s_comp)
        torch.cuda.synchronize(dev)
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / nsteps


def run_e2e(args, wl, params, grads, states, step, t, world, dev):
    """End to end through AdafactorStep, as a training loop with host-resident
    gradients would drive it: every step copies that step's bf16 grads from
    pinned host memory to the device, runs the step, and reads back the step's
    metric, the per-tensor sum(p^2) of the updated parameters (one float64
    per tensor, from which the host forms the parameter norm).  Grads for
    step t+1 go up on their own stream, into the second of two device grad
    buffers, while step t runs (E2EUploads).

    A second, shorter measurement (`param_readback`) also copies every updated
    fp32 parameter back to pinned host memory each step (one flat pinned
    buffer), for callers that keep the master weights on the host."""
    n = len(params)
    psq = torch.zeros(n, dtype=torch.float64, device=dev)
    for k, st in enumerate(states):
        st["param_sq_sum"] = psq[k:k + 1]
    up = E2EUploads(grads, dev)
    host_m = torch.empty(n, dtype=torch.float64, pin_memory=True)
    steps = [AdafactorStep(params, up.views[b], states, **wl.hparams) for b in range(2)]
    s_comp = torch.cuda.current_stream(dev)
    readback = None

    def compute(k):
        nonlocal t
        t += 1
        steps[k % 2](t, stream=s_comp)
        host_m.copy_(psq, non_blocking=True)
        if readback is not None:
            for hp_, p in zip(readback, params):
                hp_.copy_(p, non_blocking=True)

    up.timed(2, compute, s_comp, world, dev)  # warm-up: both step objects marshalled, carry primed
    ms = up.timed(args.e2e_steps, compute, s_comp, world, dev)
    norm = float(host_m.sum().sqrt())
    link = plain_h2d_rate(up.host, up.dev_flat[0], dev, world)
    out = {"value": replica_throughput(wl.numel, world, ms), "unit": "params/s",
           "h2d_bytes_per_step": up.nbytes, "d2h_bytes_per_step": n * 8, "steps": args.e2e_steps, "ms_per_step": ms,
           "result_read": f"per-tensor sum(p^2) of the updated params ({n} float64; param norm {norm:.4f})",
           "path": "one flat pinned (huge-page backed) host buffer of bf16 grads -> device in one copy (double-buffered, own stream, "
                   "overlapping the previous step), AdafactorStep, device->host read of the step metric",
           "link": link, "host_numa": HOST_NUMA,
           "frac_of_link": (link["ms"] / ms) if ms > 0 else None}
    # (one GPU only: each rank would pin another 32 GB of host memory)
    if args.readback_steps > 0 and world == 1:
        host_pflat, readback = flat_views(params, "cpu", pin=True)
        rms = up.timed(args.readback_steps, compute, s_comp, world, dev)
        out["param_readback"] = {"ms_per_step": rms, "value": replica_throughput(wl.numel, world, rms),
                                 "d2h_bytes_per_step": sum(p.numel() * p.element_size() for p in params),
                                 "steps": args.readback_steps}
        readback = None
        del host_pflat
    for st in states:
        st.pop("param_sq_sum", None)
    up.owner.close()
    del up
    return out, t


class EmulatedRowShards:
    """The workload split by rows into R blocks, each stepped by its own
    AdafactorShardStep (the row-sharded step of the article's Step 4), the R
    "ranks" running in turn on this GPU and the all-reduces between the
    library calls done as device-side sums of the R exchange buffers.  One
    call = one step of the whole job."""

    def __init__(self, params, grads, states_fn, nshards, hparams):
        self.steps = []
        for r in range(nshards):
            ps, gs, rows = [], [], []
            for p, g in zip(params, grads):
                fact = p.dim() >= 2
                n = p.shape[-2] if fact else p.numel()
                a, b = (n * r) // nshards, (n * (r + 1)) // nshards
                ps.append((p[..., a:b, :] if fact else p.reshape(-1)[a:b]).contiguous())
                gs.append((g[..., a:b, :] if fact else g.reshape(-1)[a:b]).contiguous())
                rows.append(n)
            self.steps.append(AdafactorShardStep(ps, gs, states_fn(ps), rows, **hparams))
        self.round_bytes = self.steps[0].round1.numel() * 8 + self.steps[0].round2.numel() * 8

    def __call__(self, t):
        for st in self.steps:
            st.begin(t)
        if len(self.steps) > 1:
            tot = torch.stack([st.round1 for st in self.steps]).sum(0)
            for st in self.steps:
                st.round1.copy_(tot)
        for st in self.steps:
            st.middle(t)
        if len(self.steps) > 1:
            tot = torch.stack([st.round2 for st in self.steps]).sum(0)
            for st in self.steps:
                st.round2.copy_(tot)
        for st in self.steps:
            st.end(t)


def timed_and_profiled(step, t, nsteps, stream, dev, world, clocks, profile_enable, profile_read):
    """Times nsteps steps with CUDA events on the launch stream, nothing else
    recorded in between (the step time reported), then runs nsteps more with
    the library's per-kernel event pairs on (the per-kernel table).  Returns
    (ms per timed step, the per-kernel record, the last step number)."""
    profile_read()  # drop anything recorded so far
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    w0 = time.time()
    ev0.record(stream)
    for _ in range(nsteps):
        t += 1
        step(t)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(w0, time.time())
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev) / nsteps
    profile_enable(True)
    for _ in range(nsteps):
        t += 1
        step(t)
    torch.cuda.synchronize(dev)
    profile_enable(False)
    clocks.stop()
    return ms, profile_read(), t


def run_ours(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.workload(args.workload)
    shapes = [s for _, s in wl.shapes]
    n_params = wl.numel
    beta1 = wl.hparams.get("beta1")
    q8 = bool(wl.hparams.get("exp_avg_int8"))
    params = [synth.make_param(s, k, device=dev, std=wl.param_std) for k, s in enumerate(shapes)]
    grads = [synth.make_grad(s, k, 1, device=dev, std=wl.grad_std, dtype=wl.grad_dtype, kind=wl.grad_kind)
             for k, s in enumerate(shapes)]
    if args.shards:
        # row-sharded step, every shard on this GPU (the whole tensors are freed)
        step = EmulatedRowShards(params, grads, lambda ps: init_state(ps, beta1=beta1, exp_avg_int8=q8), args.shards,
                                 wl.hparams)
        params = grads = states = None
        torch.cuda.empty_cache()
    else:
        states = init_state(params, beta1=beta1, exp_avg_int8=q8)
        step = AdafactorStep(params, grads, states, **wl.hparams)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(device_uuid(dev)).start()
    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms_per_step, kernels, t = timed_and_profiled(step, t, args.steps, stream, dev, world, clocks,
                                                 binding.adafactor_profile_enable, binding.adafactor_profile_read)
    if world > 1:
        torch.distributed.barrier()

    # ---- end to end: host grads in, host params out, through the same API
    e2e = None
    if args.e2e_steps > 0 and not args.shards:
        with numa_local(local):
            e2e, t = run_e2e(args, wl, params, grads, states, step, t, world, dev)

    grad_bytes = 2 if wl.grad_dtype == torch.bfloat16 else 4
    step_bytes, impl_bytes, slot_bytes = algorithmic_bytes(wl.shapes, grad_bytes, beta1 is not None, q8)
    peak, peak_kind = measured_hbm_peak()
    # the library's kernels in the timed region: the profiled launches plus
    # one status-word reset per library call (host_copy.cuh; not profiled;
    # the descriptor table itself is kept on the device after the first call)
    launches = sum(v[1] for v in kernels.values()) + args.steps * (args.shards or 1) * (3 if args.shards else 1)
    per_kernel = {}
    for name, (kms, kn) in kernels.items():
        if not kn:
            continue
        entry = {"ms_per_step": round(kms / args.steps, 4), "launches": kn}
        # a slot's bytes are per step; with row shards one step is several launches
        per = args.steps if args.shards else kn
        if name in slot_bytes and kms > 0:
            entry["gbs"] = round(slot_bytes[name] / (kms / per / 1e3) / 1e9, 1)
        per_kernel[name] = entry
    dom_name, (dom_ms, dom_n) = max(kernels.items(), key=lambda kv: kv[1][0])
    roofline = None
    if dom_n and dom_name in slot_bytes:
        dom_per = args.steps if args.shards else dom_n
        ach = slot_bytes[dom_name] / (dom_ms / dom_per / 1e3) / 1e9
        roofline = {"kernel": dom_name, "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(ach / peak, 4), "peak_source": peak_kind,
                    "traffic": traffic_record(dom_name, None if args.shards else args.workload),
                    "algorithmic_bytes_per_launch": slot_bytes[dom_name],
                    "avg_launch_ms": dom_ms / dom_per}
    eff_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    clk = clocks.summary()
    out = {
        "metric": METRIC, "value": replica_throughput(n_params, world, ms_per_step), "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) fp32 params, N(0,1e-3) bf16 grads resident in HBM)",
        "config": {"workload": args.workload, "description": wl.description, "params": n_params,
                   "tensors": len(shapes), "param_dtype": "fp32",
                   "grad_dtype": "bf16" if grad_bytes == 2 else "fp32",
                   "hparams": {k: v for k, v in wl.hparams.items()} or "defaults",
                   "parallelism": (f"row shards x{args.shards} on one GPU (ranks in turn, exchange summed on "
                                   "the device)" if args.shards else
                                   (f"replicas x{world}" if world > 1 else "single GPU")),
                   "l2": "inputs (params+grads) far larger than L2; no flush"},
        "effective_gbs": round(eff_gbs, 1),
        "pct_of_8tbs": round(100 * eff_gbs / NOMINAL_HBM_GBS, 2),
        "frac_of_hbm_peak": round(eff_gbs / peak, 4), "hbm_peak_gbs": peak, "hbm_peak_source": peak_kind,
        "algorithmic_bytes_per_step": step_bytes,
        "min_bytes_this_design": impl_bytes,
        "gbs_min_bytes_this_design": round(impl_bytes / (ms_per_step / 1e3) / 1e9, 1),
        "kernels": per_kernel,
        "kernels_note": "per-kernel CUDA-event times from a further run of the same number of steps with the "
                        "library's event pairs on; ms_per_step and value come from the timed steps, which record "
                        "no event between launches",
        "roofline": roofline, "gpu_launches": launches, "clocks": clk, "e2e": e2e,
    }
    if args.shards:
        out["row_shards"] = {"shards": args.shards, "exchange_bytes_per_rank_per_step": step.round_bytes}
    return out, (wl, n_params)


# ------------------------------------------------------------------ LAMB --
def lamb_bytes(n_values, grad_bytes):
    """Algorithmic HBM bytes of a LAMB step over n values: per launch of this
    design (moments pass: g, m, v, p read, m, v written; update pass: m, v, p
    read, p written), and the one-pass minimum (g, m, v, p read once; m, v, p
    written once) that a step with norms known in advance would move."""
    moments = n_values * (grad_bytes + 12 + 8)
    update = n_values * 16
    return {"k_lamb_moments": moments, "k_lamb_update": update}, moments + update, n_values * (grad_bytes + 24)


def run_lamb_e2e(args, wl, params, grads, step, t, world, dev):
    """End to end through LambStep: every step copies that step's bf16 grads
    from pinned host memory (E2EUploads: one flat buffer, one copy, own
    stream, overlapping the previous step into a second grad buffer), runs
    the step, and reads back the per-tensor trust ratios (one float64 per
    tensor) to pinned host memory."""
    n = len(params)
    up = E2EUploads(grads, dev)
    steps = [LambStep(params, up.views[b], step.states, **step.hparams) for b in range(2)]
    host_tr = torch.empty(n, dtype=torch.float64, pin_memory=True)
    s_comp = torch.cuda.current_stream(dev)

    def compute(k):
        nonlocal t
        t += 1
        steps[k % 2](t, stream=s_comp)
        trust = steps[k % 2].workspace[:8 * n].view(torch.float64)
        host_tr.copy_(trust, non_blocking=True)

    up.timed(2, compute, s_comp, world, dev)
    ms = up.timed(args.e2e_steps, compute, s_comp, world, dev)
    link = plain_h2d_rate(up.host, up.dev_flat[0], dev, world)
    out = {"value": replica_throughput(wl.numel, world, ms), "unit": "params/s", "h2d_bytes_per_step": up.nbytes,
           "d2h_bytes_per_step": n * 8, "steps": args.e2e_steps, "ms_per_step": ms,
           "result_read": f"per-tensor trust ratios ({n} float64; mean {float(host_tr.mean()):.4f})",
           "path": "one flat pinned (huge-page backed) host buffer of bf16 grads -> device in one copy (double-buffered, own stream, "
                   "overlapping the previous step), LambStep, device->host read of the trust ratios",
           "link": link, "host_numa": HOST_NUMA, "frac_of_link": (link["ms"] / ms) if ms > 0 else None}
    up.owner.close()
    del up
    return out, t


def run_lamb(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.workload(args.workload)
    shapes = [s for _, s in wl.shapes]
    params = [synth.make_param(s, k, device=dev, std=wl.param_std) for k, s in enumerate(shapes)]
    grads = [synth.make_grad(s, k, 1, device=dev, std=wl.grad_std, dtype=wl.grad_dtype, kind=wl.grad_kind)
             for k, s in enumerate(shapes)]
    states = init_lamb_state(params)
    step = LambStep(params, grads, states, **wl.hparams)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(device_uuid(dev)).start()
    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms_per_step, kernels, t = timed_and_profiled(step, t, args.steps, stream, dev, world, clocks,
                                                 binding.lamb_profile_enable, binding.lamb_profile_read)
    e2e = None
    if args.e2e_steps > 0:
        with numa_local(local):
            e2e, t = run_lamb_e2e(args, wl, params, grads, step, t, world, dev)
    grad_bytes = 2 if wl.grad_dtype == torch.bfloat16 else 4
    slot_bytes, design_bytes, one_pass_bytes = lamb_bytes(wl.numel, grad_bytes)
    peak, peak_kind = measured_hbm_peak()
    per_kernel = {}
    for name, (kms, kn) in kernels.items():
        if not kn:
            continue
        entry = {"ms_per_step": round(kms / args.steps, 4), "launches": kn}
        if name in slot_bytes and kms > 0:
            entry["gbs"] = round(slot_bytes[name] / (kms / kn / 1e3) / 1e9, 1)
        per_kernel[name] = entry
    dom_name, (dom_ms, dom_n) = max(kernels.items(), key=lambda kv: kv[1][0])
    ach = slot_bytes[dom_name] / (dom_ms / dom_n / 1e3) / 1e9
    roofline = {"kernel": dom_name, "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_source": peak_kind, "traffic": traffic_record(dom_name, args.workload),
                "algorithmic_bytes_per_launch": slot_bytes[dom_name], "avg_launch_ms": dom_ms / dom_n}
    eff = design_bytes / (ms_per_step / 1e3) / 1e9
    out = {
        "metric": LAMB_METRIC, "value": replica_throughput(wl.numel, world, ms_per_step), "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) fp32 params, N(0,1e-3) bf16 grads resident in HBM)",
        "config": {"workload": args.workload, "description": wl.description, "params": wl.numel,
                   "tensors": len(shapes), "param_dtype": "fp32", "grad_dtype": "bf16" if grad_bytes == 2 else "fp32",
                   "hparams": dict(wl.hparams) or "defaults",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs (params+grads+states) far larger than L2; no flush"},
        "effective_gbs": round(eff, 1), "frac_of_hbm_peak": round(eff / peak, 4), "hbm_peak_gbs": peak,
        "hbm_peak_source": peak_kind, "algorithmic_bytes_per_step": design_bytes,
        "one_pass_bytes_per_step": one_pass_bytes, "kernels": per_kernel, "roofline": roofline,
        "gpu_launches": sum(v[1] for v in kernels.values()),  # the descriptor table is kept on the device
        "clocks": clocks.summary(), "e2e": e2e,
    }
    return out, (wl, wl.numel)


# ------------------------------------------------------------------ CAME --
def came_panel(shape, grad_bytes):
    """Whether the CAME step takes the row-panel pass for a contiguous,
    256-byte aligned tensor: bf16 matrices with W % 8 == 0, 2048 <= W <= 14336."""
    return len(shape) >= 2 and grad_bytes == 2 and int(shape[-1]) % 8 == 0 and 2048 <= int(shape[-1]) <= 14336


def came_bytes(shapes, grad_bytes):
    """Algorithmic HBM bytes of a CAME step per launch slot of this design.
    Row-panel tensors: the panel pass reads g once (statistics and sum(u^2)).
    Other factored tensors: pass a reads g; pass b reads g.  Every factored
    tensor: pass c reads g and m and writes m; pass d reads m and p and writes
    p.  1D tensors: pass a reads g and v and writes v; pass c reads g, v, m,
    S, p and writes m, S, p.  (The row/column statistics and partial sums are
    under 0.2 % and left out.)  Returns (slots, per step, one-pass minimum
    g + m and p read and written)."""
    nf = n1 = npan = 0
    for _, s in shapes:
        n = 1
        for d in s:
            n *= int(d)
        if len(s) >= 2:
            nf += n
            if came_panel(s, grad_bytes):
                npan += n
        else:
            n1 += n
    g = grad_bytes
    slots = {"k_came_pass_a": (nf - npan) * g + n1 * (g + 8), "k_came_pass_b": (nf - npan) * g,
             "k_came_pass_c": nf * (g + 8) + n1 * (g + 28), "k_came_pass_d": nf * 12}
    if npan:
        slots["k_came_panel"] = npan * g
    slots = {k: v for k, v in slots.items() if v}
    return slots, sum(slots.values()), (nf + n1) * (g + 16)


def run_came(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.workload(args.workload)
    shapes = [s for _, s in wl.shapes]
    params = [synth.make_param(s, k, device=dev, std=wl.param_std) for k, s in enumerate(shapes)]
    grads = [synth.make_grad(s, k, 1, device=dev, std=wl.grad_std, dtype=wl.grad_dtype, kind=wl.grad_kind)
             for k, s in enumerate(shapes)]
    states = init_came_state(params)
    step = CameStep(params, grads, states, **wl.hparams)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(device_uuid(dev)).start()
    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms_per_step, kernels, t = timed_and_profiled(step, t, args.steps, stream, dev, world, clocks,
                                                 binding.came_profile_enable, binding.came_profile_read)
    grad_bytes = 2 if wl.grad_dtype == torch.bfloat16 else 4
    slot_bytes, design_bytes, one_pass_bytes = came_bytes(wl.shapes, grad_bytes)
    peak, peak_kind = measured_hbm_peak()
    per_kernel = {}
    for name, (kms, kn) in kernels.items():
        if not kn:
            continue
        entry = {"ms_per_step": round(kms / args.steps, 4), "launches": kn}
        if name in slot_bytes and kms > 0:
            # a slot launches one kernel per tensor class: bytes per step over the slot's time per step
            entry["gbs"] = round(slot_bytes[name] / (kms / args.steps / 1e3) / 1e9, 1)
        per_kernel[name] = entry
    dom_name, (dom_ms, dom_n) = max(kernels.items(), key=lambda kv: kv[1][0])
    ach = slot_bytes[dom_name] / (dom_ms / args.steps / 1e3) / 1e9
    roofline = {"kernel": dom_name, "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_source": peak_kind, "traffic": traffic_record(dom_name, args.workload),
                "algorithmic_bytes_per_launch": slot_bytes[dom_name], "avg_launch_ms": dom_ms / args.steps}
    e2e = None
    if args.e2e_steps > 0:
        with numa_local(local):
            e2e = run_came_e2e(args, wl, params, grads, states, step, t, world, dev)
    eff = design_bytes / (ms_per_step / 1e3) / 1e9
    out = {
        "metric": CAME_METRIC, "value": replica_throughput(wl.numel, world, ms_per_step), "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) fp32 params, N(0,1e-3) bf16 grads resident in HBM)",
        "config": {"workload": args.workload, "description": wl.description, "params": wl.numel,
                   "tensors": len(shapes), "param_dtype": "fp32", "grad_dtype": "bf16" if grad_bytes == 2 else "fp32",
                   "hparams": dict(wl.hparams), "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs (params+grads+states) far larger than L2; no flush"},
        "effective_gbs": round(eff, 1), "frac_of_hbm_peak": round(eff / peak, 4), "hbm_peak_gbs": peak,
        "hbm_peak_source": peak_kind, "algorithmic_bytes_per_step": design_bytes,
        "one_pass_bytes_per_step": one_pass_bytes, "kernels": per_kernel, "roofline": roofline,
        "gpu_launches": sum(v[1] for v in kernels.values()),  # the descriptor table is kept on the device
        "clocks": clocks.summary(), "e2e": e2e,
    }
    return out, (wl, wl.numel)


def run_came_e2e(args, wl, params, grads, states, step, t, world, dev):
    """End to end through CameStep: every step copies the step's bf16 grads
    from pinned host memory (E2EUploads: one flat buffer, one copy, own
    stream, into the second of two grad buffers while the previous step
    runs), runs the step, and reads back one value per tensor (the first
    updated parameter value) to pinned host memory."""
    n = len(params)
    up = E2EUploads(grads, dev)
    steps = [CameStep(params, up.views[b], states, **wl.hparams) for b in range(2)]
    heads = torch.empty(n, dtype=torch.float32, device=dev)
    host_h = torch.empty(n, dtype=torch.float32, pin_memory=True)
    s_comp = torch.cuda.current_stream(dev)
    firsts = [p.view(-1)[:1] for p in params]

    def compute(k):
        nonlocal t
        t += 1
        steps[k % 2](t, stream=s_comp)
        torch.cat(firsts, out=heads)
        host_h.copy_(heads, non_blocking=True)

    up.timed(2, compute, s_comp, world, dev)
    ms = up.timed(args.e2e_steps, compute, s_comp, world, dev)
    link = plain_h2d_rate(up.host, up.dev_flat[0], dev, world)
    out = {"value": replica_throughput(wl.numel, world, ms), "unit": "params/s", "h2d_bytes_per_step": up.nbytes,
           "d2h_bytes_per_step": n * 4, "steps": args.e2e_steps, "ms_per_step": ms,
           "result_read": f"first updated value of each tensor ({n} float32)",
           "path": "one flat pinned (huge-page backed) host buffer of bf16 grads -> device in one copy (double-buffered, own stream, "
                   "overlapping the previous step), CameStep, device->host read of one value per tensor",
           "link": link, "host_numa": HOST_NUMA, "frac_of_link": (link["ms"] / ms) if ms > 0 else None}
    up.owner.close()
    del up
    return out


def time_came_oracle(wl, idx, steps, t0=1):
    """The CAME oracle over the sampled tensors; (seconds per step, values)."""
    import numpy as np
    from oracle import came as came_oracle
    came_oracle.build()
    hp = came_oracle.CameHParams(**wl.hparams)
    shapes = [wl.shapes[k][1] for k in idx]
    ps = [synth.make_param(s, k, std=wl.param_std).double().numpy() for s, k in zip(shapes, idx)]
    sts = [came_oracle.CameState(s) for s in shapes]
    gs = [synth.make_grad(s, k, 1, std=wl.grad_std, dtype=wl.grad_dtype, kind=wl.grad_kind).double().numpy()
          for s, k in zip(shapes, idx)]
    per_step = []
    for t in range(t0, t0 + steps):
        a = time.perf_counter()
        for p, g, st in zip(ps, gs, sts):
            came_oracle.step(p, g, st, t, hp)
        per_step.append(time.perf_counter() - a)
    return per_step, int(sum(np.prod(s) if s else 1 for s in shapes))


def time_lamb_oracle(wl, idx, steps, t0=1):
    """The LAMB oracle over the sampled tensors; (seconds per step, values)."""
    import numpy as np
    from oracle import lamb as lamb_oracle
    lamb_oracle.build()
    hp = lamb_oracle.LambHParams(**wl.hparams)
    shapes = [wl.shapes[k][1] for k in idx]
    ps = [synth.make_param(s, k, std=wl.param_std).double().numpy() for s, k in zip(shapes, idx)]
    sts = [lamb_oracle.LambState(s) for s in shapes]
    gs = [synth.make_grad(s, k, 1, std=wl.grad_std, dtype=wl.grad_dtype, kind=wl.grad_kind).double().numpy()
          for s, k in zip(shapes, idx)]
    per_step = []
    for t in range(t0, t0 + steps):
        a = time.perf_counter()
        for p, g, st in zip(ps, gs, sts):
            lamb_oracle.step(p, g, st, t, hp)
        per_step.append(time.perf_counter() - a)
    return per_step, int(sum(np.prod(s) if s else 1 for s in shapes))


# ----------------------------------------------------------- oracle arms --
def oracle_sample(wl, seconds_hint=10.0):
    """A bounded sample of the workload for the CPU oracle: the tensors of one
    decoder layer (Llama workloads) or the first tensors up to ~2e8 values."""
    import numpy as np
    shapes = wl.shapes
    idx = [k for k, (name, _) in enumerate(shapes) if name.startswith("layers.0.")]
    if not idx:
        idx, tot = [], 0
        for k, (_, s) in enumerate(shapes):
            n = int(np.prod(s)) if s else 1
            if tot + n > 2e8 and idx:
                break
            idx.append(k)
            tot += n
    return idx


def time_oracle(wl, idx, steps, t0=1):
    """Runs the oracle `steps` times over the sampled tensors; returns the
    seconds spent inside the oracle and the values processed."""
    import numpy as np
    import oracle
    oracle.build()
    hp = oracle.HParams(**wl.hparams)
    shapes = [wl.shapes[k][1] for k in idx]
    ps = [synth.make_param(s, k, std=wl.param_std).double().numpy() for s, k in zip(shapes, idx)]
    sts = [oracle.State(s, beta1=wl.hparams.get("beta1") is not None) for s in shapes]
    gs = [synth.make_grad(s, k, 1, std=wl.grad_std, dtype=wl.grad_dtype, kind=wl.grad_kind).double().numpy()
          for s, k in zip(shapes, idx)]
    per_step = []
    for t in range(t0, t0 + steps):
        a = time.perf_counter()
        for p, g, st in zip(ps, gs, sts):
            oracle.step(p, g, st, t, hp)
        per_step.append(time.perf_counter() - a)
    n = int(sum(np.prod(s) if s else 1 for s in shapes))
    return per_step, n


def cpu_baseline(wl, steps=2):
    idx = oracle_sample(wl)
    per_step, n = ORACLE_TIMERS[wl.optimizer](wl, idx, steps)
    tot = sum(per_step)
    return {"value": n * steps / tot, "unit": "params/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(idx)} tensors ({n:,} values: "
                      f"{'decoder layer 0' if wl.shapes[idx[0]][0].startswith('layers.0.') else 'leading tensors'}"
                      f") x {steps} steps, float64 C oracle, single thread, inputs pre-generated",
            "seconds": tot, "host_cpus": os.cpu_count()}


ORACLE_TIMERS = {"adafactor": time_oracle, "lamb": time_lamb_oracle, "came": time_came_oracle}


def _oracle_worker(args):
    """One sampled tensor through the oracle in a worker process: (values, seconds)."""
    workload, k, steps = args
    sys.path.insert(0, ROOT)
    wl = synth.workload(workload)
    per_step, n = ORACLE_TIMERS[wl.optimizer](wl, [k], steps)
    return n * steps, sum(per_step)


def cpu_baseline_all_cores(wl, workload, steps=2):
    """The same sample with the oracle as it stands, one tensor per worker
    process on the host's cores (the oracle is per tensor, so this needs no
    change to it).  Workers are started with `spawn` (this process already
    holds a CUDA context).  Throughput = values processed / the longest
    worker's oracle time, i.e. the makespan if the workers start together."""
    import multiprocessing as mproc
    from concurrent.futures import ProcessPoolExecutor
    idx = oracle_sample(wl)
    workers = max(1, min(os.cpu_count() or 1, len(idx)))
    with ProcessPoolExecutor(max_workers=workers, mp_context=mproc.get_context("spawn")) as ex:
        res = list(ex.map(_oracle_worker, [(workload, k, steps) for k in idx]))
    vals = sum(r[0] for r in res)
    span = max(r[1] for r in res)
    return {"value": vals / span, "unit": "params/s", "cores": workers, "kind": "oracle",
            "sample": f"{len(idx)} tensors ({vals // steps:,} values) x {steps} steps, float64 C oracle, one "
                      f"tensor per worker process ({workers} of {os.cpu_count()} host cores)",
            "seconds_longest_worker": span, "host_cpus": os.cpu_count()}


def run_reference(args):
    wl = synth.workload(args.workload)
    idx = oracle_sample(wl)
    timer = ORACLE_TIMERS[wl.optimizer]
    warm, n = timer(wl, idx, args.warmup) if args.warmup else ([], 0)
    per_step, n = timer(wl, idx, args.steps, t0=args.warmup + 1)
    sec = sum(per_step) / len(per_step)
    value = n / sec
    return {
        "metric": {"lamb": LAMB_METRIC, "came": CAME_METRIC}.get(wl.optimizer, METRIC), "impl": "reference",
        "value": value, "unit": "params/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "description": wl.description, "params": wl.numel,
                   "sampled_params_per_step": n},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(idx)} tensors ({n:,} values) per step, float64 C oracle, "
                                   f"single thread"},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b",
                    choices=["llama3_8b", "llama3_8b_beta1", "llama3_8b_beta1_int8", "llama_layer", "llama_layer_bf16",
                             "llama_layer_bf16_int8", "edge", "tiny", "llama3_8b_lamb", "llama_layer_lamb", "llama3_8b_came",
                             "llama_layer_came"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--readback-steps", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shards", type=int, default=0,
                    help="run the row-sharded step with this many row shards on one GPU (exchange on the device)")
    args = ap.parse_args()
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one rank per GPU: start this same command under torch.distributed.run
        sys.exit(launch_ranks(args.gpus, os.path.abspath(__file__), sys.argv[1:]))
    world, rank, local = dist_env()
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        sys.exit(2)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    binding.load()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    runner = {"lamb": run_lamb, "came": run_came}.get(synth.workload(args.workload).optimizer, run_ours)
    out, (wl, _) = runner(args, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(wl)
            out["cpu_baseline_all_cores"] = cpu_baseline_all_cores(wl, args.workload)
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
