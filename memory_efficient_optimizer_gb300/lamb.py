"""PyTorch front end of the CUDA LAMB step (include/lamb.h).

As for Adafactor, PyTorch only provides device memory and streams: these
functions check and marshal arguments, allocate zeroed state and the
workspace, and make one call into the C library per step.

Article: Colossal-AI distributed-optimizer article, "其余优化器的关键参数速查"
(DistributedLAMB: defaults lr=1e-3, betas=(0.9, 0.999), eps=1e-6,
weight_decay=0, bias_correction=True; checks of lr, eps and betas; the
per-layer trust ratio).  The rule is the LAMB algorithm of arXiv:1904.00962.
"""
from __future__ import annotations

from typing import Iterable, Sequence

import torch

from . import binding as B

_GRAD_DTYPES = {torch.float32: B.ADAF_FLOAT32, torch.bfloat16: B.ADAF_BFLOAT16}


def make_lamb_hparams(lr=1e-3, betas=(0.9, 0.999), eps=1e-6, weight_decay=0.0,
                      bias_correction=True) -> B.lamb_hparams:
    """Validated lamb_hparams (the library's checks; a bad value raises ValueError)."""
    try:
        b1, b2 = betas
    except (TypeError, ValueError):
        raise ValueError("betas must be a pair (beta1, beta2)") from None
    hp = B.lamb_hparams(float(lr), float(b1), float(b2), float(eps), float(weight_decay),
                        1 if bias_correction else 0)
    B.lamb_validate(hp)
    return hp


def init_lamb_state(params: Sequence[torch.Tensor]) -> list:
    """Zeroed fp32 exp_avg / exp_avg_sq for each parameter."""
    return [{"exp_avg": torch.zeros_like(p, dtype=torch.float32, memory_format=torch.contiguous_format),
             "exp_avg_sq": torch.zeros_like(p, dtype=torch.float32, memory_format=torch.contiguous_format)}
            for p in params]


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


class LambStep:
    """A marshalled multi-tensor LAMB step: the descriptor array and the
    workspace are built once; every call is one C-library call."""

    def __init__(self, params: Sequence[torch.Tensor], grads: Sequence[torch.Tensor], states: Sequence[dict],
                 lr=1e-3, betas=(0.9, 0.999), eps=1e-6, weight_decay=0.0, bias_correction=True):
        params, grads, states = list(params), list(grads), list(states)
        if len(params) != len(grads) or len(params) != len(states):
            raise ValueError("params, grads and states must have the same length")
        self.hparams = dict(lr=lr, betas=tuple(betas), eps=eps, weight_decay=weight_decay,
                            bias_correction=bias_correction)
        self._hp = make_lamb_hparams(**self.hparams)
        self.params, self.grads, self.states = params, grads, states
        n = len(params)
        self.n = n
        self.device = params[0].device if n else None
        self._tensors = (B.lamb_tensor * max(1, n))()
        for k, (p, g, st) in enumerate(zip(params, grads, states)):
            if not isinstance(p, torch.Tensor) or p.dtype != torch.float32:
                raise ValueError(f"tensor {k}: params must be float32 tensors")
            if p.device.type != "cuda" or g.device != p.device or p.device != self.device:
                raise ValueError(f"tensor {k}: params and grads must be CUDA tensors on one device")
            if g.dtype not in _GRAD_DTYPES:
                raise ValueError(f"tensor {k}: grad dtype must be float32 or bfloat16")
            if tuple(g.shape) != tuple(p.shape):
                raise ValueError(f"tensor {k}: grad shape {tuple(g.shape)} != param shape {tuple(p.shape)}")
            if not p.is_contiguous() or not g.is_contiguous():
                raise ValueError(f"tensor {k}: params and grads must be contiguous")
            for name in ("exp_avg", "exp_avg_sq"):
                t = st.get(name)
                if not (isinstance(t, torch.Tensor) and t.dtype == torch.float32 and t.device == p.device
                        and t.is_contiguous() and t.numel() == p.numel()):
                    raise ValueError(f"tensor {k}: state '{name}' must be contiguous float32 with "
                                     f"{p.numel()} elements on the param's device")
            self._tensors[k] = B.lamb_tensor(_ptr(p), _ptr(g), _GRAD_DTYPES[g.dtype], p.numel(),
                                             _ptr(st["exp_avg"]), _ptr(st["exp_avg_sq"]))
        self.workspace_bytes = B.lamb_workspace_size(self._tensors, n) if n else 0
        self.workspace = (torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=self.device)
                          if n else None)

    def __call__(self, step: int, stream: torch.cuda.Stream | None = None) -> None:
        if self.n == 0:
            return
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        B.lamb_step(self._tensors, self.n, int(step), self._hp, _ptr(self.workspace), self.workspace_bytes,
                    int(stream.cuda_stream))

    def trust_ratios(self, stream: torch.cuda.Stream | None = None) -> list:
        """Trust ratios of the last step, in list order (synchronises the stream)."""
        if self.n == 0:
            return []
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return B.lamb_trust_ratios(_ptr(self.workspace), self.n, int(stream.cuda_stream))


def lamb_step(params, grads, states, step: int, lr=1e-3, betas=(0.9, 0.999), eps=1e-6, weight_decay=0.0,
              bias_correction=True, stream=None) -> None:
    """One LAMB step over a list of tensors (functional form); states come from
    init_lamb_state(), t is 1-based.  Use LambStep to marshal once."""
    LambStep(params, grads, states, lr=lr, betas=betas, eps=eps, weight_decay=weight_decay,
             bias_correction=bias_correction)(step, stream)


class Lamb(torch.optim.Optimizer):
    """torch.optim.Optimizer wrapper with the article's DistributedLAMB
    defaults; each parameter group is one call into the library."""

    def __init__(self, params: Iterable, lr=1e-3, betas=(0.9, 0.999), eps=1e-6, weight_decay=0.0,
                 bias_correction=True):
        make_lamb_hparams(lr, betas, eps, weight_decay, bias_correction)
        super().__init__(params, dict(lr=lr, betas=tuple(betas), eps=eps, weight_decay=weight_decay,
                                      bias_correction=bias_correction))
        self._plans = {}

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for gi, group in enumerate(self.param_groups):
            hp = {k: group[k] for k in ("lr", "betas", "eps", "weight_decay", "bias_correction")}
            by_step = {}
            for p in group["params"]:
                if p.grad is None:
                    continue
                st = self.state[p]
                if not st:
                    st.update(init_lamb_state([p])[0])
                    st["step"] = 0
                st["step"] += 1
                by_step.setdefault(st["step"], []).append(p)
            for t, ps in by_step.items():
                grads = [p.grad for p in ps]
                key = (gi, tuple(p.data_ptr() for p in ps), tuple(g.data_ptr() for g in grads),
                       repr(sorted(hp.items())))
                plan = self._plans.get(key)
                if plan is None:
                    states = [{k: v for k, v in self.state[p].items() if k != "step"} for p in ps]
                    plan = LambStep(ps, grads, states, **hp)
                    if len(self._plans) > 16:
                        self._plans.clear()
                    self._plans[key] = plan
                plan(t)
        return loss


def lamb_bytes_per_value(grad_bytes: int) -> dict:
    """Algorithmic HBM bytes per value: this design's two passes, and one pass
    (what a step needs if the norms were known in advance)."""
    return {"design": (grad_bytes + 12 + 8) + 16, "one_pass": grad_bytes + 12 + 12,
            "moments_pass": grad_bytes + 12 + 8, "update_pass": 16}


__all__ = ["Lamb", "LambStep", "lamb_step", "init_lamb_state", "make_lamb_hparams", "lamb_bytes_per_value"]
