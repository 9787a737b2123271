"""PyTorch front end of the CUDA CAME step (include/came.h).

PyTorch only provides device memory and streams: these functions check and
marshal arguments, allocate zeroed state and the workspace, and make one call
into the C library per step.

Article: Colossal-AI distributed-optimizer article, overview table (CAME row)
and "其余优化器的关键参数速查" (DistributedCAME: lr=None, eps=(1e-30, 1e-16),
clip_threshold=1.0, betas=(0.9, 0.999, 0.9999), weight_decay=0.0).  The rule
is the CAME algorithm of arXiv:2307.02047.
"""
from __future__ import annotations

from typing import Iterable, Sequence

import torch

from . import binding as B
from .optim import factored_dims

_GRAD_DTYPES = {torch.float32: B.ADAF_FLOAT32, torch.bfloat16: B.ADAF_BFLOAT16}


def make_came_hparams(lr=None, eps=(1e-30, 1e-16), clip_threshold=1.0, betas=(0.9, 0.999, 0.9999),
                      weight_decay=0.0) -> B.came_hparams:
    """Validated came_hparams; CAME has no default learning rate."""
    if lr is None:
        raise ValueError("CAME needs a learning rate (lr has no default)")
    try:
        e1, e2 = eps
        b1, b2, b3 = betas
    except (TypeError, ValueError):
        raise ValueError("eps must be a pair and betas a triple") from None
    hp = B.came_hparams(float(lr), float(e1), float(e2), float(clip_threshold), float(b1), float(b2), float(b3),
                        float(weight_decay))
    B.came_validate(hp)
    return hp


def init_came_state(params: Sequence[torch.Tensor]) -> list:
    """Zeroed fp32 CAME state for each parameter: exp_avg, plus factored
    second-moment and instability rows/columns (ndim >= 2) or full
    exp_avg_sq / exp_avg_res (ndim < 2)."""
    out = []
    for p in params:
        st = {"exp_avg": torch.zeros(p.shape, dtype=torch.float32, device=p.device)}
        fd = factored_dims(p.shape)
        if fd is not None:
            b, h, w = fd
            for name, size in (("exp_avg_sq_row", b * h), ("exp_avg_sq_col", b * w), ("exp_avg_res_row", b * h),
                               ("exp_avg_res_col", b * w)):
                st[name] = torch.zeros(size, dtype=torch.float32, device=p.device)
        else:
            st["exp_avg_sq"] = torch.zeros(p.numel(), dtype=torch.float32, device=p.device)
            st["exp_avg_res"] = torch.zeros(p.numel(), dtype=torch.float32, device=p.device)
        out.append(st)
    return out


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


class CameStep:
    """A marshalled multi-tensor CAME step: descriptors and workspace are
    built once; every call is one C-library call."""

    def __init__(self, params: Sequence[torch.Tensor], grads: Sequence[torch.Tensor], states: Sequence[dict],
                 lr=None, eps=(1e-30, 1e-16), clip_threshold=1.0, betas=(0.9, 0.999, 0.9999), weight_decay=0.0):
        params, grads, states = list(params), list(grads), list(states)
        if len(params) != len(grads) or len(params) != len(states):
            raise ValueError("params, grads and states must have the same length")
        self.hparams = dict(lr=lr, eps=tuple(eps), clip_threshold=clip_threshold, betas=tuple(betas),
                            weight_decay=weight_decay)
        self._hp = make_came_hparams(**self.hparams)
        self.params, self.grads, self.states = params, grads, states
        n = len(params)
        self.n = n
        self.device = params[0].device if n else None
        self._tensors = (B.came_tensor * max(1, n))()
        self._states = (B.came_state * max(1, n))()
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
            if p.dim() > B.ADAF_MAX_NDIM:
                raise ValueError(f"tensor {k}: at most {B.ADAF_MAX_NDIM} dims")
            fd = factored_dims(p.shape)
            need = ({"exp_avg": p.numel(), "exp_avg_sq_row": fd[0] * fd[1], "exp_avg_sq_col": fd[0] * fd[2],
                     "exp_avg_res_row": fd[0] * fd[1], "exp_avg_res_col": fd[0] * fd[2]} if fd is not None else
                    {"exp_avg": p.numel(), "exp_avg_sq": p.numel(), "exp_avg_res": p.numel()})
            for name, size in need.items():
                t = st.get(name)
                if not (isinstance(t, torch.Tensor) and t.dtype == torch.float32 and t.device == p.device
                        and t.is_contiguous() and t.numel() == size):
                    raise ValueError(f"tensor {k}: state '{name}' must be contiguous float32 with {size} "
                                     "elements on the param's device")
            td = self._tensors[k]
            td.p, td.g = _ptr(p), _ptr(g)
            td.grad_dtype = _GRAD_DTYPES[g.dtype]
            td.ndim = p.dim()
            for d, s in enumerate(p.shape):
                td.shape[d] = int(s)
            sd = self._states[k]
            for name in ("exp_avg", "exp_avg_sq_row", "exp_avg_sq_col", "exp_avg_res_row", "exp_avg_res_col",
                         "exp_avg_sq", "exp_avg_res"):
                setattr(sd, name, _ptr(st.get(name)))
        self.workspace_bytes = B.came_workspace_size(self._tensors, n) if n else 0
        self.workspace = (torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=self.device)
                          if n else None)

    def __call__(self, step: int, stream: torch.cuda.Stream | None = None) -> None:
        if self.n == 0:
            return
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        B.came_step(self._tensors, self._states, self.n, int(step), self._hp, _ptr(self.workspace),
                    self.workspace_bytes, int(stream.cuda_stream))


def came_step(params, grads, states, step: int, lr=None, eps=(1e-30, 1e-16), clip_threshold=1.0,
              betas=(0.9, 0.999, 0.9999), weight_decay=0.0, stream=None) -> None:
    """One CAME step over a list of tensors (functional form); states come from
    init_came_state(), t is 1-based.  Use CameStep to marshal once."""
    CameStep(params, grads, states, lr=lr, eps=eps, clip_threshold=clip_threshold, betas=betas,
             weight_decay=weight_decay)(step, stream)


class Came(torch.optim.Optimizer):
    """torch.optim.Optimizer wrapper with the article's DistributedCAME
    defaults (lr must be given); each parameter group is one library call."""

    def __init__(self, params: Iterable, lr=None, eps=(1e-30, 1e-16), clip_threshold=1.0,
                 betas=(0.9, 0.999, 0.9999), weight_decay=0.0):
        make_came_hparams(lr, eps, clip_threshold, betas, weight_decay)
        super().__init__(params, dict(lr=lr, eps=tuple(eps), clip_threshold=clip_threshold, betas=tuple(betas),
                                      weight_decay=weight_decay))
        self._plans = {}

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for gi, group in enumerate(self.param_groups):
            hp = {k: group[k] for k in ("lr", "eps", "clip_threshold", "betas", "weight_decay")}
            by_step = {}
            for p in group["params"]:
                if p.grad is None:
                    continue
                st = self.state[p]
                if not st:
                    st.update(init_came_state([p])[0])
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
                    plan = CameStep(ps, grads, states, **hp)
                    if len(self._plans) > 16:
                        self._plans.clear()
                    self._plans[key] = plan
                plan(t)
        return loss


__all__ = ["Came", "CameStep", "came_step", "init_came_state", "make_came_hparams"]
