"""PyTorch front end of the CUDA Adafactor step.

PyTorch only provides device memory and streams here: these functions check
and marshal arguments, allocate zeroed state and the workspace, and make one
call into the C library per step.  The library does all of the arithmetic.

Article: Colossal-AI distributed-optimizer article, Step 3 (defaults and
argument rules, beta1 state, factored row/col state for ndim >= 2, full
exp_avg_sq otherwise), Step 5 (the update).
"""
from __future__ import annotations

import ctypes
from typing import Iterable, Sequence

import torch

from . import binding as B

_GRAD_DTYPES = {torch.float32: B.ADAF_FLOAT32, torch.bfloat16: B.ADAF_BFLOAT16}


def make_hparams(lr=None, eps=(1e-30, 1e-3), clip_threshold=1.0, decay_rate=-0.8, beta1=None,
                 weight_decay=0.0, scale_parameter=True, relative_step=True, warmup_init=False,
                 exp_avg_int8=False, param_sq_sum_valid=False) -> B.adaf_hparams:
    """Builds and validates the hyper-parameter struct; invalid values raise
    ValueError with the library's message (e.g. "Cannot combine manual lr and
    relative_step=True options")."""
    if len(tuple(eps)) != 2:
        raise ValueError("eps must be a pair (eps1, eps2)")
    hp = B.adaf_hparams()
    hp.lr = 0.0 if lr is None else float(lr)
    hp.has_lr = 0 if lr is None else 1
    hp.eps1, hp.eps2 = float(eps[0]), float(eps[1])
    hp.clip_threshold = float(clip_threshold)
    hp.decay_rate = float(decay_rate)
    hp.beta1 = 0.0 if beta1 is None else float(beta1)
    hp.has_beta1 = 0 if beta1 is None else 1
    hp.weight_decay = float(weight_decay)
    hp.scale_parameter = int(bool(scale_parameter))
    hp.relative_step = int(bool(relative_step))
    hp.warmup_init = int(bool(warmup_init))
    hp.param_sq_sum_valid = int(bool(param_sq_sum_valid))
    hp.exp_avg_int8 = int(bool(exp_avg_int8))
    B.adafactor_validate(hp)
    return hp


def factored_dims(shape):
    """(B, H, W) for ndim >= 2 (B = product of the leading dims), else None."""
    if len(shape) < 2:
        return None
    lead = 1
    for s in shape[:-2]:
        lead *= int(s)
    return lead, int(shape[-2]), int(shape[-1])


Q8_GROUP = 128  # values per group of the 8-bit first moment, along the last dim


def q8_scale_count(shape) -> int:
    """Group scales of the 8-bit first moment of a tensor: one per 128 values
    along the last dim (a tensor with ndim < 2 is one row)."""
    n = 1
    for s in shape:
        n *= int(s)
    last = int(shape[-1]) if len(shape) >= 2 else n
    rows = n // last if last else 0
    return rows * ((last + Q8_GROUP - 1) // Q8_GROUP)


def init_state(params: Sequence[torch.Tensor], beta1=None, param_sq_sum: bool = True,
               exp_avg_int8: bool = False) -> list:
    """Zeroed optimizer state for each parameter (fp32, on the parameter's device):
    exp_avg_sq_row [*lead, H] and exp_avg_sq_col [*lead, W] for ndim >= 2, a full
    exp_avg_sq otherwise, exp_avg when beta1 is set (or, with exp_avg_int8,
    int8 exp_avg_codes [N] and fp32 exp_avg_scales, one per 128 values along the
    last dim), and a float64 param_sq_sum slot that carries sum(p^2) from one
    step to the next."""
    out = []
    for p in params:
        st = {}
        shape = tuple(p.shape)
        if len(shape) >= 2:
            st["exp_avg_sq_row"] = torch.zeros(shape[:-1], dtype=torch.float32, device=p.device)
            st["exp_avg_sq_col"] = torch.zeros(shape[:-2] + shape[-1:], dtype=torch.float32, device=p.device)
        else:
            st["exp_avg_sq"] = torch.zeros(shape, dtype=torch.float32, device=p.device)
        if beta1 is not None and exp_avg_int8:
            st["exp_avg_codes"] = torch.zeros(shape, dtype=torch.int8, device=p.device)
            st["exp_avg_scales"] = torch.zeros(max(1, q8_scale_count(shape)), dtype=torch.float32, device=p.device)
        elif beta1 is not None:
            st["exp_avg"] = torch.zeros(shape, dtype=torch.float32, device=p.device)
        if param_sq_sum:
            st["param_sq_sum"] = torch.zeros(1, dtype=torch.float64, device=p.device)
        out.append(st)
    return out


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


class AdafactorStep:
    """A marshalled multi-tensor step: the tensor/state descriptor arrays and
    the workspace are built once; every call is one C-library call."""

    def __init__(self, params: Sequence[torch.Tensor], grads: Sequence[torch.Tensor], states: Sequence[dict],
                 **hparams):
        params, grads = list(params), list(grads)
        if len(params) != len(grads) or len(params) != len(states):
            raise ValueError("params, grads and states must have the same length")
        self.hparams = dict(hparams)
        make_hparams(**self.hparams)  # validate early
        self.params, self.grads, self.states = params, grads, list(states)
        n = len(params)
        self.n = n
        self.device = params[0].device if n else None
        self._tensors = (B.adaf_tensor * max(1, n))()
        self._states = (B.adaf_state * max(1, n))()
        for k, (p, g, st) in enumerate(zip(params, grads, self.states)):
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
            for name, t in st.items():
                if name == "param_sq_sum":
                    if t.dtype != torch.float64 or t.device != p.device or t.numel() < 1:
                        raise ValueError(f"tensor {k}: param_sq_sum must be a float64 CUDA tensor")
                elif name == "exp_avg_codes":
                    if not (t.dtype == torch.int8 and t.device == p.device and t.is_contiguous()):
                        raise ValueError(f"tensor {k}: exp_avg_codes must be contiguous int8 on the param's device")
                elif not (t.dtype == torch.float32 and t.device == p.device and t.is_contiguous()):
                    raise ValueError(f"tensor {k}: state '{name}' must be contiguous float32 on the param's device")
            fd = factored_dims(p.shape)
            if fd is not None:
                for name, size in (("exp_avg_sq_row", fd[0] * fd[1]), ("exp_avg_sq_col", fd[0] * fd[2])):
                    if name not in st or st[name].numel() != size:
                        raise ValueError(f"tensor {k}: state '{name}' must have {size} elements")
            elif "exp_avg_sq" not in st or st["exp_avg_sq"].numel() != p.numel():
                raise ValueError(f"tensor {k}: state 'exp_avg_sq' must have {p.numel()} elements")
            if self.hparams.get("beta1") is not None and self.hparams.get("exp_avg_int8"):
                if ("exp_avg_codes" not in st or st["exp_avg_codes"].numel() != p.numel()
                        or "exp_avg_scales" not in st or st["exp_avg_scales"].numel() < q8_scale_count(p.shape)):
                    raise ValueError(f"tensor {k}: exp_avg_int8 needs 'exp_avg_codes' ({p.numel()}) and "
                                     f"'exp_avg_scales' ({q8_scale_count(p.shape)}) states")
            elif self.hparams.get("beta1") is not None and (
                    "exp_avg" not in st or st["exp_avg"].numel() != p.numel()):
                raise ValueError(f"tensor {k}: beta1 is set, state 'exp_avg' must have {p.numel()} elements")
            td = self._tensors[k]
            td.param, td.grad = _ptr(p), _ptr(g)
            td.grad_dtype = _GRAD_DTYPES[g.dtype]
            td.ndim = p.dim()
            for d, s in enumerate(p.shape):
                td.shape[d] = int(s)
            sd = self._states[k]
            sd.exp_avg_sq_row = _ptr(st.get("exp_avg_sq_row"))
            sd.exp_avg_sq_col = _ptr(st.get("exp_avg_sq_col"))
            sd.exp_avg_sq = _ptr(st.get("exp_avg_sq"))
            sd.exp_avg = _ptr(st.get("exp_avg"))
            sd.param_sq_sum = _ptr(st.get("param_sq_sum"))
            sd.exp_avg_codes = _ptr(st.get("exp_avg_codes"))
            sd.exp_avg_scales = _ptr(st.get("exp_avg_scales"))
        self.workspace_bytes = B.adafactor_workspace_size(self._tensors, n) if n else 0
        self.workspace = (torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=self.device)
                          if n else None)
        self._carry = all("param_sq_sum" in st for st in self.states)
        self._versions = None

    def _carry_valid(self) -> bool:
        if not self._carry or self._versions is None:
            return False
        return self._versions == [(p.data_ptr(), p._version) for p in self.params]

    def device_status(self, stream: torch.cuda.Stream | None = None) -> int:
        """Status word of the last step (0 = fine); synchronises with the stream."""
        if self.n == 0:
            return 0
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return B.adafactor_device_status(_ptr(self.workspace), int(stream.cuda_stream))

    def invalidate_param_sq_sum(self) -> None:
        """Forget the carried sum(p^2) (call after changing params behind torch's back)."""
        self._versions = None

    def __call__(self, step: int, stream: torch.cuda.Stream | None = None) -> None:
        if self.n == 0:
            make_hparams(**self.hparams)
            return
        hp = make_hparams(**self.hparams, param_sq_sum_valid=self._carry_valid())
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        B.adafactor_step(self._tensors, self._states, self.n, int(step), hp, _ptr(self.workspace),
                         self.workspace_bytes, int(stream.cuda_stream))
        self._versions = ([(p.data_ptr(), p._version) for p in self.params] if self._carry else None)


class AdafactorShardStep(AdafactorStep):
    """The step for one rank of a group that splits every tensor by rows
    (the distributed step of the article's Step 4).

    params / grads are this rank's row blocks: [..., h_k, W] of a tensor whose
    slices have global_rows[k] rows, or n_k of global_rows[k] elements for
    ndim < 2 (every rank at least one).  states come from init_state(params):
    the row and full second moments are this rank's, the column statistic
    [..., W] is the whole one and stays equal on every rank.  allreduce(t)
    must sum a float64 CUDA tensor in place over the group (for example
    ``torch.distributed.all_reduce``); None means a group of one.  Each call
    is begin, allreduce(exchange round 1), middle, allreduce(exchange round 2), end."""

    def __init__(self, params, grads, states, global_rows, allreduce=None, **hparams):
        super().__init__(params, grads, states, **hparams)
        if len(global_rows) != self.n:
            raise ValueError("global_rows needs one entry per tensor")
        self._shards = (B.adaf_shard * max(1, self.n))()
        for k, (p, gr) in enumerate(zip(self.params, global_rows)):
            if p.numel() == 0:
                raise ValueError(f"tensor {k}: a shard must hold at least one row")
            self._shards[k].global_rows = int(gr)
        self.allreduce = allreduce
        if self.n:
            ws, r1, r2 = B.adafactor_shard_sizes(self._tensors, self._shards, self.n)
            self.workspace_bytes = ws
            self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device)
            self.round1 = torch.zeros(r1 // 8, dtype=torch.float64, device=self.device)
            self.round2 = torch.zeros(r2 // 8, dtype=torch.float64, device=self.device)

    def _args(self, step, stream):
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return ((self._tensors, self._states, self._shards, self.n, int(step), self._hp, _ptr(self.workspace),
                 self.workspace_bytes), int(stream.cuda_stream))

    # The three library calls of one step, for callers that run the exchange
    # themselves: begin(t); sum round1 over the group; middle(t); sum round2;
    # end(t).
    def begin(self, step: int, stream: torch.cuda.Stream | None = None) -> None:
        self._hp = make_hparams(**self.hparams, param_sq_sum_valid=self._carry_valid())
        if self.n:
            args, cs = self._args(step, stream)
            B.adafactor_shard_begin(*args, _ptr(self.round1), cs)

    def middle(self, step: int, stream: torch.cuda.Stream | None = None) -> None:
        if self.n:
            args, cs = self._args(step, stream)
            B.adafactor_shard_middle(*args, _ptr(self.round1), _ptr(self.round2), cs)

    def end(self, step: int, stream: torch.cuda.Stream | None = None) -> None:
        if self.n:
            args, cs = self._args(step, stream)
            B.adafactor_shard_end(*args, _ptr(self.round2), cs)
        self._versions = ([(p.data_ptr(), p._version) for p in self.params] if self._carry else None)

    def __call__(self, step: int, stream: torch.cuda.Stream | None = None) -> None:
        if stream is None and self.n:
            stream = torch.cuda.current_stream(self.device)
        self.begin(step, stream)
        if self.allreduce is not None and self.n:
            with torch.cuda.stream(stream):
                self.allreduce(self.round1)
        self.middle(step, stream)
        if self.allreduce is not None and self.n:
            with torch.cuda.stream(stream):
                self.allreduce(self.round2)
        self.end(step, stream)


def adafactor_step(params, grads, states, step: int, lr=None, eps=(1e-30, 1e-3), clip_threshold=1.0,
                   decay_rate=-0.8, beta1=None, weight_decay=0.0, scale_parameter=True, relative_step=True,
                   warmup_init=False, exp_avg_int8=False, stream=None) -> None:
    """One Adafactor step over a list of tensors (functional form).  States come
    from init_state(); the step number t is 1-based.  Marshals every call; use
    AdafactorStep to marshal once and call many times."""
    hparams = dict(lr=lr, eps=eps, clip_threshold=clip_threshold, decay_rate=decay_rate, beta1=beta1,
                   weight_decay=weight_decay, scale_parameter=scale_parameter, relative_step=relative_step,
                   warmup_init=warmup_init, exp_avg_int8=exp_avg_int8)
    make_hparams(**hparams)
    AdafactorStep(params, grads, states, **hparams)(step, stream)


class Adafactor(torch.optim.Optimizer):
    """torch.optim.Optimizer wrapper with the article's Adafactor defaults.

    Each parameter group is stepped with one call into the library (one
    launch sequence for all of its tensors)."""

    def __init__(self, params: Iterable, lr=None, eps=(1e-30, 1e-3), clip_threshold=1.0, decay_rate=-0.8,
                 beta1=None, weight_decay=0.0, scale_parameter=True, relative_step=True, warmup_init=False,
                 exp_avg_int8=False):
        make_hparams(lr=lr, eps=eps, clip_threshold=clip_threshold, decay_rate=decay_rate, beta1=beta1,
                     weight_decay=weight_decay, scale_parameter=scale_parameter, relative_step=relative_step,
                     warmup_init=warmup_init, exp_avg_int8=exp_avg_int8)
        defaults = dict(lr=lr, eps=eps, clip_threshold=clip_threshold, decay_rate=decay_rate, beta1=beta1,
                        weight_decay=weight_decay, scale_parameter=scale_parameter, relative_step=relative_step,
                        warmup_init=warmup_init, exp_avg_int8=exp_avg_int8)
        super().__init__(params, defaults)
        self._plans = {}

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for gi, group in enumerate(self.param_groups):
            hp = {k: group[k] for k in ("lr", "eps", "clip_threshold", "decay_rate", "beta1", "weight_decay",
                                        "scale_parameter", "relative_step", "warmup_init", "exp_avg_int8")}
            by_step = {}
            for p in group["params"]:
                if p.grad is None:
                    continue
                st = self.state[p]
                if not st:
                    st.update(init_state([p], beta1=hp["beta1"], exp_avg_int8=hp["exp_avg_int8"])[0])
                    st["step"] = 0
                st["step"] += 1
                by_step.setdefault(st["step"], []).append(p)
            for t, ps in by_step.items():
                grads = [p.grad for p in ps]
                key = (gi, t if len(by_step) > 1 else None, tuple(p.data_ptr() for p in ps),
                       tuple(g.data_ptr() for g in grads), tuple(sorted(hp.items(), key=lambda kv: kv[0])).__repr__())
                plan = self._plans.get(key)
                if plan is None:
                    states = [{k: v for k, v in self.state[p].items() if k != "step"} for p in ps]
                    plan = AdafactorStep(ps, grads, states, **hp)
                    if len(self._plans) > 16:
                        self._plans.clear()
                    self._plans[key] = plan
                plan(t)
        return loss
