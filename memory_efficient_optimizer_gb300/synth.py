"""Seeded synthetic workloads (tensor lists, parameters, gradients).

This module only draws random inputs; it holds none of the optimizer's
arithmetic.  Both the CUDA path and the float64 oracle are fed from it, so the
two see bit-identical inputs.

Workloads (shapes as PyTorch [out, in] weights):
  * ``tiny``        one fp32 weight 256x512 plus one fp32 bias 512;
                    p ~ N(0, 0.02), g ~ N(0, 1e-2), defaults, 10 steps.
  * ``llama_layer`` one Llama-style decoder layer (q/o 4096x4096, k/v
                    1024x4096, gate/up 14336x4096, down 4096x14336, two
                    4096 RMSNorm vectors), fp32 p and g ~ N(0, 1e-3), 10 steps.
  * ``llama_layer_bf16``  the same layer with bf16 gradients (a small case
                    of the kernels the full model runs).
  * ``llama3_8b``   32 such layers + embedding 128256x4096 + lm_head
                    128256x4096 + final norm 4096 (291 tensors,
                    8,030,261,248 values); fp32 p, bf16 g ~ N(0, 1e-3).
  * ``llama3_8b_beta1``  the same shapes with a manual lr of 1e-3,
                    relative_step and scale_parameter off, beta1 0.9, weight
                    decay 0.01; g = Student-t(3 dof) * 1e-3 in bf16 with 1% of
                    the rows of every matrix zeroed (rows fixed per tensor).
  * ``llama3_8b_lamb``, ``llama_layer_lamb``  the LAMB step (article
                    defaults: lr 1e-3, betas (0.9, 0.999), eps 1e-6, bias
                    correction, weight decay 0.01) on the Llama-3-8B list or one
                    decoder layer; fp32 p, bf16 g ~ N(0, 1e-3).
  * ``llama3_8b_came``, ``llama_layer_came``  the CAME step (article
                    defaults: eps (1e-30, 1e-16), clip 1.0, betas (0.9, 0.999,
                    0.9999); lr 1e-4 and weight decay 0.01 chosen here, since
                    the article gives no lr) on the same shapes, bf16 g.
  * ``edge``        1x65536, 65536x1, 4097x3, 3x4097, 17x100003,
                    [8,1024,1024] and 2,000 matrices with H, W ~ U[1, 512];
                    fp32, g ~ N(0, 1e-2), defaults plus beta1 0.9, 10 steps.

Seeds: tensor ``idx`` at step ``t`` draws from a generator seeded with
``base_seed + 1_000_003 * idx + t``; parameters use t = 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

SEED_STRIDE = 1_000_003
ZERO_ROW_SEED_OFFSET = 500_000  # never a real step number

LLAMA_HIDDEN = 4096
LLAMA_FFN = 14336
LLAMA_KV = 1024
LLAMA_VOCAB = 128256
LLAMA_LAYERS = 32


def llama_layer_shapes(hidden=LLAMA_HIDDEN, ffn=LLAMA_FFN, kv=LLAMA_KV):
    return [
        ("q_proj", (hidden, hidden)), ("k_proj", (kv, hidden)), ("v_proj", (kv, hidden)),
        ("o_proj", (hidden, hidden)), ("gate_proj", (ffn, hidden)), ("up_proj", (ffn, hidden)),
        ("down_proj", (hidden, ffn)), ("input_layernorm", (hidden,)),
        ("post_attention_layernorm", (hidden,)),
    ]


def llama3_8b_shapes(layers=LLAMA_LAYERS):
    out = [("embed_tokens", (LLAMA_VOCAB, LLAMA_HIDDEN))]
    for layer in range(layers):
        out += [(f"layers.{layer}.{n}", s) for n, s in llama_layer_shapes()]
    out += [("norm", (LLAMA_HIDDEN,)), ("lm_head", (LLAMA_VOCAB, LLAMA_HIDDEN))]
    return out


def edge_shapes(seed=0, n_small=2000):
    rng = np.random.default_rng(seed + 12345)
    fixed = [(1, 65536), (65536, 1), (4097, 3), (3, 4097), (17, 100003), (8, 1024, 1024)]
    hw = rng.integers(1, 513, size=(n_small, 2))
    out = [(f"edge{k}", s) for k, s in enumerate(fixed)]
    out += [(f"small{k}", (int(h), int(w))) for k, (h, w) in enumerate(hw)]
    return out


@dataclass
class Workload:
    name: str
    shapes: list                      # [(name, shape), ...]
    grad_dtype: torch.dtype
    grad_std: float
    hparams: dict                     # keyword arguments of the optimizer step
    steps: int
    grad_kind: str = "normal"         # "normal" | "student_t_zero_rows"
    param_std: float = 0.02
    description: str = ""
    optimizer: str = "adafactor"      # "adafactor" | "lamb" | "came"
    extra: dict = field(default_factory=dict)

    @property
    def numel(self) -> int:
        return int(sum(int(np.prod(s)) for _, s in self.shapes))


def workload(name: str, seed: int = 0) -> Workload:
    if name == "tiny":
        return Workload(name, [("weight", (256, 512)), ("bias", (512,))], torch.float32, 1e-2,
                        {}, 10, description="256x512 fp32 weight + 512 fp32 bias, defaults")
    if name == "llama_layer":
        return Workload(name, llama_layer_shapes(), torch.float32, 1e-3, {}, 10,
                        description="one Llama-3-8B decoder layer, fp32 p and g, defaults")
    if name == "llama_layer_bf16":
        return Workload(name, llama_layer_shapes(), torch.bfloat16, 1e-3, {}, 10,
                        description="one Llama-3-8B decoder layer, fp32 p, bf16 g, defaults")
    if name == "llama3_8b":
        return Workload(name, llama3_8b_shapes(), torch.bfloat16, 1e-3, {}, 7,
                        description="Llama-3-8B (291 tensors, 8,030,261,248 params), fp32 p, "
                                    "bf16 g, defaults")
    if name == "llama3_8b_beta1":
        return Workload(name, llama3_8b_shapes(), torch.bfloat16, 1e-3,
                        dict(lr=1e-3, relative_step=False, scale_parameter=False, beta1=0.9,
                             weight_decay=0.01), 5, grad_kind="student_t_zero_rows",
                        description="Llama-3-8B shapes, lr 1e-3, beta1 0.9, wd 0.01, "
                                    "Student-t(3) bf16 grads with 1% rows zeroed")
    if name == "llama_layer_bf16_int8":
        return Workload(name, llama_layer_shapes(), torch.bfloat16, 1e-3,
                        dict(lr=1e-3, relative_step=False, scale_parameter=False, beta1=0.9,
                             weight_decay=0.01, exp_avg_int8=True), 5, grad_kind="student_t_zero_rows",
                        description="one Llama-3-8B decoder layer, bf16 grads, beta1 0.9 with the 8-bit exp_avg")
    if name == "llama3_8b_beta1_int8":
        return Workload(name, llama3_8b_shapes(), torch.bfloat16, 1e-3,
                        dict(lr=1e-3, relative_step=False, scale_parameter=False, beta1=0.9,
                             weight_decay=0.01, exp_avg_int8=True), 5, grad_kind="student_t_zero_rows",
                        description="Llama-3-8B shapes, lr 1e-3, beta1 0.9 (8-bit exp_avg, groups of 128), "
                                    "wd 0.01, Student-t(3) bf16 grads with 1% rows zeroed")
    if name == "llama3_8b_lamb":
        return Workload(name, llama3_8b_shapes(), torch.bfloat16, 1e-3, dict(weight_decay=0.01), 5,
                        description="Llama-3-8B shapes, LAMB (lr 1e-3, betas (0.9, 0.999), eps 1e-6, "
                                    "bias correction, wd 0.01), bf16 grads", optimizer="lamb")
    if name == "llama_layer_lamb":
        return Workload(name, llama_layer_shapes(), torch.bfloat16, 1e-3, dict(weight_decay=0.01), 5,
                        description="one Llama-3-8B decoder layer, LAMB (article defaults, wd 0.01), "
                                    "bf16 grads", optimizer="lamb")
    if name == "llama3_8b_came":
        return Workload(name, llama3_8b_shapes(), torch.bfloat16, 1e-3, dict(lr=1e-4, weight_decay=0.01), 5,
                        description="Llama-3-8B shapes, CAME (eps (1e-30, 1e-16), clip 1.0, betas (0.9, 0.999, "
                                    "0.9999), lr 1e-4, wd 0.01), bf16 grads", optimizer="came")
    if name == "llama_layer_came":
        return Workload(name, llama_layer_shapes(), torch.bfloat16, 1e-3, dict(lr=1e-4, weight_decay=0.01), 5,
                        description="one Llama-3-8B decoder layer, CAME (article defaults, lr 1e-4, wd 0.01), "
                                    "bf16 grads", optimizer="came")
    if name == "edge":
        return Workload(name, edge_shapes(seed), torch.float32, 1e-2, dict(beta1=0.9), 10,
                        description="edge shapes + 2,000 small matrices, fp32, beta1 0.9")
    raise KeyError(name)


def _generator(device, seed: int) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def make_param(shape, idx: int, device="cpu", std: float = 0.02, base_seed: int = 0) -> torch.Tensor:
    gen = _generator(device, base_seed + SEED_STRIDE * idx)
    return torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32) * std


def zero_rows(shape, idx: int, base_seed: int = 0) -> torch.Tensor | None:
    """Indices of the matrix rows (dim -2) zeroed in every step; None for ndim < 2."""
    if len(shape) < 2:
        return None
    h = int(shape[-2])
    k = max(1, int(0.01 * h))
    gen = _generator("cpu", base_seed + SEED_STRIDE * idx + ZERO_ROW_SEED_OFFSET)
    return torch.randperm(h, generator=gen)[:k]


def make_grad(shape, idx: int, step: int, device="cpu", std: float = 1e-2,
              dtype=torch.float32, kind: str = "normal", base_seed: int = 0) -> torch.Tensor:
    gen = _generator(device, base_seed + SEED_STRIDE * idx + int(step))
    shape = tuple(shape)
    if kind == "normal":
        g = torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std
    elif kind == "student_t_zero_rows":
        # t(3) = z0 / sqrt((z1^2 + z2^2 + z3^2) / 3)
        z0 = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        chi = torch.zeros(shape, device=device, dtype=torch.float32)
        for _ in range(3):
            z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
            chi.addcmul_(z, z)
            del z
        g = z0.div_(chi.div_(3.0).sqrt_()).mul_(std)
        del chi
        rows = zero_rows(shape, idx, base_seed)
        if rows is not None:
            g.index_fill_(len(shape) - 2, rows.to(device), 0.0)
    else:
        raise KeyError(kind)
    return g.to(dtype)
