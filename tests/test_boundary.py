"""The C-ABI boundary without a GPU: the library loads, exports every entry
point declared in include/*.h, and rejects bad arguments before any
CUDA call (so a failing call changes nothing)."""
import ctypes
import os
import re

import pytest

from memory_efficient_optimizer_gb300 import binding as B
from memory_efficient_optimizer_gb300 import build as libbuild
from memory_efficient_optimizer_gb300.optim import make_hparams

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b((?:adafactor|lamb|came)_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = declared_functions()
    assert declared, "no declarations found"
    assert declared == set(B.EXPORTS) | set(B.LAMB_EXPORTS) | set(B.CAME_EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_defaults_are_the_articles(lib):
    hp = B.adafactor_default_hparams()
    assert (hp.has_lr, hp.eps1, hp.eps2, hp.clip_threshold, hp.decay_rate) == (0, 1e-30, 1e-3, 1.0, -0.8)
    assert (hp.has_beta1, hp.weight_decay, hp.scale_parameter, hp.relative_step, hp.warmup_init) == (0, 0.0, 1, 1, 0)
    B.adafactor_validate(hp)


@pytest.mark.parametrize("kwargs,msg", [
    (dict(lr=1e-3), "Cannot combine manual lr and relative_step=True options"),
    (dict(lr=1e-3, relative_step=False, warmup_init=True), "warmup_init"),
    (dict(relative_step=False), "manual lr"),
    (dict(clip_threshold=0.0), "clip_threshold"),
    (dict(beta1=1.0), "beta1"),
    (dict(weight_decay=-1.0), "weight_decay"),
    (dict(eps=(float("nan"), 1e-3)), "eps"),
])
def test_invalid_hparams_raise_valueerror(lib, kwargs, msg):
    with pytest.raises(ValueError, match=msg):
        make_hparams(**kwargs)


def fake_list(shapes, dtype=B.ADAF_FLOAT32, addr=1 << 20):
    n = len(shapes)
    ts = (B.adaf_tensor * n)()
    ss = (B.adaf_state * n)()
    for k, shp in enumerate(shapes):
        ts[k].param = addr + k * (1 << 16)
        ts[k].grad = addr + (1 << 30) + k * (1 << 16)
        ts[k].grad_dtype = dtype
        ts[k].ndim = len(shp)
        for d, s in enumerate(shp):
            ts[k].shape[d] = s
        ss[k].exp_avg_sq_row = addr + (2 << 30)
        ss[k].exp_avg_sq_col = addr + (3 << 30)
        ss[k].exp_avg_sq = addr + (4 << 30)
    return ts, ss


def call_step(ts, ss, n, step=1, hp=None, ws=1 << 40, wsb=1 << 40):
    hp = hp or B.adafactor_default_hparams()
    return B.load().adafactor_step(ts, ss, n, step, ctypes.byref(hp), ctypes.c_void_p(ws), wsb, None)


def test_workspace_size_scales_with_the_list(lib):
    ts, _ = fake_list([(256, 512), (512,)])
    small = B.adafactor_workspace_size(ts, 2)
    ts2, _ = fake_list([(4096, 4096), (4096,)])
    big = B.adafactor_workspace_size(ts2, 2)
    assert 0 < small < big
    # column partials of a 4096x4096 matrix alone: 16 row blocks x 4096 floats
    assert big >= 16 * 4096 * 4


def test_step_argument_errors_before_any_cuda_call(lib):
    ts, ss = fake_list([(8, 16), (16,)])
    assert call_step(ts, ss, 2, step=0) == B.ADAF_ERR_INVALID_ARGUMENT
    assert "step" in B.adafactor_last_error()
    hp = B.adafactor_default_hparams()
    hp.has_lr, hp.lr = 1, 1e-3
    assert call_step(ts, ss, 2, hp=hp) == B.ADAF_ERR_INVALID_ARGUMENT
    assert B.adafactor_last_error() == "Cannot combine manual lr and relative_step=True options"
    assert B.load().adafactor_step(ts, None, 2, 1, ctypes.byref(B.adafactor_default_hparams()),
                                   ctypes.c_void_p(1 << 40), 1 << 40, None) == B.ADAF_ERR_INVALID_ARGUMENT
    # beta1 without exp_avg
    hp = B.adafactor_default_hparams()
    hp.has_beta1, hp.beta1 = 1, 0.9
    assert call_step(ts, ss, 2, hp=hp) == B.ADAF_ERR_INVALID_ARGUMENT
    assert "exp_avg" in B.adafactor_last_error()
    # factored tensor without its row state
    ts1, ss1 = fake_list([(8, 16)])
    ss1[0].exp_avg_sq_row = 0
    assert call_step(ts1, ss1, 1) == B.ADAF_ERR_INVALID_ARGUMENT
    # misaligned param and bad dtype / ndim / shape
    ts1, ss1 = fake_list([(8, 16)])
    ts1[0].param += 2
    assert call_step(ts1, ss1, 1) == B.ADAF_ERR_INVALID_ARGUMENT
    ts1, ss1 = fake_list([(8, 16)], dtype=7)
    assert call_step(ts1, ss1, 1) == B.ADAF_ERR_INVALID_ARGUMENT
    ts1, ss1 = fake_list([(8, 16)])
    ts1[0].ndim = 9
    assert call_step(ts1, ss1, 1) == B.ADAF_ERR_INVALID_ARGUMENT
    ts1, ss1 = fake_list([(8, -16)])
    assert call_step(ts1, ss1, 1) == B.ADAF_ERR_INVALID_ARGUMENT
    # carry flag without a carry slot
    hp = B.adafactor_default_hparams()
    hp.param_sq_sum_valid = 1
    assert call_step(ts, ss, 2, hp=hp) == B.ADAF_ERR_INVALID_ARGUMENT
    # workspace checks
    assert call_step(ts, ss, 2, ws=0) == B.ADAF_ERR_INVALID_ARGUMENT
    assert call_step(ts, ss, 2, ws=(1 << 40) + 8) == B.ADAF_ERR_INVALID_ARGUMENT
    need = B.adafactor_workspace_size(ts, 2)
    assert call_step(ts, ss, 2, wsb=need - 1) == B.ADAF_ERR_WORKSPACE_TOO_SMALL
    assert str(need) in B.adafactor_last_error()


# Shapes of every class (flat, rows, wide, tiled vector and element-wise, 1D)
SIZE_SHAPES = [(1, 1), (2, 3), (3, 2), (1, 5), (5, 1), (2, 2, 3), (4,), (), (600, 2100), (257, 1025), (3, 4097),
               (1000, 1032), (2, 3, 520, 264), (7, 1, 9), (1, 65536), (9000,), (700, 33), (300, 1023), (513, 7),
               (260, 1), (1030, 3), (130, 100), (91, 200), (50, 512), (40, 513), (33, 32), (17, 16), (300, 2056),
               (2, 130, 4096), (131, 4104), (67, 14336), (3, 16384), (5, 16392), (9, 2040), (7, 9000), (129, 5000),
               (1, 8192)]


@pytest.mark.parametrize("dtype", [B.ADAF_FLOAT32, B.ADAF_BFLOAT16])
@pytest.mark.parametrize("misalign", [(), (1, 5, 9), tuple(range(0, 20, 2)), tuple(range(20))])
def test_workspace_size_does_not_depend_on_pointer_alignment(lib, dtype, misalign):
    """The size query has no pointers; the step picks each tensor's path from
    its pointers' alignment (16-byte aligned rows take the vector, row-chunk
    and flat paths, others the element-wise one).  The query's size must do
    for every such choice: the step's own check passes (and, without a GPU,
    the call then fails at its first CUDA call instead)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    ts, ss = fake_list(SIZE_SHAPES, dtype=dtype)
    esz = 2 if dtype == B.ADAF_BFLOAT16 else 4
    for k in misalign:
        ts[k].grad += esz  # still aligned to its element, no longer to 16 bytes
    need = B.adafactor_workspace_size(ts, len(SIZE_SHAPES))
    assert call_step(ts, ss, len(SIZE_SHAPES), wsb=need) == B.ADAF_ERR_CUDA, B.adafactor_last_error()
    sh = fake_shards([s[-2] * 2 if len(s) >= 2 else (s[0] if s else 1) * 2 for s in SIZE_SHAPES])
    ws, r1, r2 = B.adafactor_shard_sizes(ts, sh, len(SIZE_SHAPES))
    rounds = [1 << 41]
    assert call_shard("adafactor_shard_begin", ts, ss, sh, len(SIZE_SHAPES), rounds, wsb=ws) == B.ADAF_ERR_CUDA, \
        B.adafactor_last_error()


def test_empty_list_and_empty_tensors_are_no_ops(lib):
    ts, ss = fake_list([(0, 5), (0,)])
    ts[0].param = ts[0].grad = ts[1].param = ts[1].grad = 0  # empty tensors may have no storage
    assert call_step(ts, ss, 2, ws=0, wsb=0) == B.ADAF_OK
    assert B.load().adafactor_step(None, None, 0, 1, ctypes.byref(B.adafactor_default_hparams()),
                                   None, 0, None) == B.ADAF_OK


def test_valid_call_without_gpu_reports_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    ts, ss = fake_list([(8, 16)])
    assert call_step(ts, ss, 1) == B.ADAF_ERR_CUDA
    assert B.adafactor_last_error()


def fake_shards(rows):
    sh = (B.adaf_shard * len(rows))()
    for k, r in enumerate(rows):
        sh[k].global_rows = r
    return sh


def call_shard(fn, ts, ss, sh, n, rounds, step=1, ws=1 << 40, wsb=1 << 40):
    hp = B.adafactor_default_hparams()
    return getattr(B.load(), fn)(ts, ss, sh, n, step, ctypes.byref(hp), ctypes.c_void_p(ws), wsb,
                                 *[ctypes.c_void_p(r) for r in rounds], None)


def test_shard_sizes_and_argument_errors_before_any_cuda_call(lib):
    """Row-sharded entry points: the exchange sizes depend on the leading dims
    and W only (not on a shard's rows), and every argument error is reported
    before the first CUDA call."""
    shapes = [(300, 2056), (2, 130, 4096), (9000,)]
    ts, ss = fake_list(shapes)
    sh = fake_shards([900, 390, 27000])
    ws, r1, r2 = B.adafactor_shard_sizes(ts, sh, 3)
    assert r1 == 8 * (2056 + 2 * 4096 + 1 + 2 + 3) and r2 == 8 * 3
    assert ws >= B.adafactor_workspace_size(ts, 3)
    other, _ = fake_list([(17, 2056), (2, 1, 4096), (5,)])
    assert B.adafactor_shard_sizes(other, sh, 3)[1:] == (r1, r2)
    R1, R2 = 1 << 41, 1 << 42
    inv = B.ADAF_ERR_INVALID_ARGUMENT
    assert call_shard("adafactor_shard_begin", ts, ss, None, 3, [R1]) == inv
    assert "shards" in B.adafactor_last_error()
    assert call_shard("adafactor_shard_begin", ts, ss, sh, 3, [0]) == inv
    assert "round1" in B.adafactor_last_error()
    assert call_shard("adafactor_shard_middle", ts, ss, sh, 3, [R1, 0]) == inv
    assert "round2" in B.adafactor_last_error()
    assert call_shard("adafactor_shard_end", ts, ss, sh, 3, [R2 + 4]) == inv
    assert "round2" in B.adafactor_last_error()
    small = fake_shards([100, 390, 27000])  # fewer global rows than the shard holds
    assert call_shard("adafactor_shard_begin", ts, ss, small, 3, [R1]) == inv
    assert "global_rows" in B.adafactor_last_error()
    empty, ess = fake_list([(0, 2056), (2, 130, 4096), (9000,)])
    assert call_shard("adafactor_shard_begin", empty, ess, sh, 3, [R1]) == inv
    assert "at least one row" in B.adafactor_last_error()
    with pytest.raises(ValueError, match="global_rows"):
        B.adafactor_shard_sizes(ts, small, 3)


def test_kernel_names(lib):
    names = [B.adafactor_kernel_name(k) for k in range(B.adafactor_num_kernels())]
    assert len(names) == 31 and len(set(names)) == 31
    for kind in ("k_pass1", "k_pass2", "k_apply"):
        for cls in ("vec_bf16", "vec_f32", "elem_bf16", "elem_f32", "1d", "rows_bf16", "wide_bf16", "flat_bf16",
                    "flat_f32"):
            assert f"{kind}[{cls}]" in names
    assert {"k_stats", "k_scalars", "k_clip", "k_psq"} <= set(names)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        B.load()
