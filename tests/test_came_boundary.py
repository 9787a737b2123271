"""The CAME C ABI (include/came.h) without a GPU: defaults, hyper-parameter
checks, workspace sizing and argument errors, all decided on the host before
any CUDA call."""
import pytest

from memory_efficient_optimizer_gb300 import binding as B
from memory_efficient_optimizer_gb300 import build as libbuild
from memory_efficient_optimizer_gb300.came import make_came_hparams


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.load()


def tensors(shapes, dtype=B.ADAF_FLOAT32):
    arr = (B.came_tensor * max(1, len(shapes)))()
    for k, s in enumerate(shapes):
        a = (k + 1) << 30
        arr[k].p, arr[k].g, arr[k].grad_dtype, arr[k].ndim = a, a + (1 << 28), dtype, len(s)
        for d, x in enumerate(s):
            arr[k].shape[d] = x
    return arr


def states(shapes):
    arr = (B.came_state * max(1, len(shapes)))()
    for k, s in enumerate(shapes):
        a = (k + 1) << 34
        for j, name in enumerate(("exp_avg", "exp_avg_sq_row", "exp_avg_sq_col", "exp_avg_res_row",
                                  "exp_avg_res_col", "exp_avg_sq", "exp_avg_res")):
            setattr(arr[k], name, a + (j << 28))
    return arr


def test_defaults_are_the_articles(lib):
    hp = B.came_default_hparams()
    assert (hp.eps1, hp.eps2, hp.clip_threshold) == (1e-30, 1e-16, 1.0)
    assert (hp.beta1, hp.beta2, hp.beta3, hp.weight_decay, hp.lr) == (0.9, 0.999, 0.9999, 0.0, 0.0)
    B.came_validate(hp)


def test_lr_is_required():
    with pytest.raises(ValueError, match="learning rate"):
        make_came_hparams()


@pytest.mark.parametrize("bad,msg", [(dict(lr=-1.0), "learning rate"), (dict(eps=(-1.0, 0.0)), "eps"),
                                     (dict(clip_threshold=0.0), "clip_threshold"),
                                     (dict(betas=(0.9, 0.999, 1.0)), "beta3"),
                                     (dict(weight_decay=-0.5), "weight_decay")])
def test_invalid_hparams_rejected(lib, bad, msg):
    kw = dict(lr=1e-3)
    kw.update(bad)
    with pytest.raises(ValueError, match=msg):
        make_came_hparams(**kw)


def test_workspace_size(lib):
    a = B.came_workspace_size(tensors([(64, 64), (100,)]), 2)
    b = B.came_workspace_size(tensors([(4096, 4096), (100,)]), 2)
    assert 0 < a < b and a % 256 == 0 and b % 256 == 0
    assert B.came_workspace_size(tensors([]), 0) == 0
    bad = tensors([(4, 4)])
    bad[0].ndim = B.ADAF_MAX_NDIM + 1
    with pytest.raises(ValueError, match="ndim"):
        B.came_workspace_size(bad, 1)


def test_step_argument_errors_before_cuda(lib):
    shapes = [(64, 64)]
    hp = make_came_hparams(lr=1e-3)
    need = B.came_workspace_size(tensors(shapes), 1)
    with pytest.raises(ValueError, match="step"):
        B.came_step(tensors(shapes), states(shapes), 1, 0, hp, 1 << 40, need, 0)
    with pytest.raises(ValueError, match="states"):
        B.came_step(tensors(shapes), None, 1, 1, hp, 1 << 40, need, 0)
    st = states(shapes)
    st[0].exp_avg_res_col = 0
    with pytest.raises(ValueError, match="factored state"):
        B.came_step(tensors(shapes), st, 1, 1, hp, 1 << 40, need, 0)
    st1 = states([(10,)])
    st1[0].exp_avg_res = 0
    with pytest.raises(ValueError, match="exp_avg_res"):
        B.came_step(tensors([(10,)]), st1, 1, 1, hp, 1 << 40, need, 0)
    with pytest.raises(ValueError, match="workspace"):
        B.came_step(tensors(shapes), states(shapes), 1, 1, hp, 0, need, 0)
    with pytest.raises(B.AdafactorError, match="workspace"):
        B.came_step(tensors(shapes), states(shapes), 1, 1, hp, 1 << 40, need - 1, 0)


def test_empty_list_is_a_no_op(lib):
    B.came_step(tensors([]), states([]), 0, 1, make_came_hparams(lr=1e-3), 0, 0, 0)


def test_kernel_names(lib):
    assert [B.came_kernel_name(k) for k in range(B.came_num_kernels())] == [
        "k_came_pass_a", "k_came_stats", "k_came_means", "k_came_pass_b", "k_came_clip", "k_came_pass_c",
        "k_came_pass_d", "k_came_panel"]


@pytest.mark.parametrize("dtype", [B.ADAF_FLOAT32, B.ADAF_BFLOAT16])
@pytest.mark.parametrize("misalign", [(), (1, 5, 9), tuple(range(0, 16, 2)), tuple(range(16))])
def test_workspace_size_does_not_depend_on_pointer_alignment(lib, dtype, misalign):
    """The size query has no pointers; the step picks each tensor's path from
    its pointers' alignment.  The query's size must do for every choice: the
    step's own check passes and, without a GPU, the call fails at its first
    CUDA call instead."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    shapes = [(1, 1), (2, 3), (5, 1), (2, 2, 3), (4,), (), (600, 2100), (257, 1025), (1000, 1032), (700, 33),
              (300, 2056), (2, 130, 4096), (131, 4104), (67, 14336), (3, 16384), (129, 5000)]
    t = tensors(shapes, dtype)
    for k in misalign:
        t[k].g += 2 if dtype == B.ADAF_BFLOAT16 else 4
    need = B.came_workspace_size(t, len(shapes))
    with pytest.raises(B.AdafactorError) as e:
        B.came_step(t, states(shapes), len(shapes), 1, make_came_hparams(lr=1e-3), 1 << 40, need, 0)
    assert e.value.status == B.ADAF_ERR_CUDA, str(e.value)
