"""The LAMB C ABI (include/lamb.h) without a GPU: hyper-parameter checks,
workspace sizing and argument errors, all decided on the host before any CUDA
call."""
import ctypes

import pytest

from memory_efficient_optimizer_gb300 import binding as B
from memory_efficient_optimizer_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.load()


def hp(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.0, bias_correction=1)
    d.update(kw)
    return B.lamb_hparams(**d)


def tensors(sizes, dtype=B.ADAF_FLOAT32, base=1 << 20):
    arr = (B.lamb_tensor * max(1, len(sizes)))()
    for k, n in enumerate(sizes):
        a = base * (k + 1) * 64
        arr[k] = B.lamb_tensor(a, a + 16 * base, dtype, n, a + 32 * base, a + 48 * base)
    return arr


def test_article_defaults_validate(lib):
    B.lamb_validate(hp())


@pytest.mark.parametrize("bad,msg", [(dict(lr=-1.0), "learning rate"), (dict(eps=-1e-6), "eps"),
                                     (dict(beta1=1.0), "beta1"), (dict(beta2=-0.5), "beta2"),
                                     (dict(weight_decay=-0.1), "weight_decay"), (dict(lr=float("inf")), "learning rate")])
def test_invalid_hparams_rejected(lib, bad, msg):
    with pytest.raises(ValueError, match=msg):
        B.lamb_validate(hp(**bad))


def test_workspace_size_grows_with_units(lib):
    small = B.lamb_workspace_size(tensors([10, 20]), 2)
    big = B.lamb_workspace_size(tensors([10, 8192 * 100 + 1]), 2)
    assert small > 0 and big > small
    assert small % 256 == 0 and big % 256 == 0
    assert B.lamb_workspace_size(tensors([]), 0) == 0


@pytest.mark.parametrize("sizes,dtype,msg", [([-1], B.ADAF_FLOAT32, "numel"), ([4], 7, "grad_dtype"),
                                             ([1 << 41], B.ADAF_FLOAT32, "2\\^40")])
def test_malformed_lists_rejected(lib, sizes, dtype, msg):
    with pytest.raises((ValueError, B.AdafactorError), match=msg):
        B.lamb_workspace_size(tensors(sizes, dtype), len(sizes))


def test_step_argument_errors_before_cuda(lib):
    t = tensors([100])
    with pytest.raises(ValueError, match="step"):
        B.lamb_step(t, 1, 0, hp(), 1 << 30, 1 << 20, 0)
    null = (B.lamb_tensor * 1)(B.lamb_tensor(0, 0, B.ADAF_FLOAT32, 100, 0, 0))
    with pytest.raises(ValueError, match="NULL"):
        B.lamb_step(null, 1, 1, hp(), 1 << 30, 1 << 20, 0)
    odd = (B.lamb_tensor * 1)(B.lamb_tensor(1 << 30 | 2, 1 << 31, B.ADAF_FLOAT32, 100, 1 << 32, 1 << 33))
    with pytest.raises(ValueError, match="aligned"):
        B.lamb_step(odd, 1, 1, hp(), 1 << 30, 1 << 20, 0)
    with pytest.raises(ValueError, match="workspace"):
        B.lamb_step(t, 1, 1, hp(), 0, 1 << 20, 0)
    need = B.lamb_workspace_size(t, 1)
    with pytest.raises(B.AdafactorError, match="workspace"):
        B.lamb_step(t, 1, 1, hp(), 1 << 30, need - 1, 0)
    with pytest.raises(ValueError, match="beta1"):
        B.lamb_step(t, 1, 1, hp(beta1=2.0), 1 << 30, need, 0)


def test_empty_list_is_a_no_op(lib):
    B.lamb_step(tensors([]), 0, 1, hp(), 0, 0, 0)


def test_kernel_names(lib):
    assert [B.lamb_kernel_name(k) for k in range(B.lamb_num_kernels())] == [
        "k_lamb_moments", "k_lamb_trust", "k_lamb_update"]


@pytest.mark.parametrize("dtype", [B.ADAF_FLOAT32, B.ADAF_BFLOAT16])
@pytest.mark.parametrize("misalign", [(), (1, 3), tuple(range(0, 8, 2)), tuple(range(8))])
def test_workspace_size_does_not_depend_on_pointer_alignment(lib, dtype, misalign):
    """The size query has no pointers; the step picks each tensor's path from
    its pointers' alignment.  The query's size must do for every choice: the
    step's own check passes and, without a GPU, the call fails at its first
    CUDA call instead."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    sizes = [1, 7, 100, 4096, 8192 * 3 + 5, 1 << 20, 33, 8]
    t = tensors(sizes, dtype)
    for k in misalign:
        t[k].g += 2 if dtype == B.ADAF_BFLOAT16 else 4
    need = B.lamb_workspace_size(t, len(sizes))
    with pytest.raises(B.AdafactorError) as e:
        B.lamb_step(t, len(sizes), 1, hp(), 1 << 40, need, 0)
    assert e.value.status == B.ADAF_ERR_CUDA, str(e.value)
