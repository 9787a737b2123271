"""ctypes binding of the C ABI in include/adafactor.h, include/lamb.h and
include/came.h (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: all of the step runs in the CUDA library.  Loading
fails loudly when the library has not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

ADAF_OK = 0
ADAF_ERR_INVALID_ARGUMENT = 1
ADAF_ERR_UNSUPPORTED = 2
ADAF_ERR_WORKSPACE_TOO_SMALL = 3
ADAF_ERR_CUDA = 4
ADAF_FLOAT32 = 0
ADAF_BFLOAT16 = 1
ADAF_MAX_NDIM = 8
ADAF_DEVICE_WAIT_TIMEOUT = 1

# Entry points declared in include/adafactor.h.
EXPORTS = (
    "adafactor_default_hparams", "adafactor_validate", "adafactor_workspace_size",
    "adafactor_step", "adafactor_device_status", "adafactor_last_error", "adafactor_release_cache",
    "adafactor_profile_enable", "adafactor_profile_read", "adafactor_num_kernels",
    "adafactor_kernel_name", "adafactor_step_noalloc", "adafactor_noalloc_device_status",
    "adafactor_debug_stall_copies",
    "adafactor_shard_sizes", "adafactor_shard_begin", "adafactor_shard_middle", "adafactor_shard_end",
)
# Entry points declared in include/came.h.
CAME_EXPORTS = (
    "came_default_hparams", "came_validate", "came_workspace_size", "came_step", "came_profile_enable",
    "came_profile_read", "came_num_kernels", "came_kernel_name",
)
# Entry points declared in include/lamb.h.
LAMB_EXPORTS = (
    "lamb_validate", "lamb_workspace_size", "lamb_step", "lamb_trust_ratios", "lamb_profile_enable",
    "lamb_profile_read", "lamb_num_kernels", "lamb_kernel_name",
)


class adaf_tensor(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("grad_dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * ADAF_MAX_NDIM)]


class adaf_state(ctypes.Structure):
    _fields_ = [("exp_avg_sq_row", ctypes.c_void_p), ("exp_avg_sq_col", ctypes.c_void_p),
                ("exp_avg_sq", ctypes.c_void_p), ("exp_avg", ctypes.c_void_p),
                ("param_sq_sum", ctypes.c_void_p),
                ("exp_avg_codes", ctypes.c_void_p), ("exp_avg_scales", ctypes.c_void_p)]


class adaf_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("has_lr", ctypes.c_int32),
                ("eps1", ctypes.c_double), ("eps2", ctypes.c_double),
                ("clip_threshold", ctypes.c_double), ("decay_rate", ctypes.c_double),
                ("beta1", ctypes.c_double), ("has_beta1", ctypes.c_int32),
                ("weight_decay", ctypes.c_double), ("scale_parameter", ctypes.c_int32),
                ("relative_step", ctypes.c_int32), ("warmup_init", ctypes.c_int32),
                ("param_sq_sum_valid", ctypes.c_int32), ("exp_avg_int8", ctypes.c_int32)]


class adaf_shard(ctypes.Structure):
    _fields_ = [("global_rows", ctypes.c_int64)]


class lamb_tensor(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("grad_dtype", ctypes.c_int32),
                ("numel", ctypes.c_int64), ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p)]


class lamb_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("bias_correction", ctypes.c_int32)]


class came_tensor(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("grad_dtype", ctypes.c_int32),
                ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * ADAF_MAX_NDIM)]


class came_state(ctypes.Structure):
    _fields_ = [("exp_avg", ctypes.c_void_p), ("exp_avg_sq_row", ctypes.c_void_p),
                ("exp_avg_sq_col", ctypes.c_void_p), ("exp_avg_res_row", ctypes.c_void_p),
                ("exp_avg_res_col", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("exp_avg_res", ctypes.c_void_p)]


class came_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("eps1", ctypes.c_double), ("eps2", ctypes.c_double),
                ("clip_threshold", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("beta3", ctypes.c_double), ("weight_decay", ctypes.c_double)]


class AdafactorError(RuntimeError):
    """A non-zero adaf_status other than an argument error."""

    def __init__(self, status: int, message: str):
        super().__init__(f"adafactor status {status}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Loads libmeo_adafactor.so; raises if it is missing (no CPU fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m memory_efficient_optimizer_gb300.build` "
                    "(there is no fallback implementation)")
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER
        lib.adafactor_default_hparams.restype = None
        lib.adafactor_default_hparams.argtypes = [P(adaf_hparams)]
        lib.adafactor_validate.restype = ctypes.c_int
        lib.adafactor_validate.argtypes = [P(adaf_hparams)]
        lib.adafactor_workspace_size.restype = ctypes.c_int
        lib.adafactor_workspace_size.argtypes = [P(adaf_tensor), ctypes.c_int32, P(ctypes.c_size_t)]
        lib.adafactor_step.restype = ctypes.c_int
        lib.adafactor_step.argtypes = [P(adaf_tensor), P(adaf_state), ctypes.c_int32, ctypes.c_int64,
                                       P(adaf_hparams), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.adafactor_step_noalloc.restype = ctypes.c_int
        lib.adafactor_step_noalloc.argtypes = [P(adaf_tensor), P(adaf_state), ctypes.c_int32, ctypes.c_int64,
                                               P(adaf_hparams), ctypes.c_void_p]
        lib.adafactor_noalloc_device_status.restype = ctypes.c_int
        lib.adafactor_noalloc_device_status.argtypes = [ctypes.c_void_p, P(ctypes.c_int32)]
        lib.adafactor_device_status.restype = ctypes.c_int
        lib.adafactor_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, P(ctypes.c_int32)]
        lib.adafactor_debug_stall_copies.restype = None
        lib.adafactor_debug_stall_copies.argtypes = [ctypes.c_int32]
        lib.adafactor_last_error.restype = ctypes.c_char_p
        lib.adafactor_last_error.argtypes = []
        lib.adafactor_release_cache.restype = None
        lib.adafactor_release_cache.argtypes = []
        lib.adafactor_profile_enable.restype = ctypes.c_int
        lib.adafactor_profile_enable.argtypes = [ctypes.c_int32]
        lib.adafactor_profile_read.restype = ctypes.c_int
        lib.adafactor_profile_read.argtypes = [P(ctypes.c_double), P(ctypes.c_int64), ctypes.c_int32]
        lib.adafactor_num_kernels.restype = ctypes.c_int32
        lib.adafactor_num_kernels.argtypes = []
        lib.adafactor_kernel_name.restype = ctypes.c_char_p
        lib.adafactor_kernel_name.argtypes = [ctypes.c_int32]
        lib.adafactor_shard_sizes.restype = ctypes.c_int
        lib.adafactor_shard_sizes.argtypes = [P(adaf_tensor), P(adaf_shard), ctypes.c_int32, P(ctypes.c_size_t),
                                              P(ctypes.c_size_t), P(ctypes.c_size_t)]
        shard_head = [P(adaf_tensor), P(adaf_state), P(adaf_shard), ctypes.c_int32, ctypes.c_int64,
                      P(adaf_hparams), ctypes.c_void_p, ctypes.c_size_t]
        lib.adafactor_shard_begin.restype = ctypes.c_int
        lib.adafactor_shard_begin.argtypes = shard_head + [ctypes.c_void_p, ctypes.c_void_p]
        lib.adafactor_shard_middle.restype = ctypes.c_int
        lib.adafactor_shard_middle.argtypes = shard_head + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.adafactor_shard_end.restype = ctypes.c_int
        lib.adafactor_shard_end.argtypes = shard_head + [ctypes.c_void_p, ctypes.c_void_p]
        lib.came_default_hparams.restype = None
        lib.came_default_hparams.argtypes = [P(came_hparams)]
        lib.came_validate.restype = ctypes.c_int
        lib.came_validate.argtypes = [P(came_hparams)]
        lib.came_workspace_size.restype = ctypes.c_int
        lib.came_workspace_size.argtypes = [P(came_tensor), ctypes.c_int32, P(ctypes.c_size_t)]
        lib.came_step.restype = ctypes.c_int
        lib.came_step.argtypes = [P(came_tensor), P(came_state), ctypes.c_int32, ctypes.c_int64, P(came_hparams),
                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.came_profile_enable.restype = ctypes.c_int
        lib.came_profile_enable.argtypes = [ctypes.c_int32]
        lib.came_profile_read.restype = ctypes.c_int
        lib.came_profile_read.argtypes = [P(ctypes.c_double), P(ctypes.c_int64), ctypes.c_int32]
        lib.came_num_kernels.restype = ctypes.c_int32
        lib.came_num_kernels.argtypes = []
        lib.came_kernel_name.restype = ctypes.c_char_p
        lib.came_kernel_name.argtypes = [ctypes.c_int32]
        lib.lamb_validate.restype = ctypes.c_int
        lib.lamb_validate.argtypes = [P(lamb_hparams)]
        lib.lamb_workspace_size.restype = ctypes.c_int
        lib.lamb_workspace_size.argtypes = [P(lamb_tensor), ctypes.c_int32, P(ctypes.c_size_t)]
        lib.lamb_step.restype = ctypes.c_int
        lib.lamb_step.argtypes = [P(lamb_tensor), ctypes.c_int32, ctypes.c_int64, P(lamb_hparams),
                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.lamb_trust_ratios.restype = ctypes.c_int
        lib.lamb_trust_ratios.argtypes = [ctypes.c_void_p, ctypes.c_int32, P(ctypes.c_double), ctypes.c_void_p]
        lib.lamb_profile_enable.restype = ctypes.c_int
        lib.lamb_profile_enable.argtypes = [ctypes.c_int32]
        lib.lamb_profile_read.restype = ctypes.c_int
        lib.lamb_profile_read.argtypes = [P(ctypes.c_double), P(ctypes.c_int64), ctypes.c_int32]
        lib.lamb_num_kernels.restype = ctypes.c_int32
        lib.lamb_num_kernels.argtypes = []
        lib.lamb_kernel_name.restype = ctypes.c_char_p
        lib.lamb_kernel_name.argtypes = [ctypes.c_int32]
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status == ADAF_OK:
        return
    msg = adafactor_last_error()
    if status == ADAF_ERR_INVALID_ARGUMENT:
        raise ValueError(msg)
    raise AdafactorError(status, msg)


def adafactor_default_hparams() -> adaf_hparams:
    hp = adaf_hparams()
    load().adafactor_default_hparams(ctypes.byref(hp))
    return hp


def adafactor_validate(hp: adaf_hparams) -> None:
    _check(load().adafactor_validate(ctypes.byref(hp)))


def adafactor_workspace_size(tensors, n: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().adafactor_workspace_size(tensors, int(n), ctypes.byref(out)))
    return int(out.value)


def adafactor_step(tensors, states, n: int, step: int, hp: adaf_hparams, workspace: int,
                   workspace_bytes: int, stream: int) -> None:
    _check(load().adafactor_step(tensors, states, int(n), int(step), ctypes.byref(hp),
                                 ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes),
                                 ctypes.c_void_p(stream)))


def adafactor_step_noalloc(tensors, states, n: int, step: int, hp: adaf_hparams, stream: int) -> None:
    """The step with the library's fixed scratch area (no workspace argument)."""
    _check(load().adafactor_step_noalloc(tensors, states, int(n), int(step), ctypes.byref(hp),
                                         ctypes.c_void_p(stream)))


def adafactor_shard_sizes(tensors, shards, n: int):
    """(workspace bytes, round-1 bytes, round-2 bytes) of a row-sharded step."""
    ws, r1, r2 = ctypes.c_size_t(0), ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().adafactor_shard_sizes(tensors, shards, int(n), ctypes.byref(ws), ctypes.byref(r1),
                                        ctypes.byref(r2)))
    return int(ws.value), int(r1.value), int(r2.value)


def adafactor_shard_begin(tensors, states, shards, n: int, step: int, hp: adaf_hparams, workspace: int,
                          workspace_bytes: int, round1: int, stream: int) -> None:
    _check(load().adafactor_shard_begin(tensors, states, shards, int(n), int(step), ctypes.byref(hp),
                                        ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes),
                                        ctypes.c_void_p(round1), ctypes.c_void_p(stream)))


def adafactor_shard_middle(tensors, states, shards, n: int, step: int, hp: adaf_hparams, workspace: int,
                           workspace_bytes: int, round1: int, round2: int, stream: int) -> None:
    _check(load().adafactor_shard_middle(tensors, states, shards, int(n), int(step), ctypes.byref(hp),
                                         ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes),
                                         ctypes.c_void_p(round1), ctypes.c_void_p(round2), ctypes.c_void_p(stream)))


def adafactor_shard_end(tensors, states, shards, n: int, step: int, hp: adaf_hparams, workspace: int,
                        workspace_bytes: int, round2: int, stream: int) -> None:
    _check(load().adafactor_shard_end(tensors, states, shards, int(n), int(step), ctypes.byref(hp),
                                      ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes),
                                      ctypes.c_void_p(round2), ctypes.c_void_p(stream)))


def adafactor_device_status(workspace: int, stream: int) -> int:
    out = ctypes.c_int32(0)
    _check(load().adafactor_device_status(ctypes.c_void_p(workspace), ctypes.c_void_p(stream), ctypes.byref(out)))
    return int(out.value)


def adafactor_noalloc_device_status(stream: int) -> int:
    """Status word of the last adafactor_step_noalloc() on the current device."""
    out = ctypes.c_int32(0)
    _check(load().adafactor_noalloc_device_status(ctypes.c_void_p(stream), ctypes.byref(out)))
    return int(out.value)


def adafactor_debug_stall_copies(on: bool) -> None:
    """Testing hook: make the bulk-copy producers issue nothing (see the header)."""
    load().adafactor_debug_stall_copies(1 if on else 0)


def adafactor_last_error() -> str:
    return load().adafactor_last_error().decode(errors="replace")


def adafactor_release_cache() -> None:
    load().adafactor_release_cache()


def adafactor_profile_enable(on: bool) -> None:
    _check(load().adafactor_profile_enable(1 if on else 0))


def adafactor_num_kernels() -> int:
    return int(load().adafactor_num_kernels())


def adafactor_kernel_name(k: int) -> str:
    return load().adafactor_kernel_name(int(k)).decode()


def adafactor_profile_read() -> dict:
    """{kernel name: (total ms, launches)} for the events recorded since the last read."""
    nk = adafactor_num_kernels()
    ms = (ctypes.c_double * nk)()
    launches = (ctypes.c_int64 * nk)()
    _check(load().adafactor_profile_read(ms, launches, nk))
    return {adafactor_kernel_name(k): (float(ms[k]), int(launches[k])) for k in range(nk)}


# ---- LAMB (include/lamb.h) --------------------------------------------------

def lamb_validate(hp: lamb_hparams) -> None:
    _check(load().lamb_validate(ctypes.byref(hp)))


def lamb_workspace_size(tensors, n: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().lamb_workspace_size(tensors, int(n), ctypes.byref(out)))
    return int(out.value)


def lamb_step(tensors, n: int, step: int, hp: lamb_hparams, workspace: int, workspace_bytes: int,
              stream: int) -> None:
    _check(load().lamb_step(tensors, int(n), int(step), ctypes.byref(hp), ctypes.c_void_p(workspace),
                            ctypes.c_size_t(workspace_bytes), ctypes.c_void_p(stream)))


def lamb_trust_ratios(workspace: int, n: int, stream: int) -> list:
    out = (ctypes.c_double * max(1, int(n)))()
    _check(load().lamb_trust_ratios(ctypes.c_void_p(workspace), int(n), out, ctypes.c_void_p(stream)))
    return [float(out[k]) for k in range(int(n))]


def lamb_profile_enable(on: bool) -> None:
    _check(load().lamb_profile_enable(1 if on else 0))


def lamb_num_kernels() -> int:
    return int(load().lamb_num_kernels())


def lamb_kernel_name(k: int) -> str:
    return load().lamb_kernel_name(int(k)).decode()


def lamb_profile_read() -> dict:
    """{kernel name: (total ms, launches)} for the LAMB events recorded since the last read."""
    nk = lamb_num_kernels()
    ms = (ctypes.c_double * nk)()
    launches = (ctypes.c_int64 * nk)()
    _check(load().lamb_profile_read(ms, launches, nk))
    return {lamb_kernel_name(k): (float(ms[k]), int(launches[k])) for k in range(nk)}


# ---- CAME (include/came.h) --------------------------------------------------

def came_default_hparams() -> came_hparams:
    hp = came_hparams()
    load().came_default_hparams(ctypes.byref(hp))
    return hp


def came_validate(hp: came_hparams) -> None:
    _check(load().came_validate(ctypes.byref(hp)))


def came_workspace_size(tensors, n: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load().came_workspace_size(tensors, int(n), ctypes.byref(out)))
    return int(out.value)


def came_step(tensors, states, n: int, step: int, hp: came_hparams, workspace: int, workspace_bytes: int,
              stream: int) -> None:
    _check(load().came_step(tensors, states, int(n), int(step), ctypes.byref(hp), ctypes.c_void_p(workspace),
                            ctypes.c_size_t(workspace_bytes), ctypes.c_void_p(stream)))


def came_profile_enable(on: bool) -> None:
    _check(load().came_profile_enable(1 if on else 0))


def came_num_kernels() -> int:
    return int(load().came_num_kernels())


def came_kernel_name(k: int) -> str:
    return load().came_kernel_name(int(k)).decode()


def came_profile_read() -> dict:
    """{kernel name: (total ms, launches)} for the CAME events recorded since the last read."""
    nk = came_num_kernels()
    ms = (ctypes.c_double * nk)()
    launches = (ctypes.c_int64 * nk)()
    _check(load().came_profile_read(ms, launches, nk))
    return {came_kernel_name(k): (float(ms[k]), int(launches[k])) for k in range(nk)}
