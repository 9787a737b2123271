"""Float64 CPU oracle for the CAME step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The arithmetic lives in
``came_oracle.c`` (plain C loops, float64), which states its sources and
readings; this module builds it with gcc, loads it with ctypes and marshals
numpy float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "came_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_came.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction).

    ORACLE_CAME_LIB_OVERRIDE names an already-built library to load instead
    (the mutation test runs the pins against broken copies with it)."""
    override = os.environ.get("ORACLE_CAME_LIB_OVERRIDE")
    if override:
        return override
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("eps1", ctypes.c_double), ("eps2", ctypes.c_double),
                ("clip_threshold", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("beta3", ctypes.c_double), ("weight_decay", ctypes.c_double)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_came_step.restype = ctypes.c_int
            lib.oracle_came_step.argtypes = [dp, dp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), dp, dp, dp, dp,
                                             dp, dp, dp, ctypes.c_int64, ctypes.POINTER(_HParams),
                                             ctypes.c_char_p, ctypes.c_int]
            lib.oracle_came_check_hparams.restype = ctypes.c_int
            lib.oracle_came_check_hparams.argtypes = [ctypes.POINTER(_HParams), ctypes.c_char_p, ctypes.c_int]
            _lib = lib
    return _lib


class CameOracleError(ValueError):
    pass


@dataclass
class CameHParams:
    """CAME hyper-parameters; defaults are the article's DistributedCAME ones
    (lr has none: it must be given)."""
    lr: float | None = None
    eps: tuple = (1e-30, 1e-16)
    clip_threshold: float = 1.0
    betas: tuple = (0.9, 0.999, 0.9999)
    weight_decay: float = 0.0

    def _c(self) -> _HParams:
        if self.lr is None:
            raise CameOracleError("CAME needs a learning rate (lr has no default)")
        try:
            b1, b2, b3 = self.betas
            e1, e2 = self.eps
        except (TypeError, ValueError):
            raise CameOracleError("betas must have 3 values and eps 2") from None
        return _HParams(float(self.lr), float(e1), float(e2), float(self.clip_threshold), float(b1), float(b2),
                        float(b3), float(self.weight_decay))


def check_hparams(hp: CameHParams) -> None:
    err = ctypes.create_string_buffer(256)
    c = hp._c()
    if _load().oracle_came_check_hparams(ctypes.byref(c), err, 256) != 0:
        raise CameOracleError(err.value.decode())


class CameState:
    """float64 CAME state of one tensor, zero-initialised: factored tensors
    keep row/col (second moment) and res_row/res_col (instability), others
    full v and res; every tensor keeps exp_avg."""

    def __init__(self, shape):
        shape = tuple(int(s) for s in shape)
        self.shape = shape
        n = int(np.prod(shape)) if shape else 1
        if len(shape) >= 2:
            lead = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
            self.row = np.zeros(lead * shape[-2])
            self.col = np.zeros(lead * shape[-1])
            self.res_row = np.zeros(lead * shape[-2])
            self.res_col = np.zeros(lead * shape[-1])
            self.v = self.res = None
        else:
            self.row = self.col = self.res_row = self.res_col = None
            self.v = np.zeros(n)
            self.res = np.zeros(n)
        self.exp_avg = np.zeros(n)


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def step(p: np.ndarray, g: np.ndarray, state: CameState, t: int, hp: CameHParams) -> None:
    """One oracle step on one tensor; p (float64, contiguous) is updated in place."""
    if p.dtype != np.float64 or not p.flags["C_CONTIGUOUS"]:
        raise CameOracleError("p must be a C-contiguous float64 array (updated in place)")
    p_flat = p.reshape(-1)
    g_flat = np.ascontiguousarray(g, dtype=np.float64).reshape(-1)
    if g_flat.size != p_flat.size:
        raise CameOracleError("g and p differ in size")
    shape = (ctypes.c_int64 * max(1, len(state.shape)))(*state.shape) if state.shape else (ctypes.c_int64 * 1)(1)
    err = ctypes.create_string_buffer(256)
    c = hp._c()
    rc = _load().oracle_came_step(_ptr(p_flat), _ptr(g_flat), len(state.shape), shape, _ptr(state.row),
                                  _ptr(state.col), _ptr(state.v), _ptr(state.exp_avg), _ptr(state.res_row),
                                  _ptr(state.res_col), _ptr(state.res), int(t), ctypes.byref(c), err, 256)
    if rc != 0:
        raise CameOracleError(err.value.decode())
