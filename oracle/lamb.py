"""Float64 CPU oracle for the LAMB step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The arithmetic lives in
``lamb_oracle.c`` (plain C loops, float64), which states its sources and
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
_SRC = os.path.join(_HERE, "lamb_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_lamb.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction).

    ORACLE_LAMB_LIB_OVERRIDE names an already-built library to load instead
    (the mutation test runs the pins against broken copies with it)."""
    override = os.environ.get("ORACLE_LAMB_LIB_OVERRIDE")
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
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("bias_correction", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_lamb_step.restype = ctypes.c_int
            lib.oracle_lamb_step.argtypes = [dp, dp, ctypes.c_int64, dp, dp, ctypes.c_int64,
                                             ctypes.POINTER(_HParams), dp, ctypes.c_char_p, ctypes.c_int]
            lib.oracle_lamb_check_hparams.restype = ctypes.c_int
            lib.oracle_lamb_check_hparams.argtypes = [ctypes.POINTER(_HParams), ctypes.c_char_p, ctypes.c_int]
            _lib = lib
    return _lib


@dataclass
class LambHParams:
    """LAMB hyper-parameters; defaults are the article's DistributedLAMB ones."""
    lr: float = 1e-3
    betas: tuple = (0.9, 0.999)
    eps: float = 1e-6
    weight_decay: float = 0.0
    bias_correction: bool = True

    def _c(self) -> _HParams:
        return _HParams(float(self.lr), float(self.betas[0]), float(self.betas[1]), float(self.eps),
                        float(self.weight_decay), int(bool(self.bias_correction)))


class LambOracleError(ValueError):
    pass


def check_hparams(hp: LambHParams) -> None:
    err = ctypes.create_string_buffer(256)
    c = hp._c()
    if _load().oracle_lamb_check_hparams(ctypes.byref(c), err, 256) != 0:
        raise LambOracleError(err.value.decode())


class LambState:
    """float64 LAMB state of one tensor (exp_avg, exp_avg_sq), zero-initialised."""

    def __init__(self, shape):
        shape = tuple(int(s) for s in shape)
        self.shape = shape
        n = int(np.prod(shape)) if shape else 1
        self.exp_avg = np.zeros(n, np.float64)
        self.exp_avg_sq = np.zeros(n, np.float64)
        self.trust = None  # trust ratio of the last step


def _ptr(a):
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def step(p: np.ndarray, g: np.ndarray, state: LambState, t: int, hp: LambHParams) -> float:
    """One oracle step on one tensor; p (float64, contiguous) is updated in
    place.  Returns the trust ratio used."""
    if p.dtype != np.float64 or not p.flags["C_CONTIGUOUS"]:
        raise LambOracleError("p must be a C-contiguous float64 array (updated in place)")
    p_flat = p.reshape(-1)
    g_flat = np.ascontiguousarray(g, dtype=np.float64).reshape(-1)
    if g_flat.size != p_flat.size:
        raise LambOracleError("g and p differ in size")
    err = ctypes.create_string_buffer(256)
    c = hp._c()
    trust = ctypes.c_double(0.0)
    rc = _load().oracle_lamb_step(_ptr(p_flat), _ptr(g_flat), p_flat.size, _ptr(state.exp_avg),
                                  _ptr(state.exp_avg_sq), int(t), ctypes.byref(c), ctypes.byref(trust), err, 256)
    if rc != 0:
        raise LambOracleError(err.value.decode())
    state.trust = trust.value
    return trust.value
