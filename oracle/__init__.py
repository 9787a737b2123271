"""Float64 CPU oracle for the Adafactor step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never touches it, and it never touches the product path: the two
share no code.

The arithmetic lives in ``adafactor_oracle.c`` (plain C loops, float64), which
cites the article passages it follows.  This module only builds that file with
gcc, loads it with ctypes and marshals numpy float64 arrays in and out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adafactor_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_adafactor.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction).

    ORACLE_LIB_OVERRIDE names an already-built library to load instead; the
    mutation test uses it to run the pins against deliberately broken copies."""
    override = os.environ.get("ORACLE_LIB_OVERRIDE")
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
    _fields_ = [
        ("lr", ctypes.c_double), ("has_lr", ctypes.c_int32),
        ("eps1", ctypes.c_double), ("eps2", ctypes.c_double),
        ("clip_threshold", ctypes.c_double), ("decay_rate", ctypes.c_double),
        ("beta1", ctypes.c_double), ("has_beta1", ctypes.c_int32),
        ("weight_decay", ctypes.c_double),
        ("scale_parameter", ctypes.c_int32), ("relative_step", ctypes.c_int32),
        ("warmup_init", ctypes.c_int32),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_adafactor_step.restype = ctypes.c_int
            lib.oracle_adafactor_step.argtypes = [
                dp, dp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), dp, dp, dp, dp,
                ctypes.c_int64, ctypes.POINTER(_HParams), ctypes.c_char_p, ctypes.c_int]
            lib.oracle_adafactor_step_q8.restype = ctypes.c_int
            lib.oracle_adafactor_step_q8.argtypes = [
                dp, dp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), dp, dp, dp,
                ctypes.POINTER(ctypes.c_int8), ctypes.POINTER(ctypes.c_float), dp,
                ctypes.c_int64, ctypes.POINTER(_HParams), ctypes.c_char_p, ctypes.c_int]
            i8p, f32p = ctypes.POINTER(ctypes.c_int8), ctypes.POINTER(ctypes.c_float)
            lib.oracle_q8_moment.restype = ctypes.c_int
            lib.oracle_q8_moment.argtypes = [
                dp, dp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), dp, dp, dp, i8p, f32p, dp, dp,
                ctypes.c_int64, ctypes.POINTER(_HParams), ctypes.c_char_p, ctypes.c_int]
            lib.oracle_q8_quantize.restype = None
            lib.oracle_q8_quantize.argtypes = [dp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), i8p, f32p]
            lib.oracle_q8_apply.restype = None
            lib.oracle_q8_apply.argtypes = [dp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), i8p, f32p,
                                            ctypes.c_double, ctypes.POINTER(_HParams)]
            lib.oracle_check_hparams.restype = ctypes.c_int
            lib.oracle_check_hparams.argtypes = [ctypes.POINTER(_HParams), ctypes.c_char_p, ctypes.c_int]
            lib.oracle_rho.restype = ctypes.c_double
            lib.oracle_rho.argtypes = [ctypes.POINTER(_HParams), ctypes.c_int64]
            lib.oracle_beta2.restype = ctypes.c_double
            lib.oracle_beta2.argtypes = [ctypes.POINTER(_HParams), ctypes.c_int64]
            _lib = lib
    return _lib


@dataclass
class HParams:
    """Adafactor hyper-parameters; defaults are the article's Step 3 defaults."""
    lr: float | None = None
    eps: tuple = (1e-30, 1e-3)
    clip_threshold: float = 1.0
    decay_rate: float = -0.8
    beta1: float | None = None
    weight_decay: float = 0.0
    scale_parameter: bool = True
    relative_step: bool = True
    warmup_init: bool = False

    def _c(self) -> _HParams:
        return _HParams(
            0.0 if self.lr is None else float(self.lr), 0 if self.lr is None else 1,
            float(self.eps[0]), float(self.eps[1]), float(self.clip_threshold),
            float(self.decay_rate), 0.0 if self.beta1 is None else float(self.beta1),
            0 if self.beta1 is None else 1, float(self.weight_decay),
            int(bool(self.scale_parameter)), int(bool(self.relative_step)),
            int(bool(self.warmup_init)))


class OracleError(ValueError):
    pass


def check_hparams(hp: HParams) -> None:
    err = ctypes.create_string_buffer(256)
    c = hp._c()
    if _load().oracle_check_hparams(ctypes.byref(c), err, 256) != 0:
        raise OracleError(err.value.decode())


def rho(hp: HParams, t: int) -> float:
    c = hp._c()
    return _load().oracle_rho(ctypes.byref(c), int(t))


def beta2(hp: HParams, t: int) -> float:
    c = hp._c()
    return _load().oracle_beta2(ctypes.byref(c), int(t))


Q8_GROUP = 128  # values per group of the 8-bit first moment (along the last dim)


def q8_groups(shape):
    """(rows, groups per row) of the 8-bit first moment of a tensor."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    last = shape[-1] if len(shape) >= 2 else n
    rows = n // last if last else 0
    return rows, (last + Q8_GROUP - 1) // Q8_GROUP


class State:
    """float64 optimizer state of one tensor, zero-initialised.  q8: the first
    moment is held as int8 codes and fp32 group scales (exp_avg_codes,
    exp_avg_scales) instead of float64 exp_avg."""

    def __init__(self, shape, beta1: bool, q8: bool = False):
        shape = tuple(int(s) for s in shape)
        self.shape = shape
        n = int(np.prod(shape)) if shape else 1
        if len(shape) >= 2:
            lead = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
            self.row = np.zeros(lead * shape[-2], np.float64)
            self.col = np.zeros(lead * shape[-1], np.float64)
            self.v = None
        else:
            self.row = self.col = None
            self.v = np.zeros(n, np.float64)
        self.exp_avg = np.zeros(n, np.float64) if beta1 and not q8 else None
        self.q8 = bool(q8)
        if q8:
            rows, groups = q8_groups(shape)
            self.exp_avg_codes = np.zeros(n, np.int8)
            self.exp_avg_scales = np.zeros(rows * groups, np.float32)
            self.moment = np.zeros(n, np.float64)  # the last step's new moment, before quantisation
        else:
            self.exp_avg_codes = self.exp_avg_scales = self.moment = None


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def step(p: np.ndarray, g: np.ndarray, state: State, t: int, hp: HParams) -> None:
    """One oracle step on one tensor; p (float64, contiguous) is updated in place."""
    if p.dtype != np.float64 or not p.flags["C_CONTIGUOUS"]:
        raise OracleError("p must be a C-contiguous float64 array (updated in place)")
    p_flat = p.reshape(-1)
    g_flat = np.ascontiguousarray(g, dtype=np.float64).reshape(-1)
    shape = (ctypes.c_int64 * max(1, len(state.shape)))(*state.shape) if state.shape else (ctypes.c_int64 * 1)(1)
    err = ctypes.create_string_buffer(256)
    c = hp._c()
    if state.q8:
        codes, scales = state.exp_avg_codes, state.exp_avg_scales
        assert codes.dtype == np.int8 and scales.dtype == np.float32
        assert codes.flags["C_CONTIGUOUS"] and scales.flags["C_CONTIGUOUS"]
        rc = _load().oracle_adafactor_step_q8(
            _ptr(p_flat), _ptr(g_flat), len(state.shape), shape, _ptr(state.row), _ptr(state.col),
            _ptr(state.v), codes.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)),
            scales.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), _ptr(state.moment), int(t), ctypes.byref(c),
            err, 256)
        if rc != 0:
            raise OracleError(err.value.decode())
        return
    rc = _load().oracle_adafactor_step(
        _ptr(p_flat), _ptr(g_flat), len(state.shape), shape, _ptr(state.row), _ptr(state.col),
        _ptr(state.v), _ptr(state.exp_avg), int(t), ctypes.byref(c), err, 256)
    if rc != 0:
        raise OracleError(err.value.decode())


def _shape_arg(shape):
    shape = tuple(int(s) for s in shape)
    return (ctypes.c_int64 * max(1, len(shape)))(*shape) if shape else (ctypes.c_int64 * 1)(1), len(shape)


def _i8(a):
    assert a.dtype == np.int8 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))


def _f32(a):
    assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def q8_moment(p: np.ndarray, g: np.ndarray, state: State, t: int, hp: HParams):
    """Part 1 of the 8-bit step: updates the second-moment state of `state` in
    place and returns (m, alpha): the new first moment (float64, before
    quantisation) formed from the stored codes and scales, and the step's lr.
    p is read, not changed."""
    assert state.q8
    p_flat = np.ascontiguousarray(p, dtype=np.float64).reshape(-1)
    g_flat = np.ascontiguousarray(g, dtype=np.float64).reshape(-1)
    m = np.zeros(p_flat.size, np.float64)
    alpha = ctypes.c_double(0.0)
    shp, nd = _shape_arg(state.shape)
    err = ctypes.create_string_buffer(256)
    c = hp._c()
    rc = _load().oracle_q8_moment(
        _ptr(p_flat), _ptr(g_flat), nd, shp, _ptr(state.row), _ptr(state.col), _ptr(state.v),
        _i8(state.exp_avg_codes), _f32(state.exp_avg_scales), _ptr(m), ctypes.byref(alpha), int(t),
        ctypes.byref(c), err, 256)
    if rc != 0:
        raise OracleError(err.value.decode())
    return m, alpha.value


def q8_quantize(m: np.ndarray, shape):
    """Part 2: the page's group quantiser on a moment of the given shape;
    returns (codes int8 [N], scales float32 [rows * groups])."""
    m = np.ascontiguousarray(m, dtype=np.float64).reshape(-1)
    rows, groups = q8_groups(shape)
    codes = np.zeros(m.size, np.int8)
    scales = np.zeros(rows * groups, np.float32)
    shp, nd = _shape_arg(shape)
    _load().oracle_q8_quantize(_ptr(m), nd, shp, _i8(codes), _f32(scales))
    return codes, scales


def q8_apply(p: np.ndarray, codes: np.ndarray, scales: np.ndarray, shape, alpha: float, hp: HParams) -> None:
    """Part 3: weight decay and the dequantised moment as the update, on p
    (float64, contiguous) in place."""
    if p.dtype != np.float64 or not p.flags["C_CONTIGUOUS"]:
        raise OracleError("p must be a C-contiguous float64 array (updated in place)")
    shp, nd = _shape_arg(shape)
    c = hp._c()
    _load().oracle_q8_apply(_ptr(p.reshape(-1)), nd, shp, _i8(codes), _f32(scales), float(alpha),
                            ctypes.byref(c))
