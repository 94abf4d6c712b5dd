"""CPU oracle for the log-sum-exp merge and the launch-invariant elementwise
functions (test infrastructure; see ``lse_oracle.c`` for the page and the
sections it follows).

Inputs are fp32 numpy arrays (or anything ``np.asarray`` turns into one);
results are float64 arrays: the exact quantity to double precision, against
which the kernels' fp32 results are compared within a stated bound.

parity pins: ``tests/test_oracle_lse.py``.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

import numpy as np

from . import BUILD_DIR, HERE, compile_source

SOURCE = HERE / "lse_oracle.c"
LIB_PATH = BUILD_DIR / "liblse_oracle.so"
UNARY_OPS = {"log1p": 0, "cosh": 1, "exp": 2}

_lock = threading.Lock()
_default = None
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> Path:
    with _lock:
        if force or not LIB_PATH.exists() or LIB_PATH.stat().st_mtime < SOURCE.stat().st_mtime:
            compile_source(SOURCE, LIB_PATH)
    return LIB_PATH


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


class LseOracle:
    def __init__(self, path: Path):
        L = ctypes.CDLL(str(path))
        L.oracle_lse_merge1.restype = ctypes.c_double
        L.oracle_lse_merge1.argtypes = [ctypes.c_float, ctypes.c_float]
        L.oracle_lse_merge.restype = ctypes.c_int
        L.oracle_lse_merge.argtypes = [_f64p, _f32p, _f32p, _i64]
        L.oracle_lse_merge_2d.restype = ctypes.c_int
        L.oracle_lse_merge_2d.argtypes = [_f64p, _f32p, _i64, _f32p, _i64, _i64, _i64]
        L.oracle_unary.restype = ctypes.c_int
        L.oracle_unary.argtypes = [_f64p, _f32p, _i64, ctypes.c_int]
        self._L = L

    def merge1(self, a: float, b: float) -> float:
        return float(self._L.oracle_lse_merge1(ctypes.c_float(a), ctypes.c_float(b)))

    def merge(self, a, b) -> np.ndarray:
        """log(e^a + e^b) elementwise, in double."""
        a, b = _f32(a), _f32(b)
        assert a.shape == b.shape
        out = np.empty(a.shape, dtype=np.float64)
        rc = self._L.oracle_lse_merge(out.ctypes.data_as(_f64p), a.ctypes.data_as(_f32p),
                                      b.ctypes.data_as(_f32p), a.size)
        assert rc == 0
        return out

    def merge_2d(self, a, a_stride: int, b, b_stride: int, n_rows: int, n_cols: int) -> np.ndarray:
        """Row-strided merge of flat arrays a, b: an (n_rows, n_cols) result."""
        a, b = _f32(a).ravel(), _f32(b).ravel()
        out = np.empty((n_rows, n_cols), dtype=np.float64)
        rc = self._L.oracle_lse_merge_2d(out.ctypes.data_as(_f64p), a.ctypes.data_as(_f32p), a_stride,
                                         b.ctypes.data_as(_f32p), b_stride, n_rows, n_cols)
        assert rc == 0
        return out

    def unary(self, x, op: str) -> np.ndarray:
        x = _f32(x)
        out = np.empty(x.shape, dtype=np.float64)
        rc = self._L.oracle_unary(out.ctypes.data_as(_f64p), x.ctypes.data_as(_f32p), x.size, UNARY_OPS[op])
        assert rc == 0
        return out


def lib() -> LseOracle:
    global _default
    if _default is None:
        _default = LseOracle(build())
    return _default
