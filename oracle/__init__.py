"""CPU oracle for the fused residual-add + RMSNorm forward (test infrastructure).

Only the test suite, the smoke check and the bench's CPU-baseline leg may
import this package.  The product path (the CUDA library and its binding)
never imports, links or calls it, and the two share no code.

The arithmetic lives in ``dradd_oracle.c`` (plain C, single-threaded,
``-ffp-contract=off``); this module compiles it with the host C compiler and
wraps it with ctypes.  ``lse_oracle.c`` / ``oracle.lse`` hold the log-sum-exp
merge and the launch-invariant elementwise functions.  Arrays of bf16 values are numpy ``uint16`` bit
patterns.  See the C file's header for the page and sections it follows.

parity pins: every function here is pinned by ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "dradd_oracle.c"
BUILD_DIR = HERE / "_build"
LIB_PATH = BUILD_DIR / "liboracle.so"

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

STORE_MODES = {"rne": 0, "trunc": 1, "ties_away": 2}

_lock = threading.Lock()
_default = None


def _compiler() -> str:
    for cc in (os.environ.get("CC"), "cc", "gcc"):
        if cc and shutil.which(cc):
            return cc
    raise RuntimeError("no C compiler found to build the oracle")


def compile_source(src: Path, out: Path) -> Path:
    """Compile one oracle C source into a shared library at ``out``."""
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(out.suffix + f".tmp{os.getpid()}")
    cmd = [_compiler(), *CFLAGS, "-o", str(tmp), str(src), "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> Path:
    """Build ``liboracle.so`` (and the log-sum-exp oracle's library) next to
    the sources if missing or stale."""
    with _lock:
        stale = (not LIB_PATH.exists()
                 or LIB_PATH.stat().st_mtime < SOURCE.stat().st_mtime)
        if force or stale:
            compile_source(SOURCE, LIB_PATH)
    from . import lse
    lse.build(force)
    return LIB_PATH


_u16p = ctypes.POINTER(ctypes.c_uint16)
_i8p = ctypes.POINTER(ctypes.c_int8)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_i64 = ctypes.c_int64


def _ptr(a: np.ndarray | None, typ):
    if a is None:
        return ctypes.cast(None, typ)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(typ)


def _as_u16(a) -> np.ndarray:
    """Accept numpy uint16/int16 arrays or torch bf16/int16 tensors."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        return t.numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: Path):
        self.path = Path(path)
        L = ctypes.CDLL(str(self.path))
        self._L = L
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        for name in ("oracle_bf16_rne", "oracle_bf16_trunc", "oracle_bf16_ties_away"):
            f = getattr(L, name)
            f.restype = ctypes.c_uint16
            f.argtypes = [ctypes.c_float]
        L.oracle_bf16_convert_range.restype = ctypes.c_int
        L.oracle_bf16_convert_range.argtypes = [_u16p, ctypes.c_uint64, _i64, ctypes.c_int]
        L.oracle_bf16_convert_array.restype = ctypes.c_int
        L.oracle_bf16_convert_array.argtypes = [_u16p, _f32p, _i64, ctypes.c_int]
        L.oracle_pairwise_sum.restype = ctypes.c_float
        L.oracle_pairwise_sum.argtypes = [_f32p, _i64]
        L.oracle_add_rmsnorm_fwd.restype = ctypes.c_int
        L.oracle_add_rmsnorm_fwd.argtypes = [
            _u16p, _u16p, _u16p, _u16p, _u16p, ctypes.c_float, _i64, _i64, ctypes.c_int,
            _f32p, _f32p]
        L.oracle_add_rmsnorm_quant_fwd.restype = ctypes.c_int
        L.oracle_add_rmsnorm_quant_fwd.argtypes = [
            _i8p, _f32p, _u16p, _u16p, _u16p, _u16p, ctypes.c_float, _i64, _i64, ctypes.c_int,
            _f32p, _f32p]
        L.oracle_rmsnorm_fwd.restype = ctypes.c_int
        L.oracle_rmsnorm_fwd.argtypes = [_u16p, _u16p, _u16p, ctypes.c_float, _i64, _i64, ctypes.c_int,
                                         _f32p, _f32p]
        L.oracle_rmsnorm_quant_fwd.restype = ctypes.c_int
        L.oracle_rmsnorm_quant_fwd.argtypes = [_i8p, _f32p, _u16p, _u16p, ctypes.c_float, _i64, _i64]
        L.oracle_residual_add_fwd.restype = ctypes.c_int
        L.oracle_residual_add_fwd.argtypes = [_u16p, _u16p, _u16p, _i64, ctypes.c_int]
        L.oracle_e4m3_rne.restype = ctypes.c_uint8
        L.oracle_e4m3_rne.argtypes = [ctypes.c_float]
        L.oracle_e4m3_convert_array.restype = ctypes.c_int
        L.oracle_e4m3_convert_array.argtypes = [_u8p, _f32p, _i64]
        L.oracle_rmsnorm_e4m3_fwd.restype = ctypes.c_int
        L.oracle_rmsnorm_e4m3_fwd.argtypes = [_u8p, _f32p, _u16p, _u16p, _u16p, _u16p, ctypes.c_float,
                                              _i64, _i64]
        L.oracle_e2m1_rne.restype = ctypes.c_uint8
        L.oracle_e2m1_rne.argtypes = [ctypes.c_float]
        L.oracle_e2m1_convert_array.restype = ctypes.c_int
        L.oracle_e2m1_convert_array.argtypes = [_u8p, _f32p, _i64]
        L.oracle_rmsnorm_e2m1_fwd.restype = ctypes.c_int
        L.oracle_rmsnorm_e2m1_fwd.argtypes = [_u8p, _f32p, _u16p, _u16p, _u16p, _u16p, ctypes.c_float,
                                              _i64, _i64]
        L.oracle_qk_rmsnorm_fwd.restype = ctypes.c_int
        L.oracle_qk_rmsnorm_fwd.argtypes = [ctypes.c_void_p, _f32p, _u16p, _u16p, _u16p, _u16p, _u16p,
                                            _u16p, _u16p, ctypes.c_float, ctypes.c_float, _i64, _i64,
                                            _i64, _i64, _i64]
        L.oracle_abi_version.restype = ctypes.c_int

    # ---- conversions -------------------------------------------------
    def bf16_to_f32(self, b: int) -> float:
        return self._L.oracle_bf16_to_f32(b)

    def bf16_scalar(self, f: float, mode: str = "rne") -> int:
        fn = {"rne": self._L.oracle_bf16_rne, "trunc": self._L.oracle_bf16_trunc,
              "ties_away": self._L.oracle_bf16_ties_away}[mode]
        return int(fn(ctypes.c_float(f)))

    def bf16_convert_range(self, first: int, count: int, mode: str = "rne") -> np.ndarray:
        dst = np.empty(count, dtype=np.uint16)
        rc = self._L.oracle_bf16_convert_range(_ptr(dst, _u16p), first, count, STORE_MODES[mode])
        assert rc == 0
        return dst

    def bf16_convert(self, f32: np.ndarray, mode: str = "rne") -> np.ndarray:
        src = np.ascontiguousarray(f32, dtype=np.float32)
        dst = np.empty(src.shape, dtype=np.uint16)
        rc = self._L.oracle_bf16_convert_array(_ptr(dst, _u16p), _ptr(src, _f32p), src.size,
                                                STORE_MODES[mode])
        assert rc == 0
        return dst

    def pairwise_sum(self, v: np.ndarray) -> np.float32:
        a = np.ascontiguousarray(v, dtype=np.float32)
        return np.float32(self._L.oracle_pairwise_sum(_ptr(a, _f32p), a.size))

    # ---- the method ------------------------------------------------------
    def add_rmsnorm_fwd(self, x, residual, weight, eps: float, store_mode: str = "rne",
                        threads: int = 1, return_terms: bool = False):
        """Return (out, residual_out) as uint16 arrays shaped like x.

        With return_terms, also the per-row fp32 sum of squares and 1/rms.
        threads > 1 splits the rows over threads (rows are independent, so
        the bits are the same as a single-threaded run)."""
        x, residual, weight = _as_u16(x), _as_u16(residual), _as_u16(weight)
        hidden = x.shape[-1]
        n_rows = x.size // hidden if hidden else 0
        assert residual.shape == x.shape and weight.size == hidden
        out = np.empty_like(x)
        ro = np.empty_like(x)
        ss = np.empty(n_rows, dtype=np.float32)
        inv = np.empty(n_rows, dtype=np.float32)
        mode = STORE_MODES[store_mode]
        x2, r2 = x.reshape(n_rows, hidden), residual.reshape(n_rows, hidden)
        o2, ro2 = out.reshape(n_rows, hidden), ro.reshape(n_rows, hidden)

        def run(lo: int, hi: int) -> int:
            if hi <= lo:
                return 0
            return self._L.oracle_add_rmsnorm_fwd(
                _ptr(o2[lo:hi], _u16p), _ptr(ro2[lo:hi], _u16p), _ptr(x2[lo:hi], _u16p),
                _ptr(r2[lo:hi], _u16p), _ptr(weight, _u16p), ctypes.c_float(eps),
                hi - lo, hidden, mode, _ptr(ss[lo:hi], _f32p), _ptr(inv[lo:hi], _f32p))

        for rc in _split_rows(run, n_rows, threads):
            if rc != 0:
                raise RuntimeError(f"oracle_add_rmsnorm_fwd failed with {rc}")
        if return_terms:
            return out, ro, ss, inv
        return out, ro

    def add_rmsnorm_quant_fwd(self, x, residual, weight, eps: float, store_mode: str = "rne",
                              threads: int = 1, return_terms: bool = False):
        """Return (out_q int8, scale fp32 per row, residual_out uint16)."""
        x, residual, weight = _as_u16(x), _as_u16(residual), _as_u16(weight)
        hidden = x.shape[-1]
        n_rows = x.size // hidden if hidden else 0
        assert residual.shape == x.shape and weight.size == hidden
        q = np.empty(x.shape, dtype=np.int8)
        scale = np.empty(n_rows, dtype=np.float32)
        ro = np.empty_like(x)
        ss = np.empty(n_rows, dtype=np.float32)
        inv = np.empty(n_rows, dtype=np.float32)
        mode = STORE_MODES[store_mode]
        x2, r2 = x.reshape(n_rows, hidden), residual.reshape(n_rows, hidden)
        q2, ro2 = q.reshape(n_rows, hidden), ro.reshape(n_rows, hidden)

        def run(lo: int, hi: int) -> int:
            if hi <= lo:
                return 0
            return self._L.oracle_add_rmsnorm_quant_fwd(
                _ptr(q2[lo:hi], _i8p), _ptr(scale[lo:hi], _f32p), _ptr(ro2[lo:hi], _u16p),
                _ptr(x2[lo:hi], _u16p), _ptr(r2[lo:hi], _u16p), _ptr(weight, _u16p),
                ctypes.c_float(eps), hi - lo, hidden, mode,
                _ptr(ss[lo:hi], _f32p), _ptr(inv[lo:hi], _f32p))

        for rc in _split_rows(run, n_rows, threads):
            if rc != 0:
                raise RuntimeError(f"oracle_add_rmsnorm_quant_fwd failed with {rc}")
        if return_terms:
            return q, scale, ro, ss, inv
        return q, scale, ro


    def rmsnorm_fwd(self, x, weight, eps: float, store_mode: str = "rne", threads: int = 1,
                    return_terms: bool = False):
        """Plain RMSNorm: out (uint16 array shaped like x)."""
        x, weight = _as_u16(x), _as_u16(weight)
        hidden = x.shape[-1]
        n_rows = x.size // hidden if hidden else 0
        assert weight.size == hidden
        out = np.empty_like(x)
        ss = np.empty(n_rows, dtype=np.float32)
        inv = np.empty(n_rows, dtype=np.float32)
        x2, o2 = x.reshape(n_rows, hidden), out.reshape(n_rows, hidden)
        mode = STORE_MODES[store_mode]

        def run(lo: int, hi: int) -> int:
            if hi <= lo:
                return 0
            return self._L.oracle_rmsnorm_fwd(
                _ptr(o2[lo:hi], _u16p), _ptr(x2[lo:hi], _u16p), _ptr(weight, _u16p), ctypes.c_float(eps),
                hi - lo, hidden, mode, _ptr(ss[lo:hi], _f32p), _ptr(inv[lo:hi], _f32p))

        for rc in _split_rows(run, n_rows, threads):
            if rc != 0:
                raise RuntimeError(f"oracle_rmsnorm_fwd failed with {rc}")
        return (out, ss, inv) if return_terms else out

    def rmsnorm_quant_fwd(self, x, weight, eps: float, threads: int = 1):
        """Plain RMSNorm, int8 out: (out_q, scale)."""
        x, weight = _as_u16(x), _as_u16(weight)
        hidden = x.shape[-1]
        n_rows = x.size // hidden if hidden else 0
        q = np.empty(x.shape, dtype=np.int8)
        scale = np.empty(n_rows, dtype=np.float32)
        x2, q2 = x.reshape(n_rows, hidden), q.reshape(n_rows, hidden)

        def run(lo: int, hi: int) -> int:
            if hi <= lo:
                return 0
            return self._L.oracle_rmsnorm_quant_fwd(
                _ptr(q2[lo:hi], _i8p), _ptr(scale[lo:hi], _f32p), _ptr(x2[lo:hi], _u16p),
                _ptr(weight, _u16p), ctypes.c_float(eps), hi - lo, hidden)

        for rc in _split_rows(run, n_rows, threads):
            if rc != 0:
                raise RuntimeError(f"oracle_rmsnorm_quant_fwd failed with {rc}")
        return q, scale

    def residual_add_fwd(self, x, residual, store_mode: str = "rne"):
        """The residual update alone: residual_out (uint16, shaped like x)."""
        x, residual = _as_u16(x), _as_u16(residual)
        assert residual.shape == x.shape
        ro = np.empty_like(x)
        rc = self._L.oracle_residual_add_fwd(_ptr(ro, _u16p), _ptr(x, _u16p), _ptr(residual, _u16p),
                                             x.size, STORE_MODES[store_mode])
        if rc != 0:
            raise RuntimeError(f"oracle_residual_add_fwd failed with {rc}")
        return ro


    def e4m3_scalar(self, f: float) -> int:
        return int(self._L.oracle_e4m3_rne(ctypes.c_float(f)))

    def e4m3_convert(self, f32: np.ndarray) -> np.ndarray:
        src = np.ascontiguousarray(f32, dtype=np.float32)
        dst = np.empty(src.shape, dtype=np.uint8)
        assert self._L.oracle_e4m3_convert_array(_ptr(dst, _u8p), _ptr(src, _f32p), src.size) == 0
        return dst

    def rmsnorm_fp8_fwd(self, x, weight, eps: float, residual=None, threads: int = 1):
        """Per-row e4m3 out: (out_q uint8 codes, scale fp32) for plain RMSNorm,
        or (out_q, scale, residual_out) with a residual."""
        x, weight = _as_u16(x), _as_u16(weight)
        hidden = x.shape[-1]
        n_rows = x.size // hidden if hidden else 0
        r = _as_u16(residual) if residual is not None else None
        q = np.empty(x.shape, dtype=np.uint8)
        scale = np.empty(n_rows, dtype=np.float32)
        ro = np.empty_like(x) if r is not None else None
        x2, q2 = x.reshape(n_rows, hidden), q.reshape(n_rows, hidden)
        r2 = r.reshape(n_rows, hidden) if r is not None else None
        ro2 = ro.reshape(n_rows, hidden) if r is not None else None

        def run(lo: int, hi: int) -> int:
            if hi <= lo:
                return 0
            return self._L.oracle_rmsnorm_e4m3_fwd(
                _ptr(q2[lo:hi], _u8p), _ptr(scale[lo:hi], _f32p),
                _ptr(ro2[lo:hi] if r is not None else None, _u16p), _ptr(x2[lo:hi], _u16p),
                _ptr(r2[lo:hi] if r is not None else None, _u16p), _ptr(weight, _u16p),
                ctypes.c_float(eps), hi - lo, hidden)

        for rc in _split_rows(run, n_rows, threads):
            if rc != 0:
                raise RuntimeError(f"oracle_rmsnorm_e4m3_fwd failed with {rc}")
        return (q, scale) if r is None else (q, scale, ro)


    def e2m1_scalar(self, f: float) -> int:
        return int(self._L.oracle_e2m1_rne(ctypes.c_float(f)))

    def e2m1_convert(self, f32: np.ndarray) -> np.ndarray:
        src = np.ascontiguousarray(f32, dtype=np.float32)
        dst = np.empty(src.shape, dtype=np.uint8)
        assert self._L.oracle_e2m1_convert_array(_ptr(dst, _u8p), _ptr(src, _f32p), src.size) == 0
        return dst

    def rmsnorm_fp4_fwd(self, x, weight, eps: float, residual=None, threads: int = 1):
        """Per-row e2m1 out, two codes per byte: (out_q [n, h/2] uint8, scale)
        for plain RMSNorm, or (out_q, scale, residual_out) with a residual."""
        x, weight = _as_u16(x), _as_u16(weight)
        hidden = x.shape[-1]
        n_rows = x.size // hidden if hidden else 0
        r = _as_u16(residual) if residual is not None else None
        q = np.empty((n_rows, hidden // 2), dtype=np.uint8)
        scale = np.empty(n_rows, dtype=np.float32)
        ro = np.empty_like(x) if r is not None else None
        x2 = x.reshape(n_rows, hidden)
        r2 = r.reshape(n_rows, hidden) if r is not None else None
        ro2 = ro.reshape(n_rows, hidden) if r is not None else None

        def run(lo: int, hi: int) -> int:
            if hi <= lo:
                return 0
            return self._L.oracle_rmsnorm_e2m1_fwd(
                _ptr(q[lo:hi], _u8p), _ptr(scale[lo:hi], _f32p),
                _ptr(ro2[lo:hi] if r is not None else None, _u16p), _ptr(x2[lo:hi], _u16p),
                _ptr(r2[lo:hi] if r is not None else None, _u16p), _ptr(weight, _u16p),
                ctypes.c_float(eps), hi - lo, hidden)

        for rc in _split_rows(run, n_rows, threads):
            if rc != 0:
                raise RuntimeError(f"oracle_rmsnorm_e2m1_fwd failed with {rc}")
        return (q, scale) if r is None else (q, scale, ro)

    def qk_rmsnorm_fwd(self, q, q_weight, k, k_weight, q_eps: float, k_eps: float,
                       group_size: int = 0, q_residual=None):
        """Fused q/k RMSNorm: returns a dict with q_out (bf16 bit patterns,
        shaped like q, when group_size == 0; else e4m3 codes, uint8), q_scale
        ([n_q, q_hidden / group_size] fp32, or None), q_residual_out (with a
        q residual, else None) and k_out (bf16 bit patterns shaped like k).
        q or k may have zero rows."""
        q, qw, k, kw = _as_u16(q), _as_u16(q_weight), _as_u16(k), _as_u16(k_weight)
        hq, hk = q.shape[-1], k.shape[-1]
        nq = q.size // hq if hq else 0
        nk = k.size // hk if hk else 0
        qr = _as_u16(q_residual) if q_residual is not None else None
        if group_size:
            q_out = np.empty(q.shape, dtype=np.uint8)
            q_scale = np.empty((nq, hq // group_size), dtype=np.float32)
        else:
            q_out = np.empty(q.shape, dtype=np.uint16)
            q_scale = None
        qro = np.empty_like(q) if qr is not None else None
        k_out = np.empty_like(k)
        rc = self._L.oracle_qk_rmsnorm_fwd(
            q_out.ctypes.data_as(ctypes.c_void_p), _ptr(q_scale, _f32p), _ptr(qro, _u16p),
            _ptr(k_out, _u16p), _ptr(q, _u16p), _ptr(qr, _u16p), _ptr(qw, _u16p), _ptr(k, _u16p),
            _ptr(kw, _u16p), ctypes.c_float(q_eps), ctypes.c_float(k_eps), nq, hq, nk, hk,
            int(group_size))
        if rc != 0:
            raise RuntimeError(f"oracle_qk_rmsnorm_fwd failed with {rc}")
        return {"q_out": q_out, "q_scale": q_scale, "q_residual_out": qro, "k_out": k_out}


def _split_rows(run, n_rows: int, threads: int):
    threads = max(1, min(int(threads), n_rows or 1))
    if threads == 1:
        return [run(0, n_rows)]
    step = -(-n_rows // threads)
    with ThreadPoolExecutor(threads) as ex:  # ctypes releases the GIL
        return list(ex.map(lambda lo: run(lo, min(n_rows, lo + step)),
                           range(0, n_rows, step)))


def lib() -> Oracle:
    """The default oracle, built on first use."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))
