"""Deterministic fused residual-add + RMSNorm forward for GB300 (sm_103a).

Thin Python binding of the C ABI in include/dradd.h (libdradd.so): it only
marshals arguments (tensor pointers, sizes, the current CUDA stream) and
turns status codes into exceptions.  Every step of the computation runs in
the CUDA kernels of the library; there is no Python or CPU fallback, and
every call fails loudly if the library cannot be loaded.

    from deterministic_residual_add_gb300 import add_rmsnorm_fwd
    out, residual_out = add_rmsnorm_fwd(x, residual, weight, eps)

The operation is rmsnorm2d_fwd_with_add as defined on the ROCm/aiter issue
#5151 page ("Steps to Reproduce", reference()), with round-to-nearest-even
bf16 stores and a reduction order that never depends on the launch.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from pathlib import Path

__all__ = [
    "add_rmsnorm_fwd", "add_rmsnorm_quant_fwd", "add_rmsnorm_fwd_with_config",
    "add_rmsnorm_quant_fwd_with_config", "rmsnorm_fwd", "rmsnorm_quant_fwd", "residual_add_fwd",
    "add_rmsnorm_fp8_fwd", "rmsnorm_fp8_fwd", "add_rmsnorm_fp4_fwd", "rmsnorm_fp4_fwd",
    "fused_qk_rmsnorm_group_quant_fwd", "qk_resolve_config", "QkPlan",
    "lse_merge_fwd", "invariant_unary_fwd", "UNARY_OPS",
    "LaunchConfig", "DraddError", "resolve_config",
    "device_status", "last_device_status", "bf16_convert_range", "status_string", "abi_version", "lib",
    "library_path", "VARIANT_AUTO", "VARIANT_ROWS", "VARIANT_STAGED", "VARIANT_SPLIT", "VARIANT_WARP",
    "VARIANT_CHUNK", "MAX_HIDDEN",
]

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "libdradd.so"
MAX_HIDDEN = 32768
VARIANT_AUTO, VARIANT_ROWS, VARIANT_STAGED, VARIANT_SPLIT, VARIANT_WARP, VARIANT_CHUNK = 0, 1, 2, 3, 4, 5
OP_ADD_RMSNORM, OP_ADD_RMSNORM_QUANT, OP_RMSNORM, OP_RMSNORM_QUANT = 0, 1, 2, 3
OP_ADD_RMSNORM_FP8, OP_RMSNORM_FP8 = 4, 5
OP_ADD_RMSNORM_FP4, OP_RMSNORM_FP4 = 6, 7

STATUS_NAMES = {
    0: "OK", 1: "NULL_PTR", 2: "BAD_SHAPE", 3: "UNSUPPORTED_HIDDEN", 4: "MISALIGNED",
    5: "BAD_EPS", 6: "ALIAS", 7: "CUDA", 8: "TIMEOUT", 9: "BAD_CONFIG", 10: "UNDRAINED",
}


class DraddError(RuntimeError):
    """A non-zero status from libdradd."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)}")


class _LaunchCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "variant", "threads_per_row", "rows_per_cta", "grid_ctas", "stages", "fault_inject",
        "wait_limit_us", "serialize", "blocks_per_thread", "cluster_ctas")]


@dataclass
class LaunchConfig:
    """Mirror of dradd_launch_cfg; 0 = automatic.  Never changes results."""
    variant: int = 0
    threads_per_row: int = 0
    rows_per_cta: int = 0
    grid_ctas: int = 0
    stages: int = 0
    fault_inject: int = 0
    wait_limit_us: int = 0
    serialize: int = 0
    blocks_per_thread: int = 0
    cluster_ctas: int = 0

    def _c(self) -> _LaunchCfg:
        return _LaunchCfg(self.variant, self.threads_per_row, self.rows_per_cta, self.grid_ctas,
                          self.stages, self.fault_inject, self.wait_limit_us, self.serialize,
                          self.blocks_per_thread, self.cluster_ctas)

    @staticmethod
    def _from_c(c: _LaunchCfg) -> "LaunchConfig":
        return LaunchConfig(c.variant, c.threads_per_row, c.rows_per_cta, c.grid_ctas, c.stages,
                            c.fault_inject, c.wait_limit_us, c.serialize, c.blocks_per_thread, c.cluster_ctas)


class _QkPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "variant", "threads_per_cta", "dyn_smem_bytes", "q_threads_per_row", "q_rows_per_cta", "q_stages",
        "q_ctas", "k_threads_per_row", "k_rows_per_cta", "k_stages", "k_ctas")]


@dataclass
class QkPlan:
    """Mirror of dradd_qk_plan: how a fused q/k call spreads its rows."""
    variant: int
    threads_per_cta: int
    dyn_smem_bytes: int
    q_threads_per_row: int
    q_rows_per_cta: int
    q_stages: int
    q_ctas: int
    k_threads_per_row: int
    k_rows_per_cta: int
    k_stages: int
    k_ctas: int


_lib = None
_vp, _i64, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float


def library_path() -> Path:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libdradd.so (built by deterministic_residual_add_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m deterministic_residual_add_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(str(LIB_PATH))
    bf16_args = [_vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp]
    quant_args = [_vp, _vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp]
    cfgp = ctypes.POINTER(_LaunchCfg)
    qk_args = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _f32, _i64, _i64, _i64, _i64, _i64, _vp]
    for name, args in [("add_rmsnorm_fwd", bf16_args),
                       ("add_rmsnorm_quant_fwd", quant_args),
                       ("add_rmsnorm_fwd_with_config", bf16_args + [cfgp]),
                       ("add_rmsnorm_quant_fwd_with_config", quant_args + [cfgp]),
                       ("rmsnorm_fwd", [_vp, _vp, _vp, _f32, _i64, _i64, _vp]),
                       ("rmsnorm_quant_fwd", [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp]),
                       ("rmsnorm_fwd_with_config", [_vp, _vp, _vp, _f32, _i64, _i64, _vp, cfgp]),
                       ("rmsnorm_quant_fwd_with_config", [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp, cfgp]),
                       ("residual_add_fwd", [_vp, _vp, _vp, _i64, _i64, _vp]),
                       ("add_rmsnorm_fp8_fwd", quant_args),
                       ("add_rmsnorm_fp8_fwd_with_config", quant_args + [cfgp]),
                       ("rmsnorm_fp8_fwd", [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp]),
                       ("rmsnorm_fp8_fwd_with_config", [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp, cfgp]),
                       ("add_rmsnorm_fp4_fwd", quant_args),
                       ("add_rmsnorm_fp4_fwd_with_config", quant_args + [cfgp]),
                       ("rmsnorm_fp4_fwd", [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp]),
                       ("rmsnorm_fp4_fwd_with_config", [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp, cfgp]),
                       ("dradd_resolve_config", [_i64, _i64, ctypes.c_int, ctypes.c_int, cfgp]),
                       ("fused_qk_rmsnorm_group_quant_fwd", qk_args),
                       ("fused_qk_rmsnorm_group_quant_fwd_with_config", qk_args + [cfgp]),
                       ("dradd_qk_resolve_config", [_i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                                    cfgp, ctypes.POINTER(_QkPlan)]),
                       ("lse_merge_fwd", [_vp, _vp, _vp, _i64, _vp]),
                       ("lse_merge_2d_fwd", [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _vp]),
                       ("lse_merge_2d_fwd_with_config", [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _vp, cfgp]),
                       ("invariant_unary_fwd", [_vp, _vp, _i64, ctypes.c_int, _vp]),
                       ("invariant_unary_fwd_with_config", [_vp, _vp, _i64, ctypes.c_int, _vp, cfgp]),
                       ("dradd_device_status", [_vp, ctypes.c_int]),
                       ("dradd_last_device_status", [_vp]),
                       ("dradd_bf16_convert_range", [_vp, ctypes.c_uint64, _i64, ctypes.c_int, _vp])]:
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.dradd_status_string.argtypes = [ctypes.c_int]
    L.dradd_status_string.restype = ctypes.c_char_p
    L.dradd_abi_version.argtypes = []
    L.dradd_abi_version.restype = ctypes.c_int
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().dradd_status_string(int(status)).decode()


def abi_version() -> int:
    return int(lib().dradd_abi_version())


def _check(status: int, where: str):
    if status != 0:
        raise DraddError(status, where)


# ----------------------------------------------------------- tensor marshalling
def _torch():
    import torch
    return torch


def _stream_handle(stream, device) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _bf16_ptr(t, name: str, n: int | None = None) -> int:
    torch = _torch()
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must hold bf16 (got {t.dtype})")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if n is not None and t.numel() != n:
        raise ValueError(f"{name} has {t.numel()} elements, expected {n}")
    return t.data_ptr()


def _shape(x, hidden):
    hidden = int(x.shape[-1]) if hidden is None else int(hidden)
    n_rows = x.numel() // hidden if hidden > 0 else 0
    return n_rows, hidden


def add_rmsnorm_fwd(x, residual, weight, eps: float = 1e-6, *, out=None, residual_out=None,
                    stream=None, config: LaunchConfig | None = None):
    """out, residual_out = rmsnorm2d_fwd_with_add(x, residual, weight, eps).

    x, residual: CUDA bf16 tensors [..., hidden]; weight: [hidden].  out and
    residual_out are allocated like x unless given (residual_out may be
    `residual` itself, out may be `x`).  Enqueued on `stream` (default: the
    current stream of x's device)."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    if out is None:
        out = torch.empty_like(x)
    if residual_out is None:
        residual_out = torch.empty_like(x)
    args = (_bf16_ptr(out, "out", n), _bf16_ptr(residual_out, "residual_out", n),
            _bf16_ptr(x, "x", n), _bf16_ptr(residual, "residual", n),
            _bf16_ptr(weight, "weight", hidden), float(eps), n_rows, hidden,
            _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().add_rmsnorm_fwd(*args), "add_rmsnorm_fwd")
        else:
            c = config._c()
            _check(lib().add_rmsnorm_fwd_with_config(*args, ctypes.byref(c)),
                   "add_rmsnorm_fwd_with_config")
    return out, residual_out


def _check_quant_outs(out_q, scale, n, n_rows):
    torch = _torch()
    if out_q.dtype != torch.int8 or not out_q.is_cuda or not out_q.is_contiguous() or out_q.numel() != n:
        raise ValueError("out_q must be a contiguous CUDA int8 tensor shaped like x")
    if (scale.dtype != torch.float32 or not scale.is_cuda or not scale.is_contiguous()
            or scale.numel() != n_rows):
        raise ValueError("scale must be a contiguous CUDA float32 tensor with one entry per row")


def add_rmsnorm_quant_fwd(x, residual, weight, eps: float = 1e-6, *, out_q=None, scale=None,
                          residual_out=None, stream=None, config: LaunchConfig | None = None):
    """out_q (int8), scale (fp32 per row), residual_out (bf16) of the quant variant."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    if out_q is None:
        out_q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    if residual_out is None:
        residual_out = torch.empty_like(x)
    _check_quant_outs(out_q, scale, n, n_rows)
    args = (out_q.data_ptr(), scale.data_ptr(), _bf16_ptr(residual_out, "residual_out", n),
            _bf16_ptr(x, "x", n), _bf16_ptr(residual, "residual", n),
            _bf16_ptr(weight, "weight", hidden), float(eps), n_rows, hidden,
            _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().add_rmsnorm_quant_fwd(*args), "add_rmsnorm_quant_fwd")
        else:
            c = config._c()
            _check(lib().add_rmsnorm_quant_fwd_with_config(*args, ctypes.byref(c)),
                   "add_rmsnorm_quant_fwd_with_config")
    return out_q, scale, residual_out


def add_rmsnorm_fwd_with_config(x, residual, weight, eps, config: LaunchConfig, **kw):
    return add_rmsnorm_fwd(x, residual, weight, eps, config=config, **kw)


def add_rmsnorm_quant_fwd_with_config(x, residual, weight, eps, config: LaunchConfig, **kw):
    return add_rmsnorm_quant_fwd(x, residual, weight, eps, config=config, **kw)


def resolve_config(n_rows: int, hidden: int, quant: bool = False, sm_count: int = 152,
                   config: LaunchConfig | None = None, add: bool = True, fp8: bool = False,
                   fp4: bool = False) -> LaunchConfig:
    """The configuration the library would launch for this shape (no GPU
    work when sm_count > 0); add=False for plain RMSNorm, fp8=True / fp4=True
    for the e4m3 / e2m1 output."""
    if fp4:
        op = OP_ADD_RMSNORM_FP4 if add else OP_RMSNORM_FP4
    elif fp8:
        op = OP_ADD_RMSNORM_FP8 if add else OP_RMSNORM_FP8
    else:
        op = (OP_ADD_RMSNORM if add else OP_RMSNORM) + (1 if quant else 0)
    c = (config or LaunchConfig())._c()
    _check(lib().dradd_resolve_config(int(n_rows), int(hidden), op, int(sm_count), ctypes.byref(c)),
           "dradd_resolve_config")
    return LaunchConfig._from_c(c)


def rmsnorm_fwd(x, weight, eps: float = 1e-6, *, out=None, stream=None,
                config: LaunchConfig | None = None):
    """Plain RMSNorm (no residual): out = bf16_rne((x * inv) * weight)."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    if out is None:
        out = torch.empty_like(x)
    args = (_bf16_ptr(out, "out", n), _bf16_ptr(x, "x", n), _bf16_ptr(weight, "weight", hidden),
            float(eps), n_rows, hidden, _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().rmsnorm_fwd(*args), "rmsnorm_fwd")
        else:
            c = config._c()
            _check(lib().rmsnorm_fwd_with_config(*args, ctypes.byref(c)), "rmsnorm_fwd_with_config")
    return out


def rmsnorm_quant_fwd(x, weight, eps: float = 1e-6, *, out_q=None, scale=None, stream=None,
                      config: LaunchConfig | None = None):
    """Plain RMSNorm with per-row symmetric int8 out: (out_q, scale)."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    if out_q is None:
        out_q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _check_quant_outs(out_q, scale, n, n_rows)
    args = (out_q.data_ptr(), scale.data_ptr(), _bf16_ptr(x, "x", n), _bf16_ptr(weight, "weight", hidden),
            float(eps), n_rows, hidden, _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().rmsnorm_quant_fwd(*args), "rmsnorm_quant_fwd")
        else:
            c = config._c()
            _check(lib().rmsnorm_quant_fwd_with_config(*args, ctypes.byref(c)),
                   "rmsnorm_quant_fwd_with_config")
    return out_q, scale


def _fp8_outs(x, out_q, scale):
    torch = _torch()
    if out_q is None:
        out_q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    if out_q.dtype != torch.uint8:
        raise ValueError("out_q must hold uint8 e4m3 codes")
    return out_q, scale


def add_rmsnorm_fp8_fwd(x, residual, weight, eps: float = 1e-6, *, out_q=None, scale=None,
                        residual_out=None, stream=None, config: LaunchConfig | None = None):
    """Residual-add + RMSNorm with per-row e4m3 out: (out_q uint8 codes,
    scale, residual_out)."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    out_q, scale = _fp8_outs(x, out_q, scale)
    if residual_out is None:
        residual_out = torch.empty_like(x)
    _check_quant_outs(out_q.view(torch.int8), scale, n, n_rows)
    args = (out_q.data_ptr(), scale.data_ptr(), _bf16_ptr(residual_out, "residual_out", n),
            _bf16_ptr(x, "x", n), _bf16_ptr(residual, "residual", n),
            _bf16_ptr(weight, "weight", hidden), float(eps), n_rows, hidden,
            _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().add_rmsnorm_fp8_fwd(*args), "add_rmsnorm_fp8_fwd")
        else:
            c = config._c()
            _check(lib().add_rmsnorm_fp8_fwd_with_config(*args, ctypes.byref(c)),
                   "add_rmsnorm_fp8_fwd_with_config")
    return out_q, scale, residual_out


def rmsnorm_fp8_fwd(x, weight, eps: float = 1e-6, *, out_q=None, scale=None, stream=None,
                    config: LaunchConfig | None = None):
    """Plain RMSNorm with per-row e4m3 out: (out_q uint8 codes, scale)."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    out_q, scale = _fp8_outs(x, out_q, scale)
    _check_quant_outs(out_q.view(torch.int8), scale, n, n_rows)
    args = (out_q.data_ptr(), scale.data_ptr(), _bf16_ptr(x, "x", n), _bf16_ptr(weight, "weight", hidden),
            float(eps), n_rows, hidden, _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().rmsnorm_fp8_fwd(*args), "rmsnorm_fp8_fwd")
        else:
            c = config._c()
            _check(lib().rmsnorm_fp8_fwd_with_config(*args, ctypes.byref(c)), "rmsnorm_fp8_fwd_with_config")
    return out_q, scale


def _fp4_outs(x, out_q, scale):
    torch = _torch()
    if out_q is None:
        out_q = torch.empty(x.shape[:-1] + (x.shape[-1] // 2,), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    if (out_q.dtype != torch.uint8 or not out_q.is_cuda or not out_q.is_contiguous()
            or out_q.numel() * 2 != x.numel()):
        raise ValueError("out_q must be a contiguous CUDA uint8 tensor of hidden / 2 bytes per row")
    if (scale.dtype != torch.float32 or not scale.is_cuda or not scale.is_contiguous()
            or scale.numel() * x.shape[-1] != x.numel()):
        raise ValueError("scale must be a contiguous CUDA float32 tensor with one entry per row")
    return out_q, scale


def add_rmsnorm_fp4_fwd(x, residual, weight, eps: float = 1e-6, *, out_q=None, scale=None,
                        residual_out=None, stream=None, config: LaunchConfig | None = None):
    """Residual-add + RMSNorm with per-row e2m1 out: (out_q [..., h/2] uint8,
    two codes per byte with the even element in the low nibble; scale;
    residual_out)."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    out_q, scale = _fp4_outs(x, out_q, scale)
    if residual_out is None:
        residual_out = torch.empty_like(x)
    args = (out_q.data_ptr(), scale.data_ptr(), _bf16_ptr(residual_out, "residual_out", n),
            _bf16_ptr(x, "x", n), _bf16_ptr(residual, "residual", n),
            _bf16_ptr(weight, "weight", hidden), float(eps), n_rows, hidden,
            _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().add_rmsnorm_fp4_fwd(*args), "add_rmsnorm_fp4_fwd")
        else:
            c = config._c()
            _check(lib().add_rmsnorm_fp4_fwd_with_config(*args, ctypes.byref(c)),
                   "add_rmsnorm_fp4_fwd_with_config")
    return out_q, scale, residual_out


def rmsnorm_fp4_fwd(x, weight, eps: float = 1e-6, *, out_q=None, scale=None, stream=None,
                    config: LaunchConfig | None = None):
    """Plain RMSNorm with per-row e2m1 out: (out_q [..., h/2] uint8, scale)."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    out_q, scale = _fp4_outs(x, out_q, scale)
    args = (out_q.data_ptr(), scale.data_ptr(), _bf16_ptr(x, "x", n), _bf16_ptr(weight, "weight", hidden),
            float(eps), n_rows, hidden, _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().rmsnorm_fp4_fwd(*args), "rmsnorm_fp4_fwd")
        else:
            c = config._c()
            _check(lib().rmsnorm_fp4_fwd_with_config(*args, ctypes.byref(c)), "rmsnorm_fp4_fwd_with_config")
    return out_q, scale


def residual_add_fwd(x, residual, *, residual_out=None, stream=None):
    """residual_out = bf16_rne(fp32(x) + fp32(residual))."""
    torch = _torch()
    n_rows, hidden = _shape(x, None)
    n = n_rows * hidden
    if residual_out is None:
        residual_out = torch.empty_like(x)
    args = (_bf16_ptr(residual_out, "residual_out", n), _bf16_ptr(x, "x", n),
            _bf16_ptr(residual, "residual", n), n_rows, hidden, _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        _check(lib().residual_add_fwd(*args), "residual_add_fwd")
    return residual_out


def fused_qk_rmsnorm_group_quant_fwd(q, q_weight, k, k_weight, q_eps: float = 1e-6, k_eps: float = 1e-6, *,
                                     group_size: int = 0, q_residual=None, q_out=None, q_scale=None,
                                     q_residual_out=None, k_out=None, stream=None,
                                     config: LaunchConfig | None = None):
    """Fused q/k RMSNorm in one launch: q rows (optionally + q_residual) with
    bf16 out (group_size 0) or per-group e4m3 out, k rows plain with bf16
    out.  Returns (q_out, q_scale, q_residual_out, k_out); q_scale is None
    for bf16 out, q_residual_out None without a q residual."""
    torch = _torch()
    n_q, hq = _shape(q, None)
    n_k, hk = _shape(k, None)
    nq, nk = n_q * hq, n_k * hk
    g = int(group_size)
    if q_out is None:
        q_out = torch.empty(q.shape, dtype=torch.uint8 if g else torch.bfloat16, device=q.device)
    if g:
        if q_out.dtype != torch.uint8:
            raise ValueError("q_out must hold uint8 e4m3 codes")
        if q_scale is None:
            q_scale = torch.empty((*q.shape[:-1], hq // g if hq % g == 0 else 0), dtype=torch.float32,
                                  device=q.device)
        _check_quant_outs(q_out.view(torch.int8), q_scale.view(-1), nq, n_q * (hq // g) if hq % g == 0 else 0)
        q_out_ptr, scale_ptr = q_out.data_ptr(), q_scale.data_ptr()
    else:
        q_out_ptr, scale_ptr = _bf16_ptr(q_out, "q_out", nq), 0
    if q_residual is not None and q_residual_out is None:
        q_residual_out = torch.empty_like(q)
    if k_out is None:
        k_out = torch.empty_like(k)
    args = (q_out_ptr, scale_ptr,
            _bf16_ptr(q_residual_out, "q_residual_out", nq) if q_residual is not None else 0,
            _bf16_ptr(k_out, "k_out", nk), _bf16_ptr(q, "q", nq),
            _bf16_ptr(q_residual, "q_residual", nq) if q_residual is not None else 0,
            _bf16_ptr(q_weight, "q_weight", hq), _bf16_ptr(k, "k", nk), _bf16_ptr(k_weight, "k_weight", hk),
            float(q_eps), float(k_eps), n_q, hq, n_k, hk, g, _stream_handle(stream, q.device))
    with torch.cuda.device(q.device):
        if config is None:
            _check(lib().fused_qk_rmsnorm_group_quant_fwd(*args), "fused_qk_rmsnorm_group_quant_fwd")
        else:
            c = config._c()
            _check(lib().fused_qk_rmsnorm_group_quant_fwd_with_config(*args, ctypes.byref(c)),
                   "fused_qk_rmsnorm_group_quant_fwd_with_config")
    return q_out, (q_scale if g else None), (q_residual_out if q_residual is not None else None), k_out


def qk_resolve_config(n_q_rows: int, q_hidden: int, n_k_rows: int, k_hidden: int, group_size: int = 0,
                      q_residual: bool = False, sm_count: int = 152,
                      config: LaunchConfig | None = None) -> QkPlan:
    """The plan the fused q/k call would use.  sm_count > 0: no GPU needed
    (the real call then sizes the automatic grid by the device's
    occupancy); sm_count <= 0: the current device's plan, grid included."""
    plan = _QkPlan()
    c = config._c() if config is not None else None
    _check(lib().dradd_qk_resolve_config(int(n_q_rows), int(q_hidden), int(n_k_rows), int(k_hidden),
                                         int(group_size), int(bool(q_residual)), int(sm_count),
                                         ctypes.byref(c) if c is not None else None, ctypes.byref(plan)),
           "dradd_qk_resolve_config")
    return QkPlan(*(getattr(plan, f) for f, _ in _QkPlan._fields_))


UNARY_OPS = {"log1p": 0, "cosh": 1, "exp": 2}


def _f32_ptr(t, name: str) -> int:
    torch = _torch()
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32 (got {t.dtype})")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr()


def _elem_stride(t, name: str) -> tuple[int, int, int]:
    """(rows, cols, row stride) of a 1-D or 2-D tensor with unit column stride."""
    if t.dim() == 1:
        if t.numel() > 1 and t.stride(0) != 1:
            raise ValueError(f"{name} must have unit stride")
        return (1 if t.numel() else 0), t.numel(), t.numel()
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 1-D, or 2-D with unit column stride")
    return t.shape[0], t.shape[1], t.stride(0) if t.shape[0] > 1 else t.shape[1]


def lse_merge_fwd(lse_a, lse_b, *, out=None, stream=None, config: LaunchConfig | None = None):
    """log(e^a + e^b) elementwise (fp32): 1-D tensors, or 2-D views with any
    row stride (e.g. the second half of each row of a running lse).  out may
    be lse_a or lse_b (in place)."""
    torch = _torch()
    if out is None:
        out = torch.empty(lse_a.shape, dtype=torch.float32, device=lse_a.device)
    ra, ca, sa = _elem_stride(lse_a, "lse_a")
    rb, cb, sb = _elem_stride(lse_b, "lse_b")
    ro, co, so = _elem_stride(out, "out")
    if (ra, ca) != (rb, cb) or (ra, ca) != (ro, co):
        raise ValueError("lse_a, lse_b and out must have the same shape")
    args = (_f32_ptr(out, "out"), so, _f32_ptr(lse_a, "lse_a"), sa, _f32_ptr(lse_b, "lse_b"), sb, ra, ca,
            _stream_handle(stream, lse_a.device))
    with torch.cuda.device(lse_a.device):
        if config is None:
            _check(lib().lse_merge_2d_fwd(*args), "lse_merge_2d_fwd")
        else:
            c = config._c()
            _check(lib().lse_merge_2d_fwd_with_config(*args, ctypes.byref(c)), "lse_merge_2d_fwd_with_config")
    return out


def invariant_unary_fwd(x, op: str = "log1p", *, out=None, stream=None, config: LaunchConfig | None = None):
    """log1p / cosh / exp of a contiguous fp32 tensor, launch-invariant."""
    torch = _torch()
    if out is None:
        out = torch.empty_like(x)
    if not x.is_contiguous() or not out.is_contiguous() or out.numel() != x.numel():
        raise ValueError("x and out must be contiguous and the same size")
    args = (_f32_ptr(out, "out"), _f32_ptr(x, "x"), x.numel(), UNARY_OPS[op], _stream_handle(stream, x.device))
    with torch.cuda.device(x.device):
        if config is None:
            _check(lib().invariant_unary_fwd(*args), "invariant_unary_fwd")
        else:
            c = config._c()
            _check(lib().invariant_unary_fwd_with_config(*args, ctypes.byref(c)), "invariant_unary_fwd_with_config")
    return out


def device_status(stream=None, clear: bool = True, device=None) -> int:
    """Synchronise the stream and return the device status (0, TIMEOUT=8 or
    UNDRAINED=10)."""
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(device):
        return int(lib().dradd_device_status(_stream_handle(stream, device), int(clear)))


def last_device_status(stream=None, device=None) -> int:
    """Synchronise the stream, return the device status (0, TIMEOUT=8 or
    UNDRAINED=10) recorded since the last read, and reset it."""
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(device):
        return int(lib().dradd_last_device_status(_stream_handle(stream, device)))


def bf16_convert_range(out, first: int, count: int, method: int = 0, stream=None):
    """Test hook: device conversion of fp32 patterns first..first+count-1."""
    torch = _torch()
    _check(lib().dradd_bf16_convert_range(_bf16_ptr(out, "out"), int(first), int(count), int(method),
                                          _stream_handle(stream, out.device)),
           "dradd_bf16_convert_range")
    return out
