"""Helpers for the GPU tests: run the CUDA path through the binding (C ABI)
and compare with the oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import refs
import deterministic_residual_add_gb300 as dr

THREADS = oracle.default_threads()


def dev():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    return torch.device("cuda", 0)


def to_dev(t: torch.Tensor) -> torch.Tensor:
    return t.to(dev())


def gpu_fwd(x, r, w, eps, config=None):
    out, ro = dr.add_rmsnorm_fwd(to_dev(x), to_dev(r), to_dev(w), eps, config=config)
    torch.cuda.synchronize()
    return refs.u16(out), refs.u16(ro)


def gpu_quant(x, r, w, eps, config=None):
    q, scale, ro = dr.add_rmsnorm_quant_fwd(to_dev(x), to_dev(r), to_dev(w), eps, config=config)
    torch.cuda.synchronize()
    return q.cpu().numpy(), scale.cpu().numpy(), refs.u16(ro)


def assert_bits_equal(got: np.ndarray, exp: np.ndarray, what: str):
    if np.array_equal(got, exp):
        return
    bad = np.argwhere(got != exp)
    i = tuple(bad[0])
    raise AssertionError(f"{what}: {len(bad)} of {got.size} differ; first at {i}: "
                         f"got {hex(int(got[i]))} expected {hex(int(exp[i]))}")


def max_ulp_vs_f64(out_bits, x, r, w, eps) -> float:
    y64, _ = refs.add_rmsnorm_f64(x, r, w, eps)
    return float((np.abs(refs.bf16_value(out_bits) - y64) / refs.ulp_bf16(y64)).max())
