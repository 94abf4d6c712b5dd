"""The log-sum-exp merge and invariant unary entry points on the host,
without a GPU: argument checks only.  Every call made here returns before
any CUDA runtime call; nothing is launched."""
import ctypes

import pytest

import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import build as drbuild

MB = 1 << 20
BASE = 1 << 42
OUT, A, B = (BASE + i * 256 * MB for i in range(3))


@pytest.fixture(scope="module")
def L():
    drbuild.build()
    return dr.lib()


def merge2d(L, out=OUT, so=64, a=A, sa=64, b=B, sb=64, rows=4, cols=64, cfg=None):
    if cfg is None:
        return L.lse_merge_2d_fwd(out, so, a, sa, b, sb, rows, cols, None)
    c = cfg._c()
    return L.lse_merge_2d_fwd_with_config(out, so, a, sa, b, sb, rows, cols, None, ctypes.byref(c))


@pytest.mark.parametrize("kw,code", [
    (dict(rows=-1), 2), (dict(cols=-1), 2), (dict(so=63), 2), (dict(sa=10), 2), (dict(sb=0), 2),
    (dict(rows=1 << 60, so=1 << 10, sa=1 << 10, sb=1 << 10), 2),
    (dict(out=0), 1), (dict(a=0), 1), (dict(b=0), 1),
    (dict(out=OUT + 2), 4), (dict(a=A + 1), 4), (dict(b=B + 3), 4),
    (dict(out=A + 4), 6),            # shifted alias of a
    (dict(out=A, so=128, sa=64), 6),  # same address, other stride
    (dict(out=B + 256), 6),
    (dict(rows=0), 0), (dict(cols=0), 0),
])
def test_merge_argument_errors(L, kw, code):
    assert merge2d(L, **kw) == code


def test_merge_in_place_passes_the_checks(L):
    # exact aliasing reaches the device query (which fails without a GPU)
    assert merge2d(L, out=A) not in (1, 2, 4, 6, 9)
    assert merge2d(L, out=B) not in (1, 2, 4, 6, 9)
    # second half of each row of a running lse, in place
    assert merge2d(L, out=A + 128, so=64, a=A + 128, sa=64, b=B, sb=32, rows=8, cols=32) not in (1, 2, 4, 6, 9)


@pytest.mark.parametrize("cfg", [dr.LaunchConfig(threads_per_row=16), dr.LaunchConfig(threads_per_row=2048),
                                 dr.LaunchConfig(threads_per_row=96), dr.LaunchConfig(blocks_per_thread=3),
                                 dr.LaunchConfig(blocks_per_thread=16), dr.LaunchConfig(variant=1),
                                 dr.LaunchConfig(rows_per_cta=1), dr.LaunchConfig(stages=1),
                                 dr.LaunchConfig(fault_inject=1), dr.LaunchConfig(wait_limit_us=5),
                                 dr.LaunchConfig(grid_ctas=-1), dr.LaunchConfig(serialize=2)])
def test_merge_bad_configs(L, cfg):
    assert merge2d(L, cfg=cfg) == 9


def test_with_config_needs_config(L):
    assert L.lse_merge_2d_fwd_with_config(OUT, 64, A, 64, B, 64, 4, 64, None, None) == 1
    assert L.invariant_unary_fwd_with_config(OUT, A, 64, 0, None, None) == 1


@pytest.mark.parametrize("args,code", [
    ((OUT, A, -1, 0), 2), ((OUT, A, 64, 3), 9), ((OUT, A, 64, -1), 9), ((0, A, 64, 0), 1), ((OUT, 0, 64, 1), 1),
    ((OUT + 2, A, 64, 0), 4), ((OUT, A + 1, 64, 2), 4), ((A + 8, A, 64, 0), 6), ((OUT, A, 0, 0), 0),
])
def test_unary_argument_errors(L, args, code):
    assert L.invariant_unary_fwd(*args, None) == code


def test_flat_merge_shapes(L):
    assert L.lse_merge_fwd(OUT, A, B, -5, None) == 2
    assert L.lse_merge_fwd(OUT, A, B, 0, None) == 0
    assert L.lse_merge_fwd(0, A, B, 7, None) == 1
    assert L.lse_merge_fwd(A + 4, A, B, 7, None) == 6
