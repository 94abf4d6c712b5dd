"""CUDA path vs the CPU oracle, element by element, bit for bit: residual_out
and out (bf16 variant), q, scale and residual_out (int8 variant), on every
workload at full size, in the automatic launch configuration (the one the
bench times), plus ragged and edge shapes.  Also within 1 bf16 ulp of fp64."""
import numpy as np
import pytest
import torch

import refs
from deterministic_residual_add_gb300 import inputs
from gpu_util import THREADS, assert_bits_equal, gpu_fwd, gpu_quant, max_ulp_vs_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "2048x4096", "4096x8192", "16384x4096", "8192x2048"])
def test_bf16_workloads_bit_exact(orc, name):
    c = inputs.WORKLOADS[name].make()
    out, ro = gpu_fwd(c["x"], c["residual"], c["weight"], c["eps"])
    eo, ero = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"], threads=THREADS)
    assert_bits_equal(ro, ero, f"{name} residual_out")
    assert_bits_equal(out, eo, f"{name} out")
    rows = slice(0, 256)
    assert max_ulp_vs_f64(out[rows], c["x"][rows], c["residual"][rows], c["weight"], c["eps"]) <= 1.0


def test_chain_shape_first_call_bit_exact(orc):
    ch = inputs.CHAIN4096
    r0, w = ch.initial()
    x0 = ch.delta(0)
    out, ro = gpu_fwd(x0, r0, w, ch.eps)
    eo, ero = orc.add_rmsnorm_fwd(x0, r0, w, ch.eps, threads=THREADS)
    assert_bits_equal(ro, ero, "4096x4096 residual_out")
    assert_bits_equal(out, eo, "4096x4096 out")


@pytest.mark.parametrize("name", ["quant2048x16384", "2048x4096", "8192x2048", "8192x4096"])
def test_quant_workload_bit_exact(orc, name):
    c = inputs.WORKLOADS[name].make()
    q, scale, ro = gpu_quant(c["x"], c["residual"], c["weight"], c["eps"])
    eq, escale, ero = orc.add_rmsnorm_quant_fwd(c["x"], c["residual"], c["weight"], c["eps"],
                                               threads=THREADS)
    assert_bits_equal(ro, ero, "quant residual_out")
    assert_bits_equal(scale.view(np.uint32), escale.view(np.uint32), "quant scale")
    assert_bits_equal(q.view(np.uint8), eq.view(np.uint8), "quant q")
    y64, _ = refs.add_rmsnorm_f64(c["x"][:64], c["residual"][:64], c["weight"], c["eps"])
    q64, _ = refs.quant_f64(y64)
    assert np.abs(q[:64].astype(np.int64) - q64).max() <= 1


@pytest.mark.parametrize("n_rows,hidden", [
    (1, 8), (3, 16), (65, 24), (7, 64), (5, 200), (33, 1000), (3, 1024), (17, 3000),
    (9, 4104), (2, 8192), (3, 8200), (4, 12288), (2, 16384), (2, 24576), (1, 32768),
])
def test_ragged_shapes_bit_exact(orc, n_rows, hidden):
    g = inputs.generator(n_rows * 100003 + hidden)
    x = inputs.normal_bf16(g, (n_rows, hidden), 0.0, 1.0)
    r = inputs.normal_bf16(g, (n_rows, hidden), 0.0, 4.0)
    w = inputs.normal_bf16(g, (hidden,), 1.0, 0.1)
    out, ro = gpu_fwd(x, r, w, 1e-6)
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6, threads=THREADS)
    assert_bits_equal(ro, ero, "residual_out")
    assert_bits_equal(out, eo, "out")
    q, scale, ro2 = gpu_quant(x, r, w, 1e-6)
    eq, escale, _ = orc.add_rmsnorm_quant_fwd(x, r, w, 1e-6, threads=THREADS)
    assert_bits_equal(ro2, ero, "quant residual_out")
    assert_bits_equal(scale.view(np.uint32), escale.view(np.uint32), "scale")
    assert_bits_equal(q.view(np.uint8), eq.view(np.uint8), "q")


def test_rounding_edge_rows(orc):
    c = inputs.edge_rows(16, 1024)
    out, ro = gpu_fwd(c["x"], c["residual"], c["weight"], c["eps"])
    eo, ero = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"])
    assert_bits_equal(ro, ero, "edge residual_out")
    assert_bits_equal(out, eo, "edge out")
    # the ties resolve to even (see the edge table in tests/pins.py)
    got = set(zip(refs.u16(c["x"]).ravel().tolist(), ro.ravel().tolist()))
    assert (0x3F80, 0x3F80) in got and (0x3F81, 0x3F82) in got


def test_tie_past_largest_finite_rounds_to_inf(orc):
    # 0x7F7F + 0x7B00 sums to 0x7F7F8000, a tie that rounds to +inf; the
    # row's sum of squares overflows, so out is compared on NaN-ness only.
    x = torch.full((2, 64), 0, dtype=torch.int16)
    r = torch.zeros_like(x)
    x[0, :] = 0x7F7F
    r[0, :] = 0x7B00
    x[1, 5] = 0x3F80
    xb, rb = x.view(torch.bfloat16), r.view(torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    out, ro = gpu_fwd(xb, rb, w, 1e-6)
    eo, ero = orc.add_rmsnorm_fwd(xb, rb, w, 1e-6)
    assert_bits_equal(ro, ero, "residual_out")
    assert np.all(ro[0] == 0x7F80)
    nan_got = np.isnan(refs.bf16_value(out))
    nan_exp = np.isnan(refs.bf16_value(eo))
    assert np.array_equal(nan_got, nan_exp)
    assert_bits_equal(out[~nan_exp], eo[~nan_exp], "finite out")


def test_special_rows(orc):
    """Zero rows, cancelling rows, subnormal rows, huge rows and constant
    rows in one call."""
    h = 2048
    g = inputs.generator(99)
    x = refs.u16(inputs.normal_bf16(g, (8, h), 0.0, 1.0)).copy()
    r = refs.u16(inputs.normal_bf16(g, (8, h), 0.0, 1.0)).copy()
    x[0] = 0; r[0] = 0                              # zero row
    r[1] = x[1] ^ 0x8000                            # x + (-x)
    x[2] = (x[2] & 0x807F); r[2] = (r[2] & 0x807F)  # subnormals
    x[3] = (x[3] & 0x807F) | 0x7E00                 # ~1e38 magnitudes (no overflow in acc)
    r[3] = 0
    x[4] = 0x4040; r[4] = 0                         # constant 3.0
    x[5] = (x[5] & 0x807F) | 0x0080; r[5] = 0       # smallest normals
    w = refs.u16(inputs.normal_bf16(g, (h,), 1.0, 0.1))
    tx, tr, tw = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) for a in (x, r, w))
    out, ro = gpu_fwd(tx, tr, tw, 1e-6)
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6)
    assert_bits_equal(ro, ero, "residual_out")
    assert_bits_equal(out, eo, "out")


@pytest.mark.parametrize("eps", [0.0, 1e-12, 1e-6, 0.5, 1e4])
def test_eps_values(orc, eps):
    c = inputs.WORKLOADS["tiny"].make()
    out, ro = gpu_fwd(c["x"], c["residual"], c["weight"], eps)
    eo, ero = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], eps)
    assert_bits_equal(out, eo, f"out eps={eps}")
