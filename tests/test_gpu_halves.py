"""The two halves of the op on the GPU: plain RMSNorm (bf16 and int8 out)
and the residual update alone, bit for bit against the oracle, over the
workload shapes, ragged shapes and launch configurations; outputs in place."""
import hashlib

import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import THREADS, assert_bits_equal, dev, to_dev

pytestmark = pytest.mark.gpu


def case(n, h, seed):
    g = inputs.generator(seed)
    return (inputs.normal_bf16(g, (n, h), 0.0, 1.0), inputs.normal_bf16(g, (n, h), 0.0, 4.0),
            inputs.normal_bf16(g, (h,), 1.0, 0.1))


@pytest.mark.parametrize("n,h", [(4096, 4096), (2048, 16384), (4096, 8192), (65, 24), (33, 1000),
                                 (7, 3000), (3, 32768), (1, 8), (5, 200)])
def test_rmsnorm_bit_exact(orc, n, h):
    x, _, w = case(n, h, n * 7 + h)
    out = dr.rmsnorm_fwd(to_dev(x), to_dev(w), 1e-6)
    q, s = dr.rmsnorm_quant_fwd(to_dev(x), to_dev(w), 1e-6)
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(out), orc.rmsnorm_fwd(x, w, 1e-6, threads=THREADS), "rmsnorm out")
    eq, es = orc.rmsnorm_quant_fwd(x, w, 1e-6, threads=THREADS)
    assert_bits_equal(q.cpu().numpy().view(np.uint8), eq.view(np.uint8), "rmsnorm q")
    assert_bits_equal(s.cpu().numpy().view(np.uint32), es.view(np.uint32), "rmsnorm scale")


def test_rmsnorm_negative_zero_and_in_place(orc):
    h = 1024
    x = np.zeros((2, h), np.uint16)
    x[:, ::2] = 0x8000
    x[:, 1] = 0x3F80
    tx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    w = torch.ones(h, dtype=torch.bfloat16)
    dx = to_dev(tx)
    dr.rmsnorm_fwd(dx, to_dev(w), 1e-6, out=dx)  # in place
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(dx), orc.rmsnorm_fwd(x, w, 1e-6), "in-place rmsnorm with -0")


def test_rmsnorm_one_result_group(orc):
    x, _, w = case(1024, 8192, 5)
    dx, dw = to_dev(x), to_dev(w)
    cfgs = [None, dr.LaunchConfig(variant=1, threads_per_row=512),
            dr.LaunchConfig(variant=1, threads_per_row=128, rows_per_cta=4),
            dr.LaunchConfig(variant=2, threads_per_row=1024, stages=4),
            dr.LaunchConfig(variant=2, threads_per_row=256, stages=2, grid_ctas=9),
            dr.LaunchConfig(variant=2, threads_per_row=128, stages=6, serialize=1)]
    digests = set()
    for cfg in cfgs:
        out = dr.rmsnorm_fwd(dx, dw, 1e-6, config=cfg)
        torch.cuda.synchronize()
        digests.add(hashlib.sha256(refs.u16(out).tobytes()).hexdigest())
    assert len(digests) == 1
    assert digests == {hashlib.sha256(orc.rmsnorm_fwd(x, w, 1e-6, threads=THREADS).tobytes()).hexdigest()}


@pytest.mark.parametrize("n,h", [(4096, 4096), (3, 24), (1, 8), (129, 1000), (2, 32768)])
def test_residual_add_bit_exact(orc, n, h):
    x, r, _ = case(n, h, n + 3 * h)
    ro = dr.residual_add_fwd(to_dev(x), to_dev(r))
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(ro), orc.residual_add_fwd(x, r), "residual_add")
    dx, drs = to_dev(x), to_dev(r)
    dr.residual_add_fwd(dx, drs, residual_out=drs)  # in place over the residual
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(drs), orc.residual_add_fwd(x, r), "in-place residual_add")


def test_residual_add_edges(orc):
    c = inputs.edge_rows(16, 1024)
    ro = dr.residual_add_fwd(to_dev(c["x"]), to_dev(c["residual"]))
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(ro), orc.residual_add_fwd(c["x"], c["residual"]), "edge residual_add")
