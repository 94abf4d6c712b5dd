"""The split-row variant (a thread-block cluster of 2 or 4 CTAs per row, the
slice sums combined through distributed shared memory) returns the oracle's
bits, the same bits as every other variant under every configuration, and
recovers from an expired wait as a whole cluster."""
import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import THREADS, assert_bits_equal, dev

pytestmark = pytest.mark.gpu

SHAPES = [(64, 1024), (100, 4096), (37, 4104), (2048, 4096), (16, 16384), (8, 32768), (3, 8200), (1, 2048)]


def make(n, h, seed):
    g = inputs.generator(seed)
    x = inputs.normal_bf16(g, (n, h), 0.0, 1.0)
    r = inputs.normal_bf16(g, (n, h), 0.0, 4.0)
    w = inputs.normal_bf16(g, (h,), 1.0, 0.1)
    return x, r, w


@pytest.mark.parametrize("C", [2, 4])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_parity(orc, shape, C):
    n, h = shape
    if (1 << (h - 1).bit_length()) // 8 // C < 32:
        pytest.skip("slice narrower than 256 elements")
    x, r, w = make(n, h, n + h + C)
    d = dev()
    cfg = dr.LaunchConfig(variant=dr.VARIANT_SPLIT, cluster_ctas=C)
    out, ro = dr.add_rmsnorm_fwd(x.to(d), r.to(d), w.to(d), 1e-6, config=cfg)
    plain = dr.rmsnorm_fwd(x.to(d), w.to(d), 1e-6, config=cfg)
    torch.cuda.synchronize()
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6, threads=THREADS)
    assert_bits_equal(refs.u16(ro), ero, "residual_out")
    assert_bits_equal(refs.u16(out), eo, "out")
    assert_bits_equal(refs.u16(plain), orc.rmsnorm_fwd(x, w, 1e-6, threads=THREADS), "plain out")
    assert dr.device_status() == 0


def test_configuration_invariance(orc):
    n, h = 300, 8192
    x, r, w = make(n, h, 5)
    d = dev()
    xd, rd, wd = x.to(d), r.to(d), w.to(d)
    digests = set()
    configs = [None, dr.LaunchConfig(variant=dr.VARIANT_STAGED), dr.LaunchConfig(variant=dr.VARIANT_ROWS,
                                                                               threads_per_row=512)]
    for C in (2, 4):
        for T in (32, 64, 128, 256, 512):
            K = 8192 // 8 // C // T
            if K not in (1, 2, 4, 8) or T > (1024 if K <= 2 else 512):
                continue
            for S, G in ((1, 0), (2, 2 * C), (3, 6 * C), (2, 0)):
                configs.append(dr.LaunchConfig(variant=dr.VARIANT_SPLIT, cluster_ctas=C, threads_per_row=T,
                                               stages=S, grid_ctas=G))
    configs.append(dr.LaunchConfig(variant=dr.VARIANT_SPLIT, serialize=1))
    for cfg in configs:
        out, ro = dr.add_rmsnorm_fwd(xd, rd, wd, 1e-6, config=cfg)
        torch.cuda.synchronize()
        digests.add(refs.u16(out).tobytes() + refs.u16(ro).tobytes())
    assert len(digests) == 1
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6, threads=THREADS)
    assert digests.pop() == eo.tobytes() + ero.tobytes()


def test_in_place(orc):
    x, r, w = make(128, 4096, 7)
    d = dev()
    xd, rd = x.to(d), r.to(d)
    cfg = dr.LaunchConfig(variant=dr.VARIANT_SPLIT, cluster_ctas=4)
    dr.add_rmsnorm_fwd(xd, rd, w.to(d), 1e-6, out=xd, residual_out=rd, config=cfg)
    torch.cuda.synchronize()
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6, threads=THREADS)
    assert_bits_equal(refs.u16(xd), eo, "out in place")
    assert_bits_equal(refs.u16(rd), ero, "residual_out in place")


@pytest.mark.parametrize("C", [2, 4])
def test_bounded_wait_expires_and_recovers(orc, C):
    """fault_inject withholds every CTA's first copy: the waits run out, the
    clusters learn of it at their barrier and leave together after draining
    their copies; DRADD_ERR_TIMEOUT is reported and the context stays
    usable."""
    assert dr.device_status(clear=True) == 0
    x, r, w = make(64, 4096, 9)
    d = dev()
    xd, rd, wd = x.to(d), r.to(d), w.to(d)
    cfg = dr.LaunchConfig(variant=dr.VARIANT_SPLIT, cluster_ctas=C, stages=3, grid_ctas=4 * C, fault_inject=1,
                          wait_limit_us=20000)
    dr.add_rmsnorm_fwd(xd, rd, wd, 1e-6, config=cfg)
    assert dr.device_status(clear=True) == 8
    assert dr.device_status(clear=True) == 0
    out, ro = dr.add_rmsnorm_fwd(xd, rd, wd, 1e-6, config=dr.LaunchConfig(variant=dr.VARIANT_SPLIT, cluster_ctas=C))
    torch.cuda.synchronize()
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6, threads=THREADS)
    assert_bits_equal(refs.u16(out), eo, "after timeout")
    assert dr.device_status(clear=True) == 0
