"""The C ABI on a live device: aliasing as documented, nothing written
outside the outputs (guard bands), streams, the empty call, argument errors
with real tensors, and the bounded wait of the staged kernel running out
(without faulting the GPU: the test withholds a copy, the wait expires, the
kernel records the timeout and returns, and the next call works)."""
import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import THREADS, assert_bits_equal, dev, to_dev

pytestmark = pytest.mark.gpu


def small_case(n=64, h=1024, seed=5):
    g = inputs.generator(seed)
    return (inputs.normal_bf16(g, (n, h), 0.0, 1.0), inputs.normal_bf16(g, (n, h), 0.0, 4.0),
            inputs.normal_bf16(g, (h,), 1.0, 0.1))


@pytest.mark.parametrize("variant", [dr.VARIANT_ROWS, dr.VARIANT_STAGED])
def test_in_place_aliases(orc, variant):
    x, r, w = small_case()
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6)
    cfg = dr.LaunchConfig(variant=variant)
    dx, drs, dw = to_dev(x), to_dev(r), to_dev(w)
    # residual_out == residual and out == x
    dr.add_rmsnorm_fwd(dx, drs, dw, 1e-6, out=dx, residual_out=drs, config=cfg)
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(drs), ero, "in-place residual_out")
    assert_bits_equal(refs.u16(dx), eo, "in-place out")
    # residual_out == x and out == residual
    dx, drs = to_dev(x), to_dev(r)
    dr.add_rmsnorm_fwd(dx, drs, dw, 1e-6, out=drs, residual_out=dx, config=cfg)
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(dx), ero, "swapped residual_out")
    assert_bits_equal(refs.u16(drs), eo, "swapped out")


@pytest.mark.parametrize("variant", [dr.VARIANT_ROWS, dr.VARIANT_STAGED])
def test_guard_bands_untouched(orc, variant):
    """Outputs live inside larger buffers filled with a canary; only the
    output range may change (odd row counts exercise the tail)."""
    for n in (1, 3, 65):
        x, r, w = small_case(n=n, h=1024, seed=n)
        pad = 4096
        numel = n * 1024
        canary = 0x5A5A
        big_out = torch.full((pad + numel + pad,), canary, dtype=torch.int16, device=dev())
        big_ro = torch.full_like(big_out, canary)
        big_q = torch.full((pad + numel + pad,), 0x5A, dtype=torch.int8, device=dev())
        big_s = torch.full((256 + n + 256,), 7.0, dtype=torch.float32, device=dev())
        out = big_out[pad:pad + numel].view(torch.bfloat16).view(n, 1024)
        ro = big_ro[pad:pad + numel].view(torch.bfloat16).view(n, 1024)
        cfg = dr.LaunchConfig(variant=variant)
        dr.add_rmsnorm_fwd(to_dev(x), to_dev(r), to_dev(w), 1e-6, out=out, residual_out=ro, config=cfg)
        q = big_q[pad:pad + numel].view(n, 1024)
        s = big_s[256:256 + n]
        dr.add_rmsnorm_quant_fwd(to_dev(x), to_dev(r), to_dev(w), 1e-6, out_q=q, scale=s,
                                 residual_out=ro, config=cfg)
        torch.cuda.synchronize()
        for big, fill in ((big_out, canary), (big_ro, canary)):
            h = big.cpu().numpy()
            assert np.all(h[:pad] == fill) and np.all(h[pad + numel:] == fill)
        hq = big_q.cpu().numpy()
        assert np.all(hq[:pad] == 0x5A) and np.all(hq[pad + numel:] == 0x5A)
        hs = big_s.cpu().numpy()
        assert np.all(hs[:256] == 7.0) and np.all(hs[256 + n:] == 7.0)
        eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6)
        assert_bits_equal(refs.u16(out), eo, "out")


def test_side_stream_and_empty_call(orc):
    x, r, w = small_case()
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dx, drs, dw = to_dev(x), to_dev(r), to_dev(w)
        out, ro = dr.add_rmsnorm_fwd(dx, drs, dw, 1e-6, stream=s)
    s.synchronize()
    assert_bits_equal(refs.u16(out), eo, "side stream out")
    empty = torch.empty(0, 1024, dtype=torch.bfloat16, device=dev())
    o2, r2 = dr.add_rmsnorm_fwd(empty, empty.clone(), dw, 1e-6)
    assert o2.numel() == 0 and r2.numel() == 0


def test_argument_errors_with_real_tensors():
    x = torch.zeros(4, 1024, dtype=torch.bfloat16, device=dev())
    w = torch.ones(1024, dtype=torch.bfloat16, device=dev())
    raw = torch.zeros(4 * 1024 + 8, dtype=torch.bfloat16, device=dev())
    shifted = raw[1:1 + 4 * 1024].view(4, 1024)  # 2 bytes off alignment
    with pytest.raises(dr.DraddError) as e:
        dr.add_rmsnorm_fwd(shifted, x, w, 1e-6)
    assert e.value.status == 4
    with pytest.raises(dr.DraddError) as e:
        dr.add_rmsnorm_fwd(x, x.clone(), w, 1e-6, out=raw[8:8 + 4096].view(4, 1024),
                           residual_out=raw[:4096].view(4, 1024))
    assert e.value.status == 6
    with pytest.raises(dr.DraddError) as e:
        dr.add_rmsnorm_fwd(x, x.clone(), w, float("nan"))
    assert e.value.status == 5


def test_bounded_wait_expires_and_recovers(orc):
    """fault_inject withholds each CTA's first staged copy: every CTA's wait
    runs out after wait_limit_us, the kernel records DRADD_ERR_TIMEOUT,
    drains its other copies and returns; the context stays usable."""
    assert dr.device_status(clear=True) == 0
    x, r, w = small_case(n=64, h=4096)
    dx, drs, dw = to_dev(x), to_dev(r), to_dev(w)
    cfg = dr.LaunchConfig(variant=dr.VARIANT_STAGED, stages=3, grid_ctas=8, fault_inject=1,
                          wait_limit_us=20000)
    dr.add_rmsnorm_fwd(dx, drs, dw, 1e-6, config=cfg)
    assert dr.device_status(clear=True) == 8
    assert dr.device_status(clear=True) == 0
    out, ro = dr.add_rmsnorm_fwd(dx, drs, dw, 1e-6, config=dr.LaunchConfig(variant=dr.VARIANT_STAGED))
    torch.cuda.synchronize()
    eo, ero = orc.add_rmsnorm_fwd(x, r, w, 1e-6)
    assert_bits_equal(refs.u16(out), eo, "after timeout")
    assert dr.device_status(clear=True) == 0
    # the one-argument form reads and resets in one call
    dr.add_rmsnorm_fwd(dx, drs, dw, 1e-6, config=cfg)
    assert dr.last_device_status() == 8
    assert dr.last_device_status() == 0
