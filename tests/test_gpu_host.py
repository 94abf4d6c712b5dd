"""The host-buffer driver (chunked copies overlapped with the kernels)
returns the oracle's bits, for both variants and a ragged chunking."""
import numpy as np
import pytest
import torch

import refs
from deterministic_residual_add_gb300 import inputs
from deterministic_residual_add_gb300.host import HostPipeline
from gpu_util import THREADS, assert_bits_equal, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("quant,chunk", [(False, 512), (False, 300), (True, 512), (True, 77)])
def test_host_pipeline_matches_oracle(orc, quant, chunk):
    c = inputs.WORKLOADS["2048x4096"].make(n_rows=1000)
    x_h, r_h, w_h = c["x"].pin_memory(), c["residual"].pin_memory(), c["weight"].pin_memory()
    n, h = x_h.shape
    pipe = HostPipeline(n, h, dev(), chunk_rows=chunk, quant=quant)
    ro_h = torch.empty_like(x_h).pin_memory()
    if quant:
        outs = (torch.empty(n, h, dtype=torch.int8).pin_memory(),
                torch.empty(n, dtype=torch.float32).pin_memory(), ro_h)
    else:
        outs = (torch.empty_like(x_h).pin_memory(), ro_h)
    for _ in range(2):  # the second call reuses the staging buffers
        pipe(x_h, r_h, w_h, c["eps"], outs)
        torch.cuda.synchronize()
    if quant:
        eq, es, ero = orc.add_rmsnorm_quant_fwd(c["x"], c["residual"], c["weight"], c["eps"], threads=THREADS)
        assert_bits_equal(outs[0].numpy().view(np.uint8), eq.view(np.uint8), "q")
        assert_bits_equal(outs[1].numpy().view(np.uint32), es.view(np.uint32), "scale")
    else:
        eo, ero = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"], threads=THREADS)
        assert_bits_equal(refs.u16(outs[0]), eo, "out")
    assert_bits_equal(refs.u16(ro_h), ero, "residual_out")


@pytest.mark.parametrize("quant,n", [(False, 1000), (True, 1000), (False, 4096), (False, 3)])
def test_zero_copy_matches_oracle(orc, quant, n):
    """The kernel reads and writes pinned host memory directly (the library
    sees host pointers and takes its register-load variant): the oracle's
    bits, twice in a row."""
    from deterministic_residual_add_gb300.host import add_rmsnorm_fwd_host
    c = inputs.WORKLOADS["2048x4096"].make(n_rows=min(n, 2048)) if n <= 2048 else None
    if c is None:
        ch = inputs.CHAIN4096
        r0, w = ch.initial()
        c = {"x": ch.delta(0), "residual": r0, "weight": w, "eps": 1e-6}
    x_h, r_h, w_h = c["x"].pin_memory(), c["residual"].pin_memory(), c["weight"].pin_memory()
    n, h = x_h.shape
    ro_h = torch.empty_like(x_h).pin_memory()
    if quant:
        outs = (torch.empty(n, h, dtype=torch.int8).pin_memory(),
                torch.empty(n, dtype=torch.float32).pin_memory(), ro_h)
    else:
        outs = (torch.empty_like(x_h).pin_memory(), ro_h)
    torch.cuda.set_device(dev())
    s = torch.cuda.Stream()
    for _ in range(2):
        add_rmsnorm_fwd_host(x_h, r_h, w_h, c["eps"], outs, stream=s, quant=quant)
        s.synchronize()
    if quant:
        eq, es, ero = orc.add_rmsnorm_quant_fwd(c["x"], c["residual"], c["weight"], c["eps"], threads=THREADS)
        assert_bits_equal(outs[0].numpy().view(np.uint8), eq.view(np.uint8), "q")
        assert_bits_equal(outs[1].numpy().view(np.uint32), es.view(np.uint32), "scale")
    else:
        eo, ero = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"], threads=THREADS)
        assert_bits_equal(refs.u16(outs[0]), eo, "out")
    assert_bits_equal(refs.u16(ro_h), ero, "residual_out")


def test_host_memory_rejects_explicit_staged():
    """An explicit staged configuration with a host buffer is refused before
    anything is launched; the automatic choice serves it."""
    import ctypes
    import deterministic_residual_add_gb300 as dr
    c = inputs.WORKLOADS["2048x4096"].make(n_rows=64)
    x_h, r_h, w_h = c["x"].pin_memory(), c["residual"].pin_memory(), c["weight"].pin_memory()
    out_d = torch.empty(x_h.shape, dtype=torch.bfloat16, device=dev())
    ro_d = torch.empty_like(out_d)
    cfg = dr.LaunchConfig(variant=2)._c()
    st = dr.lib().add_rmsnorm_fwd_with_config(out_d.data_ptr(), ro_d.data_ptr(), x_h.data_ptr(), r_h.data_ptr(),
                                              w_h.data_ptr(), ctypes.c_float(1e-6), 64, 4096, None, ctypes.byref(cfg))
    assert st == 9
    st = dr.lib().add_rmsnorm_fwd(out_d.data_ptr(), ro_d.data_ptr(), x_h.data_ptr(), r_h.data_ptr(),
                                  w_h.data_ptr(), ctypes.c_float(1e-6), 64, 4096, None)
    torch.cuda.synchronize()
    assert st == 0
    ref_out, ref_ro = dr.add_rmsnorm_fwd(x_h.to(dev()), r_h.to(dev()), w_h.to(dev()), 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(out_d.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(ro_d.view(torch.int16), ref_ro.view(torch.int16))
    assert dr.device_status() == 0
