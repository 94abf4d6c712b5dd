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
