"""Past 2^31 elements: 524,289 rows of 4,104 (2.15e9 elements, 4.3 GB per
bf16 tensor) through the default launch of the bf16 and int8 forms, checked
on sampled rows (first, last, around the 2^31-element boundary, random)
against the oracle.  The inputs are a fixed hash of (row, column) made on
the device; the sampled rows are rebuilt the same way for the oracle."""
import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import assert_bits_equal, dev

pytestmark = pytest.mark.gpu

N_ROWS, HIDDEN = 524289, 4104
EPS = 1e-6


def _sample_rows():
    boundary = (2 ** 31) // HIDDEN
    rnd = np.random.default_rng(0).integers(0, N_ROWS, 24).tolist()
    return sorted({0, 1, boundary - 1, boundary, boundary + 1, N_ROWS - 2, N_ROWS - 1, *rnd})


def test_more_than_2_31_elements(orc):
    assert N_ROWS * HIDDEN > 2 ** 31
    d = dev()
    free, _ = torch.cuda.mem_get_info(d)
    if free < 32 * 2 ** 30:
        pytest.skip("needs 32 GB of free device memory")
    x = torch.empty(N_ROWS, HIDDEN, dtype=torch.int16, device=d)
    r = torch.empty_like(x)
    step = 16384
    for lo in range(0, N_ROWS, step):
        rows = torch.arange(lo, min(N_ROWS, lo + step), device=d)
        x[lo:lo + len(rows)] = inputs.hashed_bf16_rows(rows, HIDDEN, 1)
        r[lo:lo + len(rows)] = inputs.hashed_bf16_rows(rows, HIDDEN, 2)
    w = inputs.normal_bf16(inputs.generator(5), (HIDDEN,), 1.0, 0.1)
    xb, rb, wd = x.view(torch.bfloat16), r.view(torch.bfloat16), w.to(d)

    idx = torch.tensor(_sample_rows(), device=d)
    xs = inputs.hashed_bf16_rows(idx, HIDDEN, 1).cpu().view(torch.bfloat16)
    rs = inputs.hashed_bf16_rows(idx, HIDDEN, 2).cpu().view(torch.bfloat16)

    out, ro = dr.add_rmsnorm_fwd(xb, rb, wd, EPS)
    torch.cuda.synchronize()
    eo, ero = orc.add_rmsnorm_fwd(xs, rs, w, EPS)
    assert_bits_equal(refs.u16(ro[idx]), ero, "sampled residual_out")
    assert_bits_equal(refs.u16(out[idx]), eo, "sampled out")
    del out
    q, scale, ro2 = dr.add_rmsnorm_quant_fwd(xb, rb, wd, EPS, residual_out=ro)
    torch.cuda.synchronize()
    eq, escale, ero2 = orc.add_rmsnorm_quant_fwd(xs, rs, w, EPS)
    assert_bits_equal(refs.u16(ro2[idx]), ero2, "quant: sampled residual_out")
    assert_bits_equal(q[idx].cpu().numpy(), eq, "quant: sampled codes")
    assert np.array_equal(scale[idx].cpu().numpy().view(np.uint32), escale.view(np.uint32))
    assert dr.device_status() == 0
    del x, r, ro, q, scale, ro2
    torch.cuda.empty_cache()
