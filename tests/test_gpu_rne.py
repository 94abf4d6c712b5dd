"""The device conversions fp32 -> bf16 over all 2^32 fp32 patterns against
the oracle's round-to-nearest-even: the one the kernels use, the integer
round-half-even, the hardware cvt.rn.bf16x2.f32 instruction and CUDA's own
__float2bfloat16_rn.  Non-NaN patterns must match bit for bit; NaN must give
a NaN."""
import numpy as np
import pytest
import torch

import deterministic_residual_add_gb300 as dr
from gpu_util import THREADS, dev

pytestmark = pytest.mark.gpu

CHUNK = 1 << 27


def test_conversion_exhaustive(orc):
    from concurrent.futures import ThreadPoolExecutor
    M = (0, 1, 2, 5)
    buf = torch.empty(len(M), CHUNK, dtype=torch.int16, device=dev())
    host = torch.empty(len(M), CHUNK, dtype=torch.int16, pin_memory=True)
    ex = ThreadPoolExecutor(THREADS)
    for first in range(0, 1 << 32, CHUNK):
        for i, m in enumerate(M):
            dr.bf16_convert_range(buf[i], first, CHUNK, m)
        host.copy_(buf)
        parts = [ex.submit(orc.bf16_convert_range, first + i, CHUNK // THREADS)
                 for i in range(0, CHUNK, CHUNK // THREADS)]
        exp = np.concatenate([p.result() for p in parts])
        pats = (np.arange(CHUNK, dtype=np.uint64) + first).astype(np.uint32)
        nan = (pats & 0x7FFFFFFF) > 0x7F800000
        got = host.numpy().view(np.uint16)
        for i, m in enumerate(M):
            g = got[i]
            bad = np.nonzero((g != exp) & ~nan)[0]
            assert bad.size == 0, (m, hex(int(pats[bad[0]])), hex(int(g[bad[0]])), hex(int(exp[bad[0]])))
            gn = g[nan]
            assert np.all(((gn & 0x7F80) == 0x7F80) & ((gn & 0x7F) != 0)), m
    ex.shutdown()
