"""fp4 e2m1 output on the GPU: the conversion the kernels use over all 2^32
fp32 inputs against the oracle's encoder, and both forms bit for bit against
the oracle (packed codes, scales, residual_out) across shapes and launch
configurations."""
import hashlib

import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import THREADS, assert_bits_equal, dev, to_dev

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


def test_e2m1_conversion_exhaustive(orc):
    from concurrent.futures import ThreadPoolExecutor
    buf = torch.empty(CHUNK, dtype=torch.int16, device=dev())
    host = torch.empty(CHUNK, dtype=torch.int16, pin_memory=True)
    ex = ThreadPoolExecutor(THREADS)
    part = CHUNK // 16
    for first in range(0, 1 << 32, CHUNK):
        dr.bf16_convert_range(buf, first, CHUNK, 4)
        host.copy_(buf)
        f = (np.arange(CHUNK, dtype=np.uint32) + np.uint32(first)).view(np.float32)
        exp = np.concatenate(list(ex.map(orc.e2m1_convert, [f[i:i + part] for i in range(0, CHUNK, part)])))
        got = (host.numpy().view(np.uint16) & 0xF).astype(np.uint8)
        nan = np.isnan(f)
        bad = np.nonzero((got != exp) & ~nan)[0]
        assert bad.size == 0, (hex(int(f[bad[0]:bad[0] + 1].view(np.uint32)[0])), got[bad[0]], exp[bad[0]])
    ex.shutdown()


def case(n, h, seed):
    g = inputs.generator(seed)
    return (inputs.normal_bf16(g, (n, h), 0.0, 1.0), inputs.normal_bf16(g, (n, h), 0.0, 4.0),
            inputs.normal_bf16(g, (h,), 1.0, 0.1))


@pytest.mark.parametrize("n,h", [(4096, 4096), (2048, 16384), (65, 24), (33, 1000), (3, 32768), (1, 8)])
def test_fp4_bit_exact(orc, n, h):
    x, r, w = case(n, h, 13 * n + h)
    q, s, ro = dr.add_rmsnorm_fp4_fwd(to_dev(x), to_dev(r), to_dev(w), 1e-6)
    qp, sp = dr.rmsnorm_fp4_fwd(to_dev(x), to_dev(w), 1e-6)
    torch.cuda.synchronize()
    eq, es, ero = orc.rmsnorm_fp4_fwd(x, w, 1e-6, residual=r, threads=THREADS)
    assert_bits_equal(q.cpu().numpy(), eq, "add fp4 codes")
    assert_bits_equal(s.cpu().numpy().view(np.uint32), es.view(np.uint32), "add fp4 scale")
    assert_bits_equal(refs.u16(ro), ero, "add fp4 residual_out")
    eqp, esp = orc.rmsnorm_fp4_fwd(x, w, 1e-6, threads=THREADS)
    assert_bits_equal(qp.cpu().numpy(), eqp, "plain fp4 codes")
    assert_bits_equal(sp.cpu().numpy().view(np.uint32), esp.view(np.uint32), "plain fp4 scale")


def test_fp4_one_result_group(orc):
    x, r, w = case(512, 8192, 9)
    dx, drs, dw = to_dev(x), to_dev(r), to_dev(w)
    cfgs = [None, dr.LaunchConfig(variant=1, threads_per_row=512),
            dr.LaunchConfig(variant=2, threads_per_row=1024, stages=2),
            dr.LaunchConfig(variant=2, threads_per_row=128, stages=3, grid_ctas=17)]
    digests = set()
    for cfg in cfgs:
        q, s, ro = dr.add_rmsnorm_fp4_fwd(dx, drs, dw, 1e-6, config=cfg)
        torch.cuda.synchronize()
        digests.add(hashlib.sha256(q.cpu().numpy().tobytes() + s.cpu().numpy().tobytes()).hexdigest())
    assert len(digests) == 1
