"""fp8 e4m3 output on the GPU: the conversion the kernels use over all 2^32
fp32 inputs against the oracle's encoder, and the residual-add and plain
forms bit for bit against the oracle (codes, scales, residual_out) across
shapes and launch configurations."""
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


def test_e4m3_conversion_exhaustive(orc):
    from concurrent.futures import ThreadPoolExecutor
    buf = torch.empty(CHUNK, dtype=torch.int16, device=dev())
    host = torch.empty(CHUNK, dtype=torch.int16, pin_memory=True)
    ex = ThreadPoolExecutor(THREADS)
    part = CHUNK // 16
    for first in range(0, 1 << 32, CHUNK):
        dr.bf16_convert_range(buf, first, CHUNK, 3)
        host.copy_(buf)
        pats = np.arange(CHUNK, dtype=np.uint32) + np.uint32(first)
        f = pats.view(np.float32)
        exp = np.concatenate(list(ex.map(orc.e4m3_convert, [f[i:i + part] for i in range(0, CHUNK, part)])))
        got = (host.numpy().view(np.uint16) & 0xFF).astype(np.uint8)
        nan = np.isnan(f)
        bad = np.nonzero((got != exp) & ~nan)[0]
        assert bad.size == 0, (hex(int(pats[bad[0]])), hex(int(got[bad[0]])), hex(int(exp[bad[0]])))
        assert np.all((got[nan] & 0x7F) == 0x7F)
    ex.shutdown()


def case(n, h, seed, r_std=4.0):
    g = inputs.generator(seed)
    return (inputs.normal_bf16(g, (n, h), 0.0, 1.0), inputs.normal_bf16(g, (n, h), 0.0, r_std),
            inputs.normal_bf16(g, (h,), 1.0, 0.1))


@pytest.mark.parametrize("n,h", [(4096, 4096), (2048, 16384), (65, 24), (33, 1000), (3, 32768), (1, 8),
                                 (7, 8200)])
def test_fp8_bit_exact(orc, n, h):
    x, r, w = case(n, h, 11 * n + h)
    q, s, ro = dr.add_rmsnorm_fp8_fwd(to_dev(x), to_dev(r), to_dev(w), 1e-6)
    qp, sp = dr.rmsnorm_fp8_fwd(to_dev(x), to_dev(w), 1e-6)
    torch.cuda.synchronize()
    eq, es, ero = orc.rmsnorm_fp8_fwd(x, w, 1e-6, residual=r, threads=THREADS)
    assert_bits_equal(q.cpu().numpy(), eq, "add fp8 codes")
    assert_bits_equal(s.cpu().numpy().view(np.uint32), es.view(np.uint32), "add fp8 scale")
    assert_bits_equal(refs.u16(ro), ero, "add fp8 residual_out")
    eqp, esp = orc.rmsnorm_fp8_fwd(x, w, 1e-6, threads=THREADS)
    assert_bits_equal(qp.cpu().numpy(), eqp, "plain fp8 codes")
    assert_bits_equal(sp.cpu().numpy().view(np.uint32), esp.view(np.uint32), "plain fp8 scale")


def test_fp8_special_rows(orc):
    """Zero rows, cancelling rows (-0 codes), subnormal and constant rows."""
    h = 2048
    g = inputs.generator(77)
    x = refs.u16(inputs.normal_bf16(g, (6, h), 0.0, 1.0)).copy()
    r = refs.u16(inputs.normal_bf16(g, (6, h), 0.0, 1.0)).copy()
    x[0] = 0; r[0] = 0
    r[1] = x[1] ^ 0x8000
    x[2] = (x[2] & 0x807F); r[2] = (r[2] & 0x807F)
    x[3] = 0xC040; r[3] = 0
    w = refs.u16(inputs.normal_bf16(g, (h,), 0.0, 1.0))
    tx, tr, tw = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) for a in (x, r, w))
    q, s, ro = dr.add_rmsnorm_fp8_fwd(to_dev(tx), to_dev(tr), to_dev(tw), 1e-6)
    torch.cuda.synchronize()
    eq, es, ero = orc.rmsnorm_fp8_fwd(x, w, 1e-6, residual=r)
    assert_bits_equal(q.cpu().numpy(), eq, "codes")
    assert_bits_equal(s.cpu().numpy().view(np.uint32), es.view(np.uint32), "scales")


def test_fp8_one_result_group(orc):
    x, r, w = case(1024, 8192, 3)
    dx, drs, dw = to_dev(x), to_dev(r), to_dev(w)
    cfgs = [None, dr.LaunchConfig(variant=1, threads_per_row=512),
            dr.LaunchConfig(variant=1, threads_per_row=128, rows_per_cta=4),
            dr.LaunchConfig(variant=2, threads_per_row=1024, stages=2),
            dr.LaunchConfig(variant=2, threads_per_row=256, stages=3, grid_ctas=13),
            dr.LaunchConfig(variant=2, threads_per_row=128, stages=1, serialize=1)]
    digests = set()
    for cfg in cfgs:
        q, s, ro = dr.add_rmsnorm_fp8_fwd(dx, drs, dw, 1e-6, config=cfg)
        torch.cuda.synchronize()
        digests.add(hashlib.sha256(q.cpu().numpy().tobytes() + s.cpu().numpy().tobytes()).hexdigest())
    assert len(digests) == 1
    eq, es, _ = orc.rmsnorm_fp8_fwd(x, w, 1e-6, residual=r, threads=THREADS)
    assert digests == {hashlib.sha256(eq.tobytes() + es.tobytes()).hexdigest()}
