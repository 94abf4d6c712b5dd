"""The staged pair kernel (plain RMSNorm with int8, e4m3 or e2m1 out, two
rows per thread: LaunchConfig(variant=STAGED, rows_per_cta=2)) on the GPU,
bit for bit against the oracle: full-size and ragged shapes with odd and
even row counts, its launch shapes (threads, stages, grid), rows with
special values (NaN, an overflowing sum, a zero row with eps = 0, -inf),
non-finite weights, the configurations it refuses and the bounded wait."""
import hashlib

import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import THREADS, assert_bits_equal, to_dev

pytestmark = pytest.mark.gpu


def pair(**kw):
    return dr.LaunchConfig(variant=dr.VARIANT_STAGED, rows_per_cta=2, **kw)


def case(n, h, seed):
    g = inputs.generator(seed)
    return inputs.normal_bf16(g, (n, h), 0.0, 1.0), inputs.normal_bf16(g, (h,), 1.0, 0.1)


def u8(t):
    return t.cpu().numpy().view(np.uint8)


def u32(t):
    return t.cpu().numpy().view(np.uint32)


def run_quant(orc, x, w, eps, config, e2m1_rows=slice(None)):
    """int8, e4m3 and e2m1 plain forms on the GPU and in the oracle; e4m3
    NaN codes compare by NaN-ness, e2m1 codes on e2m1_rows only (the format
    has no NaN)."""
    dx, dw = to_dev(x), to_dev(w)
    q, s = dr.rmsnorm_quant_fwd(dx, dw, eps, config=config)
    q8, s8 = dr.rmsnorm_fp8_fwd(dx, dw, eps, config=config)
    q4, s4 = dr.rmsnorm_fp4_fwd(dx, dw, eps, config=config)
    torch.cuda.synchronize()
    eq, es = orc.rmsnorm_quant_fwd(x, w, eps, threads=THREADS)
    eq8, es8 = orc.rmsnorm_fp8_fwd(x, w, eps, threads=THREADS)
    eq4, es4 = orc.rmsnorm_fp4_fwd(x, w, eps, threads=THREADS)
    assert_bits_equal(u8(q), eq.view(np.uint8), "int8 codes")
    assert_bits_equal(u32(s), es.view(np.uint32), "int8 scales")
    assert_bits_equal(u32(s8), es8.view(np.uint32), "e4m3 scales")
    g8, e8 = u8(q8), eq8.view(np.uint8)
    nan8 = (e8 & 0x7F) == 0x7F
    assert np.array_equal((g8 & 0x7F) == 0x7F, nan8)
    assert_bits_equal(g8[~nan8], e8[~nan8], "e4m3 codes")
    assert_bits_equal(u32(s4), es4.view(np.uint32), "e2m1 scales")
    assert_bits_equal(u8(q4)[e2m1_rows], eq4.view(np.uint8)[e2m1_rows], "e2m1 codes")


@pytest.mark.parametrize("n,h", [(4096, 4096), (4095, 4096), (513, 2048), (37, 1000), (9, 4000), (1, 4096),
                                 (2, 256), (130, 3000), (77, 8192)])
def test_plain_quantised_forms_bit_exact(orc, n, h):
    x, w = case(n, h, n * 29 + h)
    run_quant(orc, x, w, 1e-6, pair())


def test_launch_shapes_one_result(orc):
    x, w = case(333, 4096, 5)
    dx, dw = to_dev(x), to_dev(w)
    cfgs = [pair(threads_per_row=T, stages=S, grid_ctas=G)
            for T in (128, 256, 512) for S in (1, 3) for G in (0, 1, 7)]
    cfgs += [pair(serialize=1), None]
    digests = set()
    for cfg in cfgs:
        q, s = dr.rmsnorm_quant_fwd(dx, dw, 1e-6, config=cfg)
        q8, s8 = dr.rmsnorm_fp8_fwd(dx, dw, 1e-6, config=cfg)
        torch.cuda.synchronize()
        digests.add(hashlib.sha256(u8(q).tobytes() + u32(s).tobytes() + u8(q8).tobytes()
                                   + u32(s8).tobytes()).hexdigest())
    assert len(digests) == 1
    eq, es = orc.rmsnorm_quant_fwd(x, w, 1e-6, threads=THREADS)
    eq8, es8 = orc.rmsnorm_fp8_fwd(x, w, 1e-6, threads=THREADS)
    assert digests == {hashlib.sha256(eq.view(np.uint8).tobytes() + es.view(np.uint32).tobytes()
                                      + eq8.view(np.uint8).tobytes() + es8.view(np.uint32).tobytes()).hexdigest()}


# rows of special_rows without a special value (their y is finite)
ORDINARY = [0, 5, 6, 7, 8]


def special_rows(h, seed):
    """Nine rows (so the last pair holds one row): a NaN in x, a sum of
    squares that overflows, an all-zero row (with eps = 0: 1 / sqrt(0) is
    infinite), a -inf in x, plus the ORDINARY rows; bf16 bit patterns."""
    x, w = case(9, h, seed)
    xb = refs.u16(x).copy()
    xb[1, 5] = 0x7FC0           # NaN
    xb[2, :] = 0x7F00           # 2^127: squares overflow
    xb[3, :] = 0x0000           # zero row
    xb[4, 7] = 0xFF80           # -inf
    return torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16), w


@pytest.mark.parametrize("h", [1024, 4096])
def test_special_rows_match_the_oracle(orc, h):
    x, w = special_rows(h, h + 11)
    run_quant(orc, x, w, 0.0, pair(), e2m1_rows=ORDINARY)
    run_quant(orc, x, w, 1e-6, pair(), e2m1_rows=ORDINARY)
    # the rows in the other position of each pair
    xs = torch.cat([x[:1], x])
    run_quant(orc, xs, w, 1e-6, pair(), e2m1_rows=[r + 1 for r in ORDINARY] + [0])


def test_non_finite_weights_match_the_oracle(orc):
    x, w = case(7, 1024, 9)
    wb = refs.u16(w).copy()
    wb[3] = 0x7F80              # +inf weight
    wb[10] = 0x7FC0             # NaN weight
    tw = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16)
    run_quant(orc, x, tw, 1e-6, pair(), e2m1_rows=slice(0, 0))


def test_configurations_it_refuses():
    x, w = case(8, 4096, 3)
    dx, dw = to_dev(x), to_dev(w)
    r = to_dev(case(8, 4096, 4)[0])
    for call in (lambda: dr.rmsnorm_fwd(dx, dw, 1e-6, config=pair()),              # bf16 out
                 lambda: dr.add_rmsnorm_quant_fwd(dx, r, dw, 1e-6, config=pair()),  # residual form
                 lambda: dr.rmsnorm_quant_fwd(to_dev(case(8, 16384, 5)[0]), to_dev(case(8, 16384, 5)[1]), 1e-6,
                                              config=pair(threads_per_row=256))):  # K = 8
        with pytest.raises(dr.DraddError) as e:
            call()
        assert e.value.status == 9


def test_bounded_wait_expires_and_recovers(orc):
    """fault_inject withholds each CTA's first copy: its wait runs out after
    wait_limit_us, the kernel records DRADD_ERR_TIMEOUT, drains its other
    copies and returns; the context stays usable."""
    assert dr.device_status(clear=True) == 0
    x, w = case(64, 2048, 6)
    dx, dw = to_dev(x), to_dev(w)
    cfg = pair(stages=3, grid_ctas=4, fault_inject=1, wait_limit_us=20000)
    dr.rmsnorm_quant_fwd(dx, dw, 1e-6, config=cfg)
    assert dr.device_status(clear=True) == 8
    q, s = dr.rmsnorm_quant_fwd(dx, dw, 1e-6, config=pair())
    torch.cuda.synchronize()
    eq, es = orc.rmsnorm_quant_fwd(x, w, 1e-6)
    assert_bits_equal(u8(q), eq.view(np.uint8), "after timeout")
    assert dr.device_status(clear=True) == 0


@pytest.mark.parametrize("n,h", [(4096, 512), (16384, 512), (9001, 400), (301, 480)])
def test_plain_quantised_at_512_in_the_automatic_plan(orc, n, h):
    """P = 512 in the automatic plan: the pair kernel with K = 1 below 8192
    rows, one row a CTA with K = 2 beyond; bit for bit either way."""
    x, w = case(n, h, n + h)
    run_quant(orc, x, w, 1e-6, None)
