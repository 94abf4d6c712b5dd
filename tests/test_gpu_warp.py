"""The warp-per-row variant on the GPU, bit for bit against the oracle: every
entry point of the main op (residual-add and plain RMSNorm; bf16, int8,
e4m3 and e2m1 out) at full-size and ragged shapes, its launch shapes (warps
per CTA, grid), and rows with special values (NaN, an overflowing sum, a
zero row with eps = 0, non-finite weights), which take the exact int8
path; the register and staged variants are held to the same rows."""
import hashlib

import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import THREADS, assert_bits_equal, to_dev

pytestmark = pytest.mark.gpu

WARP = dr.LaunchConfig(variant=dr.VARIANT_WARP)


def case(n, h, seed):
    g = inputs.generator(seed)
    return (inputs.normal_bf16(g, (n, h), 0.0, 1.0), inputs.normal_bf16(g, (n, h), 0.0, 4.0),
            inputs.normal_bf16(g, (h,), 1.0, 0.1))


def u8(t):
    return t.cpu().numpy().view(np.uint8)


def u32(t):
    return t.cpu().numpy().view(np.uint32)


def run_all(orc, x, r, w, eps, config, add, e2m1_rows=slice(None)):
    """Every output kind of one form (add or plain) on the GPU and in the
    oracle; asserts bit equality (e4m3 NaN codes by NaN-ness; e2m1 codes on
    e2m1_rows only: the format has no NaN, and a NaN y's code is not part
    of the contract)."""
    dx, dw = to_dev(x), to_dev(w)
    dr_ = to_dev(r) if add else None
    if add:
        out, ro = dr.add_rmsnorm_fwd(dx, dr_, dw, eps, config=config)
        q, s, ro_q = dr.add_rmsnorm_quant_fwd(dx, dr_, dw, eps, config=config)
        q8, s8, _ = dr.add_rmsnorm_fp8_fwd(dx, dr_, dw, eps, config=config)
        q4, s4, _ = dr.add_rmsnorm_fp4_fwd(dx, dr_, dw, eps, config=config)
        torch.cuda.synchronize()
        eo, ero = orc.add_rmsnorm_fwd(x, r, w, eps, threads=THREADS)
        eq, es, _ = orc.add_rmsnorm_quant_fwd(x, r, w, eps, threads=THREADS)
        eq8, es8, _ = orc.rmsnorm_fp8_fwd(x, w, eps, residual=r, threads=THREADS)
        eq4, es4, _ = orc.rmsnorm_fp4_fwd(x, w, eps, residual=r, threads=THREADS)
        nan_r = np.isnan(refs.bf16_value(ero))  # NaN compares by NaN-ness only
        for got_r, what in ((refs.u16(ro), "residual_out"), (refs.u16(ro_q), "quant residual_out")):
            assert np.array_equal(np.isnan(refs.bf16_value(got_r)), nan_r), what
            assert_bits_equal(got_r[~nan_r], ero[~nan_r], what)
    else:
        out = dr.rmsnorm_fwd(dx, dw, eps, config=config)
        q, s = dr.rmsnorm_quant_fwd(dx, dw, eps, config=config)
        q8, s8 = dr.rmsnorm_fp8_fwd(dx, dw, eps, config=config)
        q4, s4 = dr.rmsnorm_fp4_fwd(dx, dw, eps, config=config)
        torch.cuda.synchronize()
        eo = orc.rmsnorm_fwd(x, w, eps, threads=THREADS)
        eq, es = orc.rmsnorm_quant_fwd(x, w, eps, threads=THREADS)
        eq8, es8 = orc.rmsnorm_fp8_fwd(x, w, eps, threads=THREADS)
        eq4, es4 = orc.rmsnorm_fp4_fwd(x, w, eps, threads=THREADS)
    got_o = refs.u16(out)
    nan_o = np.isnan(refs.bf16_value(eo))
    assert np.array_equal(np.isnan(refs.bf16_value(got_o)), nan_o)
    assert_bits_equal(got_o[~nan_o], eo[~nan_o], "bf16 out")
    assert_bits_equal(u8(q), eq.view(np.uint8), "int8 codes")
    assert_bits_equal(u32(s), es.view(np.uint32), "int8 scales")
    assert_bits_equal(u32(s8), es8.view(np.uint32), "e4m3 scales")
    g8, e8 = u8(q8), eq8.view(np.uint8)
    nan8 = (e8 & 0x7F) == 0x7F
    assert np.array_equal((g8 & 0x7F) == 0x7F, nan8)
    assert_bits_equal(g8[~nan8], e8[~nan8], "e4m3 codes")
    assert_bits_equal(u32(s4), es4.view(np.uint32), "e2m1 scales")
    assert_bits_equal(u8(q4)[e2m1_rows], eq4.view(np.uint8)[e2m1_rows], "e2m1 codes")


@pytest.mark.parametrize("n,h", [(4096, 4096), (512, 2048), (37, 1000), (9, 4000), (5, 200), (3, 256),
                                 (130, 3000)])
def test_plain_forms_bit_exact(orc, n, h):
    x, r, w = case(n, h, n * 31 + h)
    run_all(orc, x, r, w, 1e-6, WARP, add=False)


@pytest.mark.parametrize("n,h", [(2048, 2048), (65, 1024), (37, 1000), (5, 200), (300, 1536)])
def test_residual_forms_bit_exact(orc, n, h):
    x, r, w = case(n, h, n * 37 + h)
    run_all(orc, x, r, w, 1e-6, WARP, add=True)


def test_launch_shapes_one_result_group(orc):
    x, r, w = case(333, 4096, 3)
    dx, dw = to_dev(x), to_dev(w)
    cfgs = [dr.LaunchConfig(variant=dr.VARIANT_WARP, rows_per_cta=R, grid_ctas=G, stages=S)
            for R in (1, 3, 8) for G in (0, 1, 5) for S in (1, 3)] + [None]
    digests = set()
    for cfg in cfgs:
        q, s = dr.rmsnorm_quant_fwd(dx, dw, 1e-6, config=cfg)
        out = dr.rmsnorm_fwd(dx, dw, 1e-6, config=cfg)
        torch.cuda.synchronize()
        digests.add(hashlib.sha256(u8(q).tobytes() + u32(s).tobytes() + refs.u16(out).tobytes()).hexdigest())
    assert len(digests) == 1
    eq, es = orc.rmsnorm_quant_fwd(x, w, 1e-6, threads=THREADS)
    eo = orc.rmsnorm_fwd(x, w, 1e-6, threads=THREADS)
    assert digests == {hashlib.sha256(eq.view(np.uint8).tobytes() + es.view(np.uint32).tobytes()
                                      + eo.tobytes()).hexdigest()}


def test_shapes_the_variant_does_not_take():
    dx = to_dev(case(4, 8192, 1)[0])
    w = to_dev(case(4, 8192, 1)[2])
    with pytest.raises(dr.DraddError) as e:
        dr.rmsnorm_fwd(dx, w, 1e-6, config=WARP)  # P = 8192: 32 blocks a lane
    assert e.value.status == 9
    x, r, w = case(4, 4096, 2)
    with pytest.raises(dr.DraddError) as e:
        dr.add_rmsnorm_fwd(to_dev(x), to_dev(r), to_dev(w), 1e-6, config=WARP)  # residual, K = 16
    assert e.value.status == 9
    for bad in (dr.LaunchConfig(variant=dr.VARIANT_WARP, rows_per_cta=17),
                dr.LaunchConfig(variant=dr.VARIANT_WARP, threads_per_row=64),
                dr.LaunchConfig(variant=dr.VARIANT_WARP, rows_per_cta=16, stages=8)):  # past shared memory
        with pytest.raises(dr.DraddError) as e:
            dr.rmsnorm_fwd(to_dev(x), to_dev(w), 1e-6, config=bad)
        assert e.value.status == 9


def test_bounded_wait_expires_and_recovers(orc):
    """fault_inject withholds each CTA's first group copy: its wait runs out
    after wait_limit_us, the kernel records DRADD_ERR_TIMEOUT, drains its
    other copies and returns; the context stays usable."""
    assert dr.device_status(clear=True) == 0
    x, r, w = case(64, 2048, 4)
    dx, dw = to_dev(x), to_dev(w)
    cfg = dr.LaunchConfig(variant=dr.VARIANT_WARP, rows_per_cta=4, stages=3, grid_ctas=4, fault_inject=1,
                          wait_limit_us=20000)
    dr.rmsnorm_quant_fwd(dx, dw, 1e-6, config=cfg)
    assert dr.device_status(clear=True) == 8
    q, s = dr.rmsnorm_quant_fwd(dx, dw, 1e-6, config=WARP)
    torch.cuda.synchronize()
    eq, es = orc.rmsnorm_quant_fwd(x, w, 1e-6)
    assert_bits_equal(u8(q), eq.view(np.uint8), "after timeout")
    assert dr.device_status(clear=True) == 0


# rows of special_rows without a special value (their y is finite)
ORDINARY = [0, 5, 6, 7]


def special_rows(h, seed):
    """Rows that leave the finite path: a NaN in x, a sum of squares that
    overflows, an all-zero row (with eps = 0: 1 / sqrt(0) is infinite), a
    -inf in x, plus the ORDINARY rows; bf16 bit patterns."""
    x, r, w = case(8, h, seed)
    xb = refs.u16(x).copy()
    xb[1, 5] = 0x7FC0           # NaN
    xb[2, :] = 0x7F00           # 2^127: squares overflow
    xb[3, :] = 0x0000           # zero row
    xb[4, 7] = 0xFF80           # -inf
    rb = np.zeros_like(xb)
    tx = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    tr = torch.from_numpy(rb.view(np.int16)).view(torch.bfloat16)
    return tx, tr, w


@pytest.mark.parametrize("variant", [dr.VARIANT_WARP, dr.VARIANT_STAGED, dr.VARIANT_ROWS])
@pytest.mark.parametrize("h", [1024, 4096])
def test_special_rows_match_the_oracle(orc, variant, h):
    x, r, w = special_rows(h, h + variant)
    cfg = dr.LaunchConfig(variant=variant)
    run_all(orc, x, r, w, 0.0, cfg, add=False, e2m1_rows=ORDINARY)
    run_all(orc, x, r, w, 1e-6, cfg, add=False, e2m1_rows=ORDINARY)
    if variant != dr.VARIANT_WARP or h <= 2048:
        run_all(orc, x, r, w, 1e-6, cfg, add=True, e2m1_rows=ORDINARY)


@pytest.mark.parametrize("variant", [dr.VARIANT_WARP, dr.VARIANT_STAGED, dr.VARIANT_ROWS])
def test_non_finite_weights_match_the_oracle(orc, variant):
    x, r, w = case(6, 1024, 9)
    wb = refs.u16(w).copy()
    wb[3] = 0x7F80              # +inf weight
    wb[10] = 0x7FC0             # NaN weight
    tw = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16)
    none = slice(0, 0)  # every row holds a NaN y (the NaN weight's column)
    run_all(orc, x, r, tw, 1e-6, dr.LaunchConfig(variant=variant), add=False, e2m1_rows=none)
    run_all(orc, x, r, tw, 1e-6, dr.LaunchConfig(variant=variant), add=True, e2m1_rows=none)
