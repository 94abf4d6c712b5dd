"""Fused q/k RMSNorm on the GPU through the C ABI, against the oracle bit
for bit: per-group e4m3 codes and scales, bf16 q out, q residual_out and
k out, at the shapes of a low-rank q / kv norm (1536 + 512 per token), of a
per-head q/k norm (heads of 128), ragged and single-sided calls; the same
bits under every launch configuration; equal to the single-set entry points;
in place."""
import numpy as np
import pytest
import torch

import refs
import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import inputs
from gpu_util import assert_bits_equal, dev

pytestmark = pytest.mark.gpu


def make(seed, nq, hq, nk, hk, with_res, q_std=1.0):
    g = inputs.generator(seed)
    q = inputs.normal_bf16(g, (nq, hq), 0.0, q_std)
    r = inputs.normal_bf16(g, (nq, hq), 0.0, 4.0) if with_res else None
    qw = inputs.normal_bf16(g, (hq,), 1.0, 0.1)
    k = inputs.normal_bf16(g, (nk, hk), 0.0, 2.0)
    kw = inputs.normal_bf16(g, (hk,), 1.0, 0.1)
    return q, r, qw, k, kw


def run_gpu(q, r, qw, k, kw, group, q_eps, k_eps, config=None):
    d = dev()
    res = dr.fused_qk_rmsnorm_group_quant_fwd(
        q.to(d), qw.to(d), k.to(d), kw.to(d), q_eps, k_eps, group_size=group,
        q_residual=None if r is None else r.to(d), config=config)
    torch.cuda.synchronize()
    return res


def compare(orc, q, r, qw, k, kw, group, q_eps, k_eps, got, what=""):
    exp = orc.qk_rmsnorm_fwd(q, qw, k, kw, q_eps, k_eps, group_size=group, q_residual=r)
    qo, qs, qro, ko = got
    if group:
        assert_bits_equal(qo.cpu().numpy(), exp["q_out"], f"{what} q codes")
        assert_bits_equal(qs.cpu().numpy().view(np.uint32), exp["q_scale"].view(np.uint32), f"{what} q scales")
    else:
        assert qs is None
        assert_bits_equal(refs.u16(qo), exp["q_out"], f"{what} q out")
    if r is not None:
        assert_bits_equal(refs.u16(qro), exp["q_residual_out"], f"{what} q residual_out")
    else:
        assert qro is None
    assert_bits_equal(refs.u16(ko), exp["k_out"], f"{what} k out")


CASES = [
    # nq, hq, nk, hk, group, residual, q_eps, k_eps
    (256, 1536, 256, 512, 128, True, 1e-6, 1e-6),
    (256, 1536, 256, 512, 128, False, 1e-6, 1e-6),
    (4096, 1536, 4096, 512, 128, True, 1e-6, 1e-6),
    (64 * 32, 128, 64 * 8, 128, 0, False, 1e-6, 1e-6),
    (300, 4096, 300, 512, 0, True, 1e-5, 0.5),
    (37, 200, 53, 24, 8, True, 0.0, 1e-6),
    (5, 1000, 3, 8, 8, False, 1e-6, 0.0),
    (16, 16384, 16, 512, 256, True, 1e-6, 1e-6),
    (8, 8192, 4, 8192, 64, False, 1e-6, 1e-6),
    (24, 2048, 24, 16384, 32, True, 1e-6, 1e-6),
    (0, 1536, 100, 512, 128, True, 1e-6, 1e-6),
    (100, 1536, 0, 512, 128, True, 1e-6, 1e-6),
    (1, 8, 1, 16, 8, True, 1e-6, 1e-6),
    (3, 64, 2, 64, 16, False, 1e-6, 1e-6),
    # q rows whose data fill at most three quarters of their warp slices
    (77, 1280, 45, 512, 128, True, 1e-6, 1e-6),
    (70, 640, 33, 768, 64, True, 1e-6, 1e-6),
    (66, 768, 20, 1024, 0, True, 1e-6, 1e-6),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("r" if c[5] else ""))
def test_parity(orc, case):
    nq, hq, nk, hk, group, with_res, qe, ke = case
    q, r, qw, k, kw = make(hash(case) % 1000, nq, hq, nk, hk, with_res)
    got = run_gpu(q, r, qw, k, kw, group, qe, ke)
    compare(orc, q, r, qw, k, kw, group, qe, ke, got)
    assert dr.device_status() == 0


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("r" if c[5] else ""))
def test_parity_warp_rows(orc, case):
    """The warp-per-row mode on every case whose two sides it takes (both
    256 <= P <= 2048)."""
    nq, hq, nk, hk, group, with_res, qe, ke = case
    cfg = dr.LaunchConfig(variant=dr.VARIANT_WARP)
    try:
        dr.qk_resolve_config(nq, hq, nk, hk, group, q_residual=with_res, config=cfg)
    except dr.DraddError as e:
        assert e.status == 9
        pytest.skip("a side outside 256 <= P <= 2048")
    q, r, qw, k, kw = make(hash(case) % 1000 + 1, nq, hq, nk, hk, with_res)
    got = run_gpu(q, r, qw, k, kw, group, qe, ke, config=cfg)
    compare(orc, q, r, qw, k, kw, group, qe, ke, got, what="warp")
    assert dr.device_status() == 0


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("r" if c[5] else ""))
def test_parity_chunk_rows(orc, case):
    """The chunked-q mode on every case it takes (q 512 < P <= 4096, k
    256 <= P <= 2048 or no k rows)."""
    nq, hq, nk, hk, group, with_res, qe, ke = case
    cfg = dr.LaunchConfig(variant=dr.VARIANT_CHUNK)
    try:
        dr.qk_resolve_config(nq, hq, nk, hk, group, q_residual=with_res, config=cfg)
    except dr.DraddError as e:
        assert e.status == 9
        pytest.skip("a side outside the chunked mode's widths")
    q, r, qw, k, kw = make(hash(case) % 1000 + 2, nq, hq, nk, hk, with_res)
    got = run_gpu(q, r, qw, k, kw, group, qe, ke, config=cfg)
    compare(orc, q, r, qw, k, kw, group, qe, ke, got, what="chunk")
    assert dr.device_status() == 0


CONFIGS = ([None] +
           [dr.LaunchConfig(variant=1, threads_per_row=B, grid_ctas=G)
            for B in (64, 128, 256, 512) for G in (0, 2, 7, 1000)] +
           [dr.LaunchConfig(variant=2, threads_per_row=B, grid_ctas=G, stages=S)
            for B, G, S in ((64, 0, 1), (128, 2, 2), (256, 7, 3), (512, 0, 4), (128, 1000, 8), (256, 3, 1))] +
           [dr.LaunchConfig(variant=v, threads_per_row=128, blocks_per_thread=K)
            for v in (1, 2) for K in (2, 4, 8)] +
           [dr.LaunchConfig(variant=dr.VARIANT_WARP, threads_per_row=B, grid_ctas=G)
            for B in (64, 256) for G in (0, 3)] +
           [dr.LaunchConfig(variant=dr.VARIANT_CHUNK, stages=S, grid_ctas=G) for S, G in ((1, 0), (3, 5), (2, 2))] +
           [dr.LaunchConfig(serialize=1), dr.LaunchConfig(variant=1, serialize=1)])


@pytest.mark.parametrize("group,with_res", [(128, True), (0, False), (16, False)])
def test_launch_configuration_invariance(orc, group, with_res):
    q, r, qw, k, kw = make(7, 123, 1536, 77, 512, with_res)
    exp = orc.qk_rmsnorm_fwd(q, qw, k, kw, 1e-6, 1e-6, group_size=group, q_residual=r)
    digests = set()
    ran = 0
    for cfg in CONFIGS:
        try:
            dr.qk_resolve_config(123, 1536, 77, 512, group, q_residual=with_res, config=cfg)
        except dr.DraddError as e:
            # a register-variant split whose threads would straddle groups
            assert e.status == 9 and cfg is not None and cfg.variant == 1 and group
            continue
        ran += 1
        qo, qs, qro, ko = run_gpu(q, r, qw, k, kw, group, 1e-6, 1e-6, config=cfg)
        parts = [(qo.cpu().numpy() if group else refs.u16(qo)).tobytes(), refs.u16(ko).tobytes()]
        if group:
            parts.append(qs.cpu().numpy().tobytes())
        if with_res:
            parts.append(refs.u16(qro).tobytes())
        digests.add(hash(b"".join(parts)))
        compare(orc, q, r, qw, k, kw, group, 1e-6, 1e-6, (qo, qs, qro, ko), what=str(cfg))
    assert len(digests) == 1 and ran >= 20
    assert exp["k_out"].size > 0


def test_equals_single_set_calls():
    d = dev()
    q, r, qw, k, kw = make(11, 96, 4096, 80, 1024, True)
    qd, rd, qwd, kd, kwd = (t.to(d) for t in (q, r, qw, k, kw))
    qo, _, qro, ko = dr.fused_qk_rmsnorm_group_quant_fwd(qd, qwd, kd, kwd, 1e-6, 1e-5, q_residual=rd)
    out, ro = dr.add_rmsnorm_fwd(qd, rd, qwd, 1e-6)
    kk = dr.rmsnorm_fwd(kd, kwd, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(qo.view(torch.int16), out.view(torch.int16))
    assert torch.equal(qro.view(torch.int16), ro.view(torch.int16))
    assert torch.equal(ko.view(torch.int16), kk.view(torch.int16))
    # one group per row is the per-row e4m3 output
    q, r, qw, k, kw = make(12, 50, 256, 3, 64, True)
    qd, rd, qwd, kd, kwd = (t.to(d) for t in (q, r, qw, k, kw))
    qo, qs, qro, _ = dr.fused_qk_rmsnorm_group_quant_fwd(qd, qwd, kd, kwd, 1e-6, 1e-6, group_size=256,
                                                         q_residual=rd)
    c8, s8, ro8 = dr.add_rmsnorm_fp8_fwd(qd, rd, qwd, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(qo, c8) and torch.equal(qs[:, 0], s8) and torch.equal(qro.view(torch.int16),
                                                                           ro8.view(torch.int16))


def test_in_place(orc):
    d = dev()
    q, r, qw, k, kw = make(13, 64, 1536, 64, 512, True)
    exp = orc.qk_rmsnorm_fwd(q, qw, k, kw, 1e-6, 1e-6, group_size=0, q_residual=r)
    qd, rd, kd = q.to(d), r.to(d), k.to(d)
    dr.fused_qk_rmsnorm_group_quant_fwd(qd, qw.to(d), kd, kw.to(d), 1e-6, 1e-6, q_residual=rd, q_out=qd,
                                        q_residual_out=rd, k_out=kd)
    torch.cuda.synchronize()
    assert_bits_equal(refs.u16(qd), exp["q_out"], "q in place")
    assert_bits_equal(refs.u16(rd), exp["q_residual_out"], "residual in place")
    assert_bits_equal(refs.u16(kd), exp["k_out"], "k in place")


def test_zero_groups_and_tiny_scales(orc):
    # whole zero groups, zero rows, and weights so small that the group
    # scales are subnormal (the exact-division path of the encoder)
    q, r, qw, k, kw = make(14, 40, 512, 4, 64, False)
    q = q.clone()
    q[:, 128:256] = 0
    q[5] = 0
    qw = qw.clone()
    qw[256:384] = torch.tensor(0x0003, dtype=torch.int16).view(torch.bfloat16)   # subnormal weights
    qw[384:448] = 0
    for group in (128, 64, 8):
        got = run_gpu(q, None, qw, k, kw, group, 1e-6, 1e-6)
        compare(orc, q, None, qw, k, kw, group, 1e-6, 1e-6, got, what=f"group {group}")
        s = got[1].cpu().numpy()
        assert np.all(s[5] == 0)


@pytest.mark.parametrize("variant", [2, dr.VARIANT_WARP, dr.VARIANT_CHUNK])
def test_bounded_wait_expires_and_recovers(orc, variant):
    """fault_inject withholds each CTA's first staged copy on both sides:
    every wait runs out after wait_limit_us, the kernel records
    DRADD_ERR_TIMEOUT, drains its other copies and returns; the context
    stays usable."""
    d = dev()
    assert dr.device_status(clear=True) == 0
    q, r, qw, k, kw = make(15, 64, 1536, 64, 512, True)
    qd, rd, qwd, kd, kwd = (t.to(d) for t in (q, r, qw, k, kw))
    cfg = dr.LaunchConfig(variant=variant, stages=3, grid_ctas=8, fault_inject=1, wait_limit_us=20000)
    dr.fused_qk_rmsnorm_group_quant_fwd(qd, qwd, kd, kwd, 1e-6, 1e-6, group_size=128, q_residual=rd, config=cfg)
    assert dr.device_status(clear=True) == 8
    assert dr.device_status(clear=True) == 0
    got = run_gpu(q, r, qw, k, kw, 128, 1e-6, 1e-6)
    compare(orc, q, r, qw, k, kw, 128, 1e-6, 1e-6, got, what="after timeout")
    assert dr.device_status(clear=True) == 0
