"""The fused q/k RMSNorm entry points on the host, without a GPU: argument
checks and the launch plan.  Every call made here returns before any CUDA
runtime call; nothing is launched."""
import pytest

import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import build as drbuild

MB = 1 << 20
BASE = 1 << 41
Q, QR, QW, K, KW, QO, QS, QRO, KO = (BASE + i * 256 * MB for i in range(9))


@pytest.fixture(scope="module")
def L():
    drbuild.build()
    return dr.lib()


def call(L, qo=QO, qs=QS, qro=QRO, ko=KO, q=Q, qr=QR, qw=QW, k=K, kw=KW, q_eps=1e-6, k_eps=1e-6,
         nq=4, hq=1536, nk=4, hk=512, g=128):
    return L.fused_qk_rmsnorm_group_quant_fwd(qo, qs, qro, ko, q, qr, qw, k, kw, q_eps, k_eps, nq, hq, nk, hk,
                                              g, None)


@pytest.mark.parametrize("kw,code", [
    (dict(nq=-1), 2), (dict(nk=-1), 2), (dict(g=-8), 2), (dict(hq=0), 2), (dict(hk=-8), 2),
    (dict(hq=12), 3), (dict(hk=1001), 3), (dict(hq=16392), 3), (dict(hq=32768), 3),
    (dict(nq=1 << 62, hq=8), 2),
    (dict(g=96), 2), (dict(g=4), 2), (dict(g=512), 2), (dict(hq=200, g=16), 2),
    (dict(qo=0), 1), (dict(qs=0), 1), (dict(qro=0), 1), (dict(ko=0), 1), (dict(q=0), 1),
    (dict(qw=0), 1), (dict(k=0), 1), (dict(kw=0), 1),
    (dict(qo=QO + 8), 4), (dict(q=Q + 2), 4), (dict(qs=QS + 2), 4), (dict(qr=QR + 8), 4),
    (dict(qro=QRO + 4), 4), (dict(ko=KO + 8), 4), (dict(kw=KW + 2), 4),
    (dict(q_eps=float("nan")), 5), (dict(k_eps=-1.0), 5), (dict(k_eps=float("inf")), 5),
    (dict(qo=Q), 6),               # e4m3 codes may not overwrite q
    (dict(ko=Q), 6),               # k out over q
    (dict(qro=QR + 16), 6),        # shifted alias of the residual
    (dict(qs=QO + 1024), 6),       # scales inside the codes
    (dict(ko=KW), 6),              # output over a weight
    (dict(qro=KO), 6),             # two outputs the same buffer
])
def test_argument_errors(L, kw, code):
    assert call(L, **kw) == code


@pytest.mark.parametrize("kw", [
    dict(nq=0, nk=0),                                   # nothing to do
])
def test_noop(L, kw):
    assert call(L, **kw) == 0


def test_inactive_side_is_not_inspected(L):
    # with no k rows, k's pointers, hidden and eps are ignored: the q checks
    # still run (a NULL q_out is reported) ...
    assert call(L, nk=0, k=0, kw=0, ko=0, hk=-5, k_eps=float("nan"), qo=0) == 1
    # ... and with no q rows, q's
    assert call(L, nq=0, q=0, qw=0, qo=0, qs=0, hq=12, g=96, q_eps=-1.0, k=0) == 1


def test_bf16_q_may_be_updated_in_place_but_not_codes(L):
    # group_size 0: q_out == q is allowed (reaches the device query, which
    # fails without a GPU); with codes it is an alias error
    assert call(L, qo=Q, g=128) == 6
    assert call(L, qo=Q, g=0) not in (1, 2, 3, 4, 5, 6, 9)
    assert call(L, qro=QR, ko=K) not in (1, 2, 3, 4, 5, 6, 9)


def test_residual_out_unused_without_residual(L):
    # q_residual NULL: q_residual_out is neither required nor checked
    assert call(L, qr=0, qro=0, qo=0) == 1
    assert call(L, qr=0, qro=QO, qo=0) == 1


def test_with_config_needs_config(L):
    assert L.fused_qk_rmsnorm_group_quant_fwd_with_config(QO, QS, QRO, KO, Q, QR, QW, K, KW, 1e-6, 1e-6, 4,
                                                          1536, 4, 512, 128, None, None) == 1


# ------------------------------------------------------------------ the plan
@pytest.mark.parametrize("nq,hq,nk,hk,g", [
    (4096, 1536, 4096, 512, 128), (64 * 32, 128, 64 * 8, 128, 0), (8, 16384, 8, 512, 256),
    (1, 8, 1, 16, 8), (100000, 1536, 0, 512, 64), (0, 1536, 7, 4096, 0), (3, 200, 5, 24, 8),
    (2048, 8192, 2048, 1024, 32), (50, 256, 3, 64, 256), (7, 128, 7, 128, 128), (64, 2048, 64, 512, 8),
    (64, 1536, 64, 512, 16), (4096 * 32, 128, 4096 * 8, 128, 0), (256 * 32, 128, 256 * 8, 128, 0),
    (4096, 3072, 4096, 1024, 128), (2048, 4096, 2048, 1024, 0), (4096, 4096, 0, 512, 128), (9, 2000, 3, 4096, 0),
])
def test_plan_rules(nq, hq, nk, hk, g):
    p = dr.qk_resolve_config(nq, hq, nk, hk, g, q_residual=True, sm_count=152)
    B = p.threads_per_cta
    max_p = max(1 << (h - 1).bit_length() for n, h in ((nq, hq), (nk, hk)) if n)
    rows = nq + nk
    max_stages = 2
    min_p = min(1 << (h - 1).bit_length() for n, h in ((nq, hq), (nk, hk)) if n)
    pq = 1 << (hq - 1).bit_length()
    pk = 1 << (hk - 1).bit_length()
    if nq and 512 < pq <= 4096 and (not nk or 256 <= pk <= 2048):
        # q rows of 512 < P <= 4096: 512-element chunks, one warp each, one stage
        nw = -(-hq // 512)
        assert (p.variant, B) == (dr.VARIANT_CHUNK, 32 * nw)
        assert (p.q_threads_per_row, p.q_rows_per_cta, p.q_stages) == (32 * nw, 1, 1)
        return
    if 256 < min_p and max_p <= 2048 and rows >= 8192:
        # the low-rank q / kv class: one warp a row, rings of 2 slots, 128 threads
        assert (p.variant, B) == (dr.VARIANT_WARP, 128)
        for n, h, T, R, S, C in ((nq, hq, p.q_threads_per_row, p.q_rows_per_cta, p.q_stages, p.q_ctas),
                                 (nk, hk, p.k_threads_per_row, p.k_rows_per_cta, p.k_stages, p.k_ctas)):
            if n:
                assert (T, R, S) == (32, 4, 2) and 1 <= C <= -(-n // R)
        return
    if max_p <= 256 and rows > 16384:
        assert (p.variant, B) == (2, 128)
        least_k = 4
        max_stages = 3
    elif max_p <= 256:
        assert (p.variant, B) == (1, 128)
        least_k = 1 if rows > 4096 else 2
    elif max_p <= 2048:
        assert B == (256 if rows >= 8192 else 128)
        least_k = 1 if rows >= 8192 else 2
        # the register variant, unless its q split would span groups
        assert p.variant == 1 or (g and (1 << (hq - 1).bit_length()) // 8 // B > g // 8)
    else:
        assert p.variant == 2 and B == min(512, max(128, max_p // 8))
        least_k = 1
    for side, n, h, T, R, C in (("q", nq, hq, p.q_threads_per_row, p.q_rows_per_cta, p.q_ctas),
                                ("k", nk, hk, p.k_threads_per_row, p.k_rows_per_cta, p.k_ctas)):
        if n == 0:
            assert (T, R, C) == (0, 0, 0)
            continue
        P = 1 << (h - 1).bit_length()
        K = P // 8 // T
        assert T * R == B and K * T == P // 8 and K in (1, 2, 4, 8)
        kmin = 1
        while P // 8 // kmin > B:
            kmin *= 2
        pref = min(least_k, P // 8)
        if side == "q" and g:
            pref = min(pref, P // 8 // (g // 8))
            if p.variant == 1:
                pref = min(pref, g // 8)
                assert max(kmin, pref) <= g // 8  # else the plan takes the staged variant
        assert K == max(kmin, pref)
        assert 1 <= C <= -(-n // R)
    assert p.q_ctas + p.k_ctas <= 152 * 2048 // B
    if nq and g:
        assert g // 8 <= p.q_threads_per_row
    # staged: up to 2 stages of R rows per side (3 for short rows in large
    # batches), within 96 KiB unless one stage alone is larger
    for n, h, R, S, res in ((nq, hq, p.q_rows_per_cta, p.q_stages, True),
                            (nk, hk, p.k_rows_per_cta, p.k_stages, False)):
        if n == 0 or p.variant == 1:
            assert S == 0
            continue
        stage = (4 if res else 2) * h * R
        assert 1 <= S <= max_stages and (S * stage <= 96 * 1024 or S == 1)
        assert p.dyn_smem_bytes >= S * (stage + 8)


def test_plan_rows_variant_and_stage_limits():
    p = dr.qk_resolve_config(64, 1536, 64, 512, 128, q_residual=True, config=dr.LaunchConfig(variant=1))
    assert p.variant == 1 and p.q_stages == 0 and p.k_stages == 0 and p.dyn_smem_bytes == 0
    p = dr.qk_resolve_config(64, 1536, 64, 512, 128, q_residual=True, config=dr.LaunchConfig(stages=8))
    assert p.q_stages == 8 and p.k_stages == 8 and p.dyn_smem_bytes == 8 * (4 * 1536 + 8)
    # 16384-element q rows with a residual: 64 KiB a stage; 3 stages fit in
    # 227 KiB, 4 do not
    p = dr.qk_resolve_config(8, 16384, 0, 0, 0, q_residual=True, config=dr.LaunchConfig(stages=3))
    assert p.q_stages == 3
    with pytest.raises(dr.DraddError) as e:
        dr.qk_resolve_config(8, 16384, 0, 0, 0, q_residual=True, config=dr.LaunchConfig(stages=4))
    assert e.value.status == 9
    assert dr.qk_resolve_config(8, 16384, 0, 0, 0, q_residual=True).q_stages == 1
    assert dr.qk_resolve_config(0, 16384, 0, 0, 0).variant == 0
    p = dr.qk_resolve_config(64, 1536, 64, 512, 128, q_residual=True, config=dr.LaunchConfig(variant=2))
    assert p.variant == 2 and p.q_stages == 2


def test_plan_blocks_per_thread():
    # a preferred K is raised where the CTA size needs more, capped at P / 8
    for K in (1, 2, 4, 8):
        p = dr.qk_resolve_config(64, 1536, 64, 512, 128, config=dr.LaunchConfig(threads_per_row=128,
                                                                               blocks_per_thread=K))
        kq = 256 // p.q_threads_per_row
        kk = 64 // p.k_threads_per_row
        assert kq == max(K, 2) and kk == K
        assert p.q_threads_per_row * p.q_rows_per_cta == 128 == p.k_threads_per_row * p.k_rows_per_cta
    p = dr.qk_resolve_config(64, 16, 0, 0, 0, config=dr.LaunchConfig(blocks_per_thread=8))
    assert p.q_threads_per_row == 1


def test_plan_explicit_threads_and_grid():
    for B in (64, 128, 256, 512):
        p = dr.qk_resolve_config(64, 4096, 64, 512, 128, config=dr.LaunchConfig(threads_per_row=B))
        assert p.threads_per_cta == B
    p = dr.qk_resolve_config(64, 4096, 64, 512, 128, config=dr.LaunchConfig(threads_per_row=256, grid_ctas=7))
    assert p.q_ctas + p.k_ctas == 7 and p.q_ctas >= 1 and p.k_ctas >= 1
    p = dr.qk_resolve_config(64, 4096, 0, 512, 128, config=dr.LaunchConfig(grid_ctas=1))
    assert (p.q_ctas, p.k_ctas) == (1, 0)
    # K = 8 needs at most 256 threads; 1024 is never allowed; 32 cannot hold
    # a 4096-element row with K <= 8
    p = dr.qk_resolve_config(64, 8192, 0, 0, 0, config=dr.LaunchConfig(threads_per_row=128))
    assert p.q_threads_per_row == 128
    for cfg in (dr.LaunchConfig(threads_per_row=1024), dr.LaunchConfig(threads_per_row=32),
                dr.LaunchConfig(threads_per_row=96), dr.LaunchConfig(variant=3),
                dr.LaunchConfig(rows_per_cta=2), dr.LaunchConfig(stages=9), dr.LaunchConfig(stages=-1),
                dr.LaunchConfig(variant=1, stages=1), dr.LaunchConfig(variant=1, fault_inject=1),
                dr.LaunchConfig(grid_ctas=1), dr.LaunchConfig(serialize=2), dr.LaunchConfig(wait_limit_us=-1),
                dr.LaunchConfig(blocks_per_thread=3), dr.LaunchConfig(blocks_per_thread=16)):
        with pytest.raises(dr.DraddError) as e:
            dr.qk_resolve_config(64, 4096, 64, 512, 128, config=cfg)
        assert e.value.status == 9
    with pytest.raises(dr.DraddError) as e:
        dr.qk_resolve_config(64, 16384, 0, 0, 0, config=dr.LaunchConfig(threads_per_row=512 // 2 // 2))
    assert e.value.status == 9
    # a group never spans more lanes than a row has threads: with K > 1,
    # T > B / 2 >= 16, and a group is at most 32 blocks
    for B in (32, 64, 128, 256, 512):
        for hq in (256, 512, 2048, 8192):
            try:
                p = dr.qk_resolve_config(4, hq, 0, 0, 256, config=dr.LaunchConfig(threads_per_row=B))
            except dr.DraddError as e:
                assert e.status == 9
                continue
            assert p.q_threads_per_row >= 32


CHUNK = dr.LaunchConfig(variant=dr.VARIANT_CHUNK)


@pytest.mark.parametrize("nq,hq,nk,hk,nw", [(4096, 1536, 4096, 512, 3), (100, 1280, 0, 512, 3), (7, 600, 9, 256, 2),
                                            (33, 4096, 12, 2048, 8), (5, 3000, 5, 1024, 6)])
def test_chunk_plan(nq, hq, nk, hk, nw):
    """CHUNK: a q row is one CTA of ceil(hq / 512) warps, a chunk each; the k
    rows one warp each in CTAs of as many warps; 2 ring slots per warp; the
    CTAs at most one per q row and one per nw k rows."""
    p = dr.qk_resolve_config(nq, hq, nk, hk, 0, q_residual=True, sm_count=152, config=CHUNK)
    assert p.variant == dr.VARIANT_CHUNK and p.threads_per_cta == 32 * nw
    assert (p.q_threads_per_row, p.q_rows_per_cta, p.q_stages) == (32 * nw, 1, 2)
    assert 1 <= p.q_ctas <= nq
    if nk:
        assert (p.k_threads_per_row, p.k_rows_per_cta, p.k_stages) == (32, nw, 2)
        assert 1 <= p.k_ctas <= -(-nk // nw)
    else:
        assert p.k_ctas == 0


@pytest.mark.parametrize("nq,hq,nk,hk,kw", [
    (64, 512, 64, 512, {}),                   # q P = 512: one warp a row already
    (64, 8192, 64, 512, {}),                  # q P > 4096
    (0, 1536, 64, 512, {}),                   # no q rows
    (64, 1536, 64, 4096, {}),                 # k P > 2048
    (64, 1536, 64, 128, {}),                  # k P < 256
    (64, 1536, 64, 512, {"threads_per_row": 128}),
    (64, 1536, 64, 512, {"blocks_per_thread": 2}),
    (64, 1536, 64, 512, {"rows_per_cta": 2}),
    (64, 1536, 64, 512, {"stages": 9}),
])
def test_chunk_plan_refusals(nq, hq, nk, hk, kw):
    with pytest.raises(dr.DraddError) as e:
        dr.qk_resolve_config(nq, hq, nk, hk, 0, sm_count=152, config=dr.LaunchConfig(variant=dr.VARIANT_CHUNK, **kw))
    assert e.value.status == 9


def test_chunk_variant_is_the_fused_calls_only():
    with pytest.raises(dr.DraddError) as e:
        dr.resolve_config(4096, 4096, sm_count=152, config=CHUNK)
    assert e.value.status == 9
