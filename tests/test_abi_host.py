"""The C ABI on the host, without a GPU: the library loads, exports every
function include/dradd.h declares, and its host logic (argument checks,
configuration choice) behaves as documented.  Every call made here returns
before any CUDA runtime call; nothing is launched."""
import ctypes
import re
from pathlib import Path

import pytest

import deterministic_residual_add_gb300 as dr
from deterministic_residual_add_gb300 import build as drbuild

ROOT = Path(__file__).resolve().parents[1]
HEADERS = sorted((ROOT / "include").glob("*.h"))


@pytest.fixture(scope="module")
def L():
    drbuild.build()
    return dr.lib()


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_headers_declare_the_entry_points():
    names = declared_functions()
    for n in ("add_rmsnorm_fwd", "add_rmsnorm_quant_fwd", "add_rmsnorm_fwd_with_config",
              "add_rmsnorm_quant_fwd_with_config", "dradd_resolve_config", "dradd_device_status",
              "dradd_bf16_convert_range", "dradd_status_string", "dradd_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libdradd.so does not export {name}"


def test_abi_version_and_status_strings(L):
    assert dr.abi_version() == 1
    for code, name in dr.STATUS_NAMES.items():
        assert name in dr.status_string(code)
    assert "UNKNOWN" in dr.status_string(1234)


# Fake, 256-byte aligned "device" addresses far apart: validation reads only
# the values of the pointers, never the memory.
MB = 1 << 20
BASE = 1 << 40
X, RES, W, OUT, RO, Q, SC = (BASE + i * 256 * MB for i in range(7))


def call_bf16(L, out=OUT, ro=RO, x=X, res=RES, w=W, eps=1e-6, n=4, h=1024):
    return L.add_rmsnorm_fwd(out, ro, x, res, w, eps, n, h, None)


def call_quant(L, q=Q, sc=SC, ro=RO, x=X, res=RES, w=W, eps=1e-6, n=4, h=1024):
    return L.add_rmsnorm_quant_fwd(q, sc, ro, x, res, w, eps, n, h, None)


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), 2), (dict(h=0), 2), (dict(h=-8), 2),
    (dict(h=12), 3), (dict(h=32776), 3), (dict(h=1001), 3),
    (dict(n=1 << 62), 2),
    (dict(out=0), 1), (dict(ro=0), 1), (dict(x=0), 1), (dict(res=0), 1), (dict(w=0), 1),
    (dict(out=OUT + 8), 4), (dict(x=X + 2), 4), (dict(w=W + 4), 4),
    (dict(eps=float("nan")), 5), (dict(eps=float("inf")), 5), (dict(eps=-1e-6), 5),
    (dict(ro=OUT), 6),                 # both outputs the same buffer
    (dict(out=X + 1024), 6),           # partial overlap with x
    (dict(ro=W), 6),                   # output over the weight
    (dict(ro=RES + 16), 6),            # shifted alias of residual
])
def test_bf16_argument_errors(L, kw, code):
    assert call_bf16(L, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(sc=0), 1), (dict(sc=SC + 2), 4), (dict(q=Q + 8), 4),
    (dict(q=X), 6),                    # int8 out over the bf16 input
    (dict(sc=RO + 64), 6),             # scale inside residual_out
    (dict(h=24, n=0), 0),
])
def test_quant_argument_errors(L, kw, code):
    assert call_quant(L, **kw) == code


def test_zero_rows_is_a_noop(L):
    # n_rows == 0 succeeds before the pointers are looked at
    assert call_bf16(L, n=0, out=0, ro=0, x=0, res=0, w=0) == 0
    assert call_quant(L, n=0, q=0, sc=0, ro=0, x=0, res=0, w=0) == 0


def test_config_pointer_required(L):
    assert L.add_rmsnorm_fwd_with_config(OUT, RO, X, RES, W, 1e-6, 4, 1024, None, None) == 1


def test_convert_hook_argument_errors(L):
    assert L.dradd_bf16_convert_range(None, 0, 16, 0, None) == 1
    assert L.dradd_bf16_convert_range(OUT, 0, -1, 0, None) == 2
    assert L.dradd_bf16_convert_range(OUT + 1, 0, 16, 0, None) == 4
    assert L.dradd_bf16_convert_range(OUT, 0, 16, 6, None) == 9
    assert L.dradd_bf16_convert_range(OUT, 0, 0, 0, None) == 0


# --------------------------------------------------------- configuration choice
def test_auto_config_covers_every_supported_hidden(L):
    for h in range(8, dr.MAX_HIDDEN + 1, 8):
        c = dr.resolve_config(4096, h, sm_count=152)
        P = 1 << (h - 1).bit_length()
        T, R = c.threads_per_row, c.rows_per_cta
        K = P // 8 // T
        assert T * K * 8 == P and K in (1, 2, 4, 8)
        assert (T * R) % 32 == 0 and T * R <= (1024 if K <= 2 else 512)
        # 512 <= P <= 2048 with 4096 rows: the warp-per-row variant (one warp
        # a row); longer rows staged, shorter ones in registers
        assert c.variant == (dr.VARIANT_WARP if 256 < h <= 2048 else
                             dr.VARIANT_STAGED if h > 256 else dr.VARIANT_ROWS)
        if c.variant == dr.VARIANT_WARP:
            assert (T, R, c.stages, c.blocks_per_thread) == (32, 4, 3, P // 256)
        if c.variant == dr.VARIANT_STAGED:
            assert 1 <= c.stages <= 8 and c.stages * 4 * h <= 232448
        assert c.grid_ctas >= 1


def test_auto_grid(L):
    c = dr.resolve_config(4096, 4096, sm_count=152)
    assert (c.variant, c.threads_per_row, c.rows_per_cta, c.stages) == (dr.VARIANT_STAGED, 128, 1, 2)
    assert c.grid_ctas % 152 == 0
    c = dr.resolve_config(2048, 4096, sm_count=152)
    assert (c.threads_per_row, c.stages) == (128, 3)
    c = dr.resolve_config(16384, 4096, sm_count=152)
    assert (c.threads_per_row, c.stages) == (128, 1)
    c = dr.resolve_config(16384, 4096, quant=True, sm_count=152)
    assert (c.threads_per_row, c.stages) == (128, 1)
    c = dr.resolve_config(4096, 4096, quant=True, sm_count=152)
    assert (c.threads_per_row, c.stages) == (128, 2)
    c = dr.resolve_config(2048, 16384, quant=True, sm_count=152)
    assert (c.variant, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 512, 2)
    assert c.grid_ctas % 152 == 0 or c.grid_ctas == 2048
    c = dr.resolve_config(4096, 8192, sm_count=152)
    assert (c.variant, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 1024, 2)
    for h in (264, 512, 1024, 2048):
        c = dr.resolve_config(4096, h, sm_count=152)
        assert (c.variant, c.threads_per_row, c.rows_per_cta, c.stages) == (dr.VARIANT_WARP, 32, 4, 3), h
    for h, T, S in [(264, 32, 4), (512, 32, 4), (1024, 64, 3), (2048, 128, 4)]:
        c = dr.resolve_config(512, h, sm_count=152)  # fewer rows: staged
        assert (c.variant, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, T, S), h
    c = dr.resolve_config(16384, 2048, quant=True, sm_count=152)
    assert (c.variant, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 64, 3)
    # few rows of 32768: the split-row cluster variant (bf16 out only)
    for n, C in ((1, 4), (64, 4), (65, 2), (160, 2)):
        c = dr.resolve_config(n, 32768, sm_count=152)
        assert (c.variant, c.cluster_ctas) == (dr.VARIANT_SPLIT, C), n
    assert dr.resolve_config(161, 32768, sm_count=152).variant == dr.VARIANT_STAGED
    assert dr.resolve_config(8, 32768, quant=True, sm_count=152).variant != dr.VARIANT_SPLIT
    c = dr.resolve_config(4096, 4096, add=False, sm_count=152)
    assert c.stages == 4
    c = dr.resolve_config(2048, 4096, add=False, sm_count=152)
    assert c.stages == 2
    c = dr.resolve_config(3, 64, sm_count=152)
    assert c.threads_per_row == 8 and c.rows_per_cta == 16 and c.grid_ctas == 1


@pytest.mark.parametrize("cfg", [
    dict(variant=4),
    dict(threads_per_row=384),              # not a power of two
    dict(threads_per_row=2048),
    dict(threads_per_row=64),               # K = 16 for P = 8192
    dict(threads_per_row=512, rows_per_cta=3),
    dict(threads_per_row=16, rows_per_cta=1),  # 16 threads is not whole warps
    dict(variant=2, threads_per_row=16),    # staged needs whole warps per row
    dict(variant=2, rows_per_cta=2),
    dict(variant=2, stages=9),
    dict(variant=1, stages=2),
    dict(variant=1, fault_inject=1),
    dict(grid_ctas=-1),
    dict(wait_limit_us=-5),
])
def test_bad_configs_rejected(L, cfg):
    with pytest.raises(dr.DraddError) as e:
        dr.resolve_config(4096, 8192, sm_count=152, config=dr.LaunchConfig(**cfg))
    assert e.value.status == 9


def test_staged_pair_rule(L):
    """rows_per_cta = 2 on the staged variant: the plain quantised forms'
    two-rows-per-thread kernel, K <= 4; refused for bf16 out, the residual
    forms and K = 8; its grid is at most one CTA per pair of rows."""
    pair = dr.LaunchConfig(variant=dr.VARIANT_STAGED, rows_per_cta=2)
    for kw in (dict(), dict(fp8=True), dict(fp4=True)):
        c = dr.resolve_config(4096, 4096, quant=True, add=False, sm_count=152, config=pair, **kw)
        assert (c.variant, c.rows_per_cta, c.threads_per_row, c.blocks_per_thread) == (dr.VARIANT_STAGED, 2, 128, 4)
        assert 1 <= c.grid_ctas <= 2048
    c = dr.resolve_config(5, 4096, quant=True, add=False, sm_count=152, config=pair)
    assert c.grid_ctas == 3
    for kw in (dict(quant=False, add=False), dict(quant=True, add=True)):
        with pytest.raises(dr.DraddError) as e:
            dr.resolve_config(4096, 4096, sm_count=152, config=pair, **kw)
        assert e.value.status == 9
    with pytest.raises(dr.DraddError) as e:
        dr.resolve_config(64, 8192, quant=True, add=False, sm_count=152,
                          config=dr.LaunchConfig(variant=dr.VARIANT_STAGED, rows_per_cta=2, threads_per_row=128))
    assert e.value.status == 9


@pytest.mark.parametrize("n,h,T", [(16384, 1024, 64), (8192, 2048, 128), (2048, 8192, 256), (1024, 16384, 512),
                                   (512, 4096, 512), (608, 4096, 512), (608, 2048, 256), (609, 2048, 128),
                                   (37, 1000, 128)])
def test_auto_plain_quantised_takes_the_pair_kernel(L, n, h, T):
    for kw in (dict(), dict(fp8=True), dict(fp4=True)):
        c = dr.resolve_config(n, h, quant=True, add=False, sm_count=152, **kw)
        assert (c.variant, c.rows_per_cta, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 2, T, 1), (n, h, kw)
        assert c.grid_ctas <= (n + 1) // 2
    # not for bf16 out, the residual forms, P = 4096 beyond 4 rows per SM, P = 512 from 8192 rows or P = 32768
    assert dr.resolve_config(4096, 4096, add=False, sm_count=152).rows_per_cta == 1
    for kw in (dict(), dict(fp8=True)):
        c = dr.resolve_config(609, 4096, quant=True, add=False, sm_count=152, **kw)
        assert (c.variant, c.rows_per_cta, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 1, 128, 2)
    assert dr.resolve_config(4096, 4096, quant=True, sm_count=152).rows_per_cta == 1
    c = dr.resolve_config(8192, 512, quant=True, add=False, sm_count=152)  # P = 512: one row a CTA from 8192 rows
    assert (c.variant, c.rows_per_cta, c.threads_per_row) == (dr.VARIANT_STAGED, 1, 32)
    assert dr.resolve_config(64, 32768, quant=True, add=False, sm_count=152).rows_per_cta == 1


def test_staged_threads_cover_the_padded_row(L):
    """Every staged and pair launch resolve accepts has T threads of K
    blocks covering the padded row exactly (T * K * 8 = P), so the first
    K / 2 blocks of every thread lie in the row: the kernels skip the
    bounds test there."""
    accepted = 0
    for h in range(8, dr.MAX_HIDDEN + 1, 8):
        P = 1 << (h - 1).bit_length()
        for T in (32, 64, 128, 256, 512, 1024):
            for rows, kw in ((1, dict(add=True)), (2, dict(quant=True, add=False))):
                cfg = dr.LaunchConfig(variant=dr.VARIANT_STAGED, threads_per_row=T, rows_per_cta=rows)
                try:
                    c = dr.resolve_config(64, h, sm_count=152, config=cfg, **kw)
                except dr.DraddError:
                    continue
                accepted += 1
                K = c.blocks_per_thread
                assert c.threads_per_row == T and T * K * 8 == P, (h, T, rows)
                if K >= 2:
                    assert (T - 1) + (K // 2 - 1) * T < h // 8, (h, T, K)
    assert accepted > 10000


def test_staged_stages_limited_by_shared_memory(L):
    with pytest.raises(dr.DraddError):
        dr.resolve_config(16, 32768, sm_count=152, config=dr.LaunchConfig(variant=2, stages=2))
    c = dr.resolve_config(16, 32768, sm_count=152, config=dr.LaunchConfig(variant=2))
    assert c.stages == 1
    c = dr.resolve_config(200, 32768, sm_count=152)  # (16 rows would take the split variant)
    assert c.variant == dr.VARIANT_STAGED and c.stages == 1 and c.threads_per_row == 512


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        dr.add_rmsnorm_fwd(x, x.clone(), torch.ones(64, dtype=torch.bfloat16), 1e-6,
                           out=x.clone(), residual_out=x.clone())


# ----------------------------------------------- plain RMSNorm, residual add
@pytest.mark.parametrize("args,code", [
    ((OUT, X, W, 1e-6, 4, 1024), None),            # valid: not called (would launch)
    ((0, X, W, 1e-6, 4, 1024), 1), ((OUT, 0, W, 1e-6, 4, 1024), 1), ((OUT, X, 0, 1e-6, 4, 1024), 1),
    ((OUT + 8, X, W, 1e-6, 4, 1024), 4), ((OUT, X, W, -1.0, 4, 1024), 5),
    ((X + 64, X, W, 1e-6, 4, 1024), 6), ((W, X, W, 1e-6, 4, 1024), 6),
    ((OUT, X, W, 1e-6, 0, 1024), 0), ((OUT, X, W, 1e-6, 4, 20), 3),
])
def test_rmsnorm_argument_errors(L, args, code):
    if code is None:
        return
    assert L.rmsnorm_fwd(*args, None) == code


def test_rmsnorm_quant_and_residual_add_errors(L):
    assert L.rmsnorm_quant_fwd(0, SC, X, W, 1e-6, 4, 1024, None) == 1
    assert L.rmsnorm_quant_fwd(Q, SC + 1, X, W, 1e-6, 4, 1024, None) == 4
    assert L.rmsnorm_quant_fwd(X, SC, X, W, 1e-6, 4, 1024, None) == 6
    assert L.residual_add_fwd(0, X, RES, 4, 1024, None) == 1
    assert L.residual_add_fwd(RO, X + 4, RES, 4, 1024, None) == 4
    assert L.residual_add_fwd(X + 32, X, RES, 4, 1024, None) == 6
    assert L.residual_add_fwd(RO, X, RES, 4, 12, None) == 3
    assert L.residual_add_fwd(RO, X, RES, -2, 1024, None) == 2
    assert L.residual_add_fwd(0, 0, 0, 0, 1024, None) == 0
    assert L.rmsnorm_fwd_with_config(OUT, X, W, 1e-6, 4, 1024, None, None) == 1


def test_resolve_op_codes(L):
    c = dr.LaunchConfig()._c()
    assert L.dradd_resolve_config(16, 1024, 8, 152, ctypes.byref(c)) == 9
    plain = dr.resolve_config(4096, 16384, add=False)
    assert plain.variant == dr.VARIANT_STAGED and plain.stages == 4 and plain.threads_per_row == 512
    # a plain-RMSNorm stage holds only x, so 32768-wide rows fit two stages
    c = dr.resolve_config(16, 32768, add=False, config=dr.LaunchConfig(variant=2, stages=2))
    assert c.stages == 2


def test_fp8_argument_errors(L):
    assert L.add_rmsnorm_fp8_fwd(0, SC, RO, X, RES, W, 1e-6, 4, 1024, None) == 1
    assert L.add_rmsnorm_fp8_fwd(Q + 4, SC, RO, X, RES, W, 1e-6, 4, 1024, None) == 4
    assert L.add_rmsnorm_fp8_fwd(Q, SC, RO, X, RES, W, float("nan"), 4, 1024, None) == 5
    assert L.add_rmsnorm_fp8_fwd(RES, SC, RO, X, RES, W, 1e-6, 4, 1024, None) == 6
    assert L.rmsnorm_fp8_fwd(Q, 0, X, W, 1e-6, 4, 1024, None) == 1
    assert L.rmsnorm_fp8_fwd(Q, SC, X, W, 1e-6, 0, 1024, None) == 0
    assert L.rmsnorm_fp8_fwd_with_config(Q, SC, X, W, 1e-6, 4, 1024, None, None) == 1
    c = dr.resolve_config(4096, 4096, add=True, fp8=True)
    assert c.variant == dr.VARIANT_STAGED and c.stages == 2
    c = dr.resolve_config(4096, 4096, add=False, fp8=True)
    assert c.stages == 2


def test_fp4_argument_errors(L):
    assert L.add_rmsnorm_fp4_fwd(0, SC, RO, X, RES, W, 1e-6, 4, 1024, None) == 1
    assert L.add_rmsnorm_fp4_fwd(Q + 8, SC, RO, X, RES, W, 1e-6, 4, 1024, None) == 4
    # 4 x 1024 codes take 2048 bytes: starting 2032 bytes before residual_out overlaps it
    assert L.add_rmsnorm_fp4_fwd(RO - 2032, SC, RO, X, RES, W, 1e-6, 4, 1024, None) == 6
    assert L.rmsnorm_fp4_fwd(Q, SC, X, W, 1e-6, 0, 1024, None) == 0
    assert L.rmsnorm_fp4_fwd_with_config(Q, SC, X, W, 1e-6, 4, 1024, None, None) == 1
    c = dr.resolve_config(2048, 16384, add=True, fp4=True)
    assert c.variant == dr.VARIANT_STAGED and c.threads_per_row == 512


def test_blocks_per_thread_sets_or_checks_threads():
    c = dr.resolve_config(4096, 4096, sm_count=152, config=dr.LaunchConfig(blocks_per_thread=2))
    assert c.threads_per_row == 256 and c.blocks_per_thread == 2
    c = dr.resolve_config(4096, 4096, sm_count=152)
    assert c.threads_per_row * c.blocks_per_thread * 8 == 4096
    for bad in (dr.LaunchConfig(threads_per_row=128, blocks_per_thread=2), dr.LaunchConfig(blocks_per_thread=3),
                dr.LaunchConfig(blocks_per_thread=16)):
        with pytest.raises(dr.DraddError) as e:
            dr.resolve_config(4096, 4096, sm_count=152, config=bad)
        assert e.value.status == 9


def test_split_variant_rules():
    split = dict(variant=dr.VARIANT_SPLIT)
    c = dr.resolve_config(1024, 8192, sm_count=152, config=dr.LaunchConfig(**split))
    assert (c.cluster_ctas, c.threads_per_row, c.blocks_per_thread, c.stages) == (2, 128, 4, 2)
    assert c.grid_ctas % 2 == 0 and c.grid_ctas <= 2 * 1024
    c = dr.resolve_config(3, 8192, sm_count=152, config=dr.LaunchConfig(**split, cluster_ctas=4))
    assert c.grid_ctas == 12 and c.threads_per_row * c.blocks_per_thread * 8 * 4 == 8192
    for bad in (dict(cluster_ctas=3), dict(cluster_ctas=8), dict(grid_ctas=3), dict(rows_per_cta=2),
                dict(threads_per_row=16), dict(threads_per_row=2048), dict(stages=9)):
        with pytest.raises(dr.DraddError) as e:
            dr.resolve_config(1024, 8192, sm_count=152, config=dr.LaunchConfig(**split, **bad))
        assert e.value.status == 9
    # slices narrower than 256 elements, quantised outputs, a cluster size
    # on another variant
    for h, q, cfg in ((256, False, dr.LaunchConfig(**split)), (512, False, dr.LaunchConfig(**split, cluster_ctas=4)),
                      (4096, True, dr.LaunchConfig(**split)),
                      (4096, False, dr.LaunchConfig(variant=dr.VARIANT_STAGED, cluster_ctas=2))):
        with pytest.raises(dr.DraddError) as e:
            dr.resolve_config(64, h, quant=q, sm_count=152, config=cfg)
        assert e.value.status == 9


def test_small_batch_choices():
    """Measured on GB300: small bf16 residual-add batches take wider CTAs."""
    assert dr.resolve_config(64, 4096, sm_count=152).threads_per_row == 256
    assert dr.resolve_config(257, 4096, sm_count=152).threads_per_row == 128
    assert dr.resolve_config(64, 4096, quant=True, sm_count=152).threads_per_row == 128
    assert dr.resolve_config(256, 8192, sm_count=152).threads_per_row == 512
    assert dr.resolve_config(64, 8192, sm_count=152).threads_per_row == 1024
    assert dr.resolve_config(1024, 8192, sm_count=152).threads_per_row == 1024


@pytest.mark.parametrize("n,stages", [(4096, 2), (6144, 2), (6687, 2), (6688, 1), (7296, 1), (12288, 1)])
def test_quantised_residual_add_stages_at_4096(L, n, stages):
    """Residual-add with quantised out at P = 4096: two stages below 44 rows
    per SM (whole rows: 152 SMs x 44 = 6688), else one."""
    for kw in (dict(), dict(fp8=True), dict(fp4=True)):
        c = dr.resolve_config(n, 4096, quant=True, sm_count=152, **kw)
        assert (c.variant, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 128, stages), (n, kw)


def test_threads_at_8192():
    """P = 8192: the bf16 residual-add takes 1024 threads (K = 1; 512 for
    batches of 65..512 rows), the quantised residual-add forms and the plain
    forms 512 (K = 2)."""
    assert dr.resolve_config(4096, 8192, sm_count=152).threads_per_row == 1024
    assert dr.resolve_config(256, 8192, sm_count=152).threads_per_row == 512
    for kw in (dict(), dict(fp8=True), dict(fp4=True)):
        c = dr.resolve_config(4096, 8192, quant=True, sm_count=152, **kw)
        assert (c.variant, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 512, 2), kw


@pytest.mark.parametrize("n,stages", [(2048, 1), (4863, 1), (4864, 3), (8192, 3), (20000, 3)])
def test_quantised_residual_add_at_2048(n, stages):
    """P = 2048, quantised residual-add: staged, 64 threads (K = 4), one
    stage below 32 rows per SM, else three (no longer one warp a row)."""
    for kw in (dict(), dict(fp8=True)):
        c = dr.resolve_config(n, 2048, quant=True, sm_count=152, **kw)
        assert (c.variant, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 64, stages), (n, kw)
    # at P = 1024 the one-warp variant stays
    assert dr.resolve_config(4096, 1024, quant=True, sm_count=152).variant == dr.VARIANT_WARP


def test_plain_quantised_at_512():
    """P = 512, plain quantised: one stage; the pair kernel (64 threads,
    K = 1) below 8192 rows, else one row a CTA (32 threads, K = 2)."""
    for kw in (dict(), dict(fp8=True), dict(fp4=True)):
        c = dr.resolve_config(4096, 512, quant=True, add=False, sm_count=152, **kw)
        assert (c.variant, c.rows_per_cta, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 2, 64, 1), kw
        c = dr.resolve_config(16384, 512, quant=True, add=False, sm_count=152, **kw)
        assert (c.variant, c.rows_per_cta, c.threads_per_row, c.stages) == (dr.VARIANT_STAGED, 1, 32, 1), kw
