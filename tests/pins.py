"""Pins of the CPU oracle against things other than itself.

Each pin takes an oracle library object and raises AssertionError if the
oracle disagrees with the page, with mathematics, or with an independent
computation.  They run against the real oracle (tests/test_oracle_*.py) and
against deliberately broken builds of it (tests/test_oracle_mutants.py),
which shows that a plausible slip in the oracle fails at least one of them.

Citations name the ROCm/aiter issue #5151 page ("rmsnorm2d_fwd_with_add
truncates fp32->bf16 on gfx942, ...") and its sections.
"""
from __future__ import annotations

import math
import numpy as np
import torch

import refs
from deterministic_residual_add_gb300 import inputs

TWO = np.float32(2.0)


def f32(v) -> np.float32:
    return np.float32(v)


def bits32(v) -> int:
    return int(np.float32(v).view(np.uint32))


# ------------------------------------------------------------------ RNE
def pin_rne_edge_table(o):
    """Hand-derived table of the four half-ulp cases (and sign mirrors) for
    the three stores: RNE (the page's fix, section "Problem Description"),
    truncation (section "Source", mode 2 = plain shift), ties away."""
    # acc bits, RNE, trunc, ties-away
    table = [
        (0x3F808000, 0x3F80, 0x3F80, 0x3F81),  # exactly half, kept LSB even
        (0x3F818000, 0x3F82, 0x3F81, 0x3F82),  # exactly half, kept LSB odd
        (0x3F807F80, 0x3F80, 0x3F80, 0x3F80),  # just below half
        (0x3F808100, 0x3F81, 0x3F80, 0x3F81),  # above half
        (0x7F7F8000, 0x7F80, 0x7F7F, 0x7F80),  # tie past the largest finite -> inf
        (0x00008000, 0x0000, 0x0000, 0x0001),  # tie between +0 and the smallest subnormal
        (0x007F8000, 0x0080, 0x007F, 0x0080),  # carry from subnormal into the first normal
    ]
    for acc, rne, trunc, away in table:
        for sign in (0, 0x80000000):
            f = np.uint32(acc | sign).view(np.float32)
            s16 = sign >> 16
            assert o.bf16_scalar(f, "rne") == rne | s16, hex(acc | sign)
            assert o.bf16_scalar(f, "trunc") == trunc | s16, hex(acc | sign)
            assert o.bf16_scalar(f, "ties_away") == away | s16, hex(acc | sign)
    # the four input pairs that produce the first four sums
    for (xb, rb), (acc, *_rest) in zip(inputs.EDGE_PAIRS, table[:4]):
        s = f32(o.bf16_to_f32(xb)) + f32(o.bf16_to_f32(rb))
        assert bits32(s) == acc


def pin_rne_vs_torch_sample(o, n_random: int = 1 << 20, seed: int = 0):
    """RNE agrees with torch's CPU cast to bf16 (the page's RNE reference,
    torch.Tensor.to(torch.bfloat16)) on finite values: every high half with a
    set of low halves around the tie, plus random patterns."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    pats = (hi[:, None] | lows[None, :]).ravel()
    rng = np.random.default_rng(seed)
    pats = np.concatenate([pats, rng.integers(0, 1 << 32, size=n_random, dtype=np.uint64)
                           .astype(np.uint32)])
    f = pats.view(np.float32)
    f = f[np.isfinite(f)]
    got = o.bf16_convert(f, "rne")
    exp = refs.u16(torch.from_numpy(f.copy()).to(torch.bfloat16))
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {hex(int(f[bad[0]].view(np.uint32)))}"


# ----------------------------------------------------------- pairwise tree
def pin_tree_worked_examples(o):
    """Hand-evaluated sums that tell the pairwise tree (adjacent pairs,
    lowest index first, zero padding at the end) from other orders."""
    e24, e23, e22 = 2.0 ** -24, 2.0 ** -23, 2.0 ** -22
    # adjacent pairing: (2^-24 + 2^-24) + (1 + 0) = 1 + 2^-23 (exact);
    # pairing by stride would give (2^-24 + 1) + (2^-24 + 0) = 1 + 2^-24 -> 1
    assert o.pairwise_sum(np.array([e24, e24, 1, 0], np.float32)) == f32(1 + e23)
    # sequential would give ((1 + 2^-24) + 2^-24) + 2^-24 = 1 (each add a tie to even)
    assert o.pairwise_sum(np.array([1, e24, e24, e24], np.float32)) == f32(1 + e23)
    # ties to even inside the tree
    assert o.pairwise_sum(np.array([1, e24], np.float32)) == f32(1)
    assert o.pairwise_sum(np.array([1 + e23, e24], np.float32)) == f32(1 + e22)
    # padding goes at the end: [a, b, c] -> (a + b) + (c + 0)
    assert o.pairwise_sum(np.array([e24, e24, 1], np.float32)) == f32(1 + e23)
    # degenerate sizes
    assert o.pairwise_sum(np.array([], np.float32)) == 0
    assert o.pairwise_sum(np.array([3.5], np.float32)) == f32(3.5)


def pin_tree_integer_rows(o, seed: int = 1):
    """On integer data whose partial sums stay below 2^24 every order is
    exact, so the tree must equal the exact integer sum (catches dropped or
    doubled terms for any length)."""
    rng = np.random.default_rng(seed)
    for n in (1, 2, 3, 7, 8, 24, 1000, 4096, 4104, 16384, 32768):
        v = rng.integers(0, max(1, (1 << 24) // n // 2), size=n)
        assert o.pairwise_sum(v.astype(np.float32)) == f32(int(v.sum()))


def pin_tree_error_bound(o, seed: int = 2):
    """|S - sum| <= g_k * sum|v|, k = ceil(log2 n), g_k = k u / (1 - k u),
    u = 2^-24: the pairwise-summation bound (Higham, Accuracy and Stability
    of Numerical Algorithms, sec. 4.2)."""
    rng = np.random.default_rng(seed)
    u = 2.0 ** -24
    for n in (5, 64, 1000, 4096, 32768):
        v = (rng.standard_normal(n) ** 2).astype(np.float32)
        exact = math.fsum(float(t) for t in v)
        k = math.ceil(math.log2(n))
        bound = k * u / (1 - k * u) * float(np.abs(v.astype(np.float64)).sum())
        assert abs(float(o.pairwise_sum(v)) - exact) <= bound


# ------------------------------------------------------------------ rows
def _bits_row(vals):
    return np.array(vals, dtype=np.uint16)


def pin_row_sum_worked_example(o):
    """Row-level tree: x = [1, 2^-12, 2^-12, 2^-12, 0, 0, 0, 0], residual 0.
    Squares [1, 2^-24, 2^-24, 2^-24, 0...]; level 1: 1 + 2^-24 -> 1 (tie to
    even), 2^-24 + 2^-24 = 2^-23; level 2: 1 + 2^-23 (exact); S = 1 + 2^-23.
    A left-to-right sum would give 1."""
    x = _bits_row([0x3F80, 0x3980, 0x3980, 0x3980, 0, 0, 0, 0])[None, :]
    r = np.zeros_like(x)
    w = np.full(8, 0x3F80, np.uint16)
    _, _, ss, _ = o.add_rmsnorm_fwd(x, r, w, 1e-6, return_terms=True)
    assert ss[0] == f32(1 + 2.0 ** -23)


def pin_residual_out_is_torch_cast(o):
    """residual_out is the round-to-nearest-even cast of fp32(x) + fp32(residual):
    bit-exact to torch's (x.float() + residual.float()).to(bfloat16), the
    page's "rne" reference in "Steps to Reproduce"."""
    cases = [inputs.WORKLOADS["tiny"].make(), inputs.edge_rows(16, 1024)]
    for c in cases:
        _, ro = o.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"])
        exp = refs.u16((c["x"].float() + c["residual"].float()).to(torch.bfloat16))
        assert np.array_equal(ro, exp)


def _f64_case(o, x, r, w, eps):
    out, ro = o.add_rmsnorm_fwd(x, r, w, eps)
    y64, acc64 = refs.add_rmsnorm_f64(x, r, w, eps)
    err = np.abs(refs.bf16_value(out) - y64) / refs.ulp_bf16(y64)
    return float(err.max())


def pin_out_within_one_ulp_of_f64(o, seed: int = 5):
    """|out - y64| <= 1 bf16 ulp of the fp64 value of the page's formula,
    over data where eps matters, non-power-of-two rows, tiny and large
    hidden, and non-constant weights."""
    g = inputs.generator(seed)
    cases = []
    t = inputs.WORKLOADS["tiny"].make()
    cases.append((t["x"], t["residual"], t["weight"]))
    for n, h, sx, sr in [(4, 24, 1.0, 1.0), (3, 1000, 1.0, 4.0), (2, 3000, 0.5, 2.0),
                         (2, 4104, 1.0, 1.0), (1, 32768, 1.0, 4.0),
                         (8, 64, 1e-3, 1e-3),     # mean(acc^2) ~ eps: eps visible
                         (8, 64, 3e-4, 0.0)]:     # eps dominates
        x = inputs.normal_bf16(g, (n, h), 0.0, sx)
        r = inputs.normal_bf16(g, (n, h), 0.0, sr) if sr else torch.zeros(n, h, dtype=torch.bfloat16)
        w = inputs.normal_bf16(g, (h,), 1.0, 0.5)
        cases.append((x, r, w))
    for x, r, w in cases:
        assert _f64_case(o, x, r, w, 1e-6) <= 1.0
    # eps = 0.1 on unit data moves the result by ~5%: must still match
    x = inputs.normal_bf16(g, (4, 128), 0.0, 1.0)
    w = inputs.normal_bf16(g, (128,), 1.0, 0.1)
    assert _f64_case(o, x, torch.zeros_like(x), w, 0.1) <= 1.0


def pin_closed_forms(o):
    """Closed forms: cancellation gives zeros; a constant row maps to the
    weight itself; a zero row gives 1/sqrt(eps)."""
    h = 256
    g = inputs.generator(7)
    w = inputs.normal_bf16(g, (h,), 0.0, 1.0)  # both signs
    x = inputs.normal_bf16(g, (3, h), 0.0, 2.0)
    neg = refs.u16(x) ^ np.uint16(0x8000)
    out, ro, ss, inv = o.add_rmsnorm_fwd(x, neg, w, 1e-6, return_terms=True)
    # x + (-x) is +0 in round-to-nearest; +0 * inv * w keeps the sign of w
    assert np.all(ro == 0)
    assert np.array_equal(out, (refs.u16(w) & np.uint16(0x8000))[None, :].repeat(3, 0))
    assert np.all(ss == 0)
    inv_exact = 1.0 / math.sqrt(float(np.float32(1e-6)))
    assert np.all(np.abs(inv.astype(np.float64) - inv_exact) <= inv_exact * 2.0 ** -23)
    # constant rows: acc = a everywhere, so acc * inv = a / sqrt(a^2 + eps),
    # within 1e-6 of sign(a); times w it rounds back to w's own bf16 value
    a_vals = [0x3F80, 0x4040, 0xC0A0, 0x3E00, 0x4B00]  # 1, 3, -5, 0.125, 2^23
    x = np.array([[a] * h for a in a_vals], dtype=np.uint16)
    out, _ = o.add_rmsnorm_fwd(x, np.zeros_like(x), w, 1e-6)
    wb = refs.u16(w)
    for i, a in enumerate(a_vals):
        exp = wb ^ np.uint16(0x8000) if a & 0x8000 else wb
        assert np.array_equal(out[i], exp), i


def pin_rows_independent(o):
    """Each row depends only on itself: permuting rows permutes outputs."""
    c = inputs.WORKLOADS["tiny"].make()
    out, ro = o.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"])
    perm = np.random.default_rng(3).permutation(c["x"].shape[0])
    out2, ro2 = o.add_rmsnorm_fwd(refs.u16(c["x"])[perm].copy(), refs.u16(c["residual"])[perm].copy(),
                                  c["weight"], c["eps"])
    assert np.array_equal(out2, out[perm]) and np.array_equal(ro2, ro[perm])


def pin_rows_exact_rational(o, n_rows: int = 24, seed: int = 11):
    """Bitwise agreement with an exact-rational evaluation of the stated
    readings on small random rows (hidden 8, 16, 24, 40): checks that the
    compiled oracle does every operation as one IEEE round-to-nearest step
    (no contraction, no excess precision, no flush to zero)."""
    rng = np.random.default_rng(seed)
    g = inputs.generator(seed)
    for i in range(n_rows):
        h = (8, 16, 24, 40)[i % 4]
        x = refs.u16(inputs.normal_bf16(g, (1, h), 0.0, 1.0))
        r = refs.u16(inputs.normal_bf16(g, (1, h), 0.0, float(rng.choice([0.01, 1.0, 4.0]))))
        w = refs.u16(inputs.normal_bf16(g, (h,), 1.0, 0.3))
        if i % 6 == 5:  # subnormal-range rows
            x = (x & np.uint16(0x807F)) | np.uint16(0x0100)
            r = r & np.uint16(0x807F)
        out, ro, ss, inv = o.add_rmsnorm_fwd(x, r, w, 1e-6, return_terms=True)
        ex = refs.row_exact(x[0], r[0], w, 1e-6)
        assert list(ro[0]) == ex["ro"], i
        assert ss[0] == ex["S"] and inv[0] == ex["inv"], i
        assert list(out[0]) == ex["out"], i


# Worked examples for the readings that the page's reference() leaves to
# torch: each input was found by search so that the stated reading and the
# alternative give different bf16 outputs; the exact-rational evaluation of
# both readings is recomputed here, and the oracle must match the stated one.
EXAMPLE_MUL_ORDER = (  # (acc * inv) * w  vs  acc * (inv * w), residual 0
    [0x3F1C, 0x3E50, 0x3CE7, 0x3F71, 0x3E4E, 0x3DF2, 0x3E83, 0x3FC8],
    [0x3FF3, 0x3FBF, 0x3FB3, 0x3F34, 0x3F04, 0x3FCD, 0x3F66, 0x3F29])
EXAMPLE_MEAN_DIV = [  # S / hidden  vs  S * (1 / hidden), hidden 24, weight 1
    0x4006, 0x3C1B, 0x3FE9, 0x3C7B, 0x404D, 0x3FF0, 0x3CFF, 0x3EA9, 0x3EEA, 0x3EAD, 0x3D7F,
    0x401E, 0x3DC6, 0x3F9D, 0x400F, 0x3FCC, 0x3D1A, 0x3E51, 0x3D46, 0x3D24, 0x3DEA, 0x3EAA,
    0x3D80, 0x3CA4]
EXAMPLE_RSQRT = [  # 1 / sqrt(v) in two rounded steps  vs  one correctly rounded rsqrt
    0x4003, 0x3D42, 0x403B, 0x3DE2, 0x407C, 0x3EC0, 0x3EA8, 0x4015]
EXAMPLE_QUANT_DIV = [  # q = rint(y / scale)  vs  rint(y * (1 / scale)), weight 1
    0xBFFB, 0x401F, 0x3FC5, 0xBF9F, 0xBD80, 0xBF5C, 0x3F54, 0x3CBE]
EXAMPLE_FP8_DIV = [  # e4m3(y / scale)  vs  e4m3(y * (1 / scale)), plain RMSNorm, weight 1
    0xBCA9, 0xBC7B, 0xBFBB, 0x3FAE, 0x3F09, 0xC028, 0x3EBA, 0x3C74]


def pin_reading_examples(o):
    cases = [
        (EXAMPLE_MUL_ORDER[0], EXAMPLE_MUL_ORDER[1], {"mul_order": "right"}),
        (EXAMPLE_MEAN_DIV, [0x3F80] * len(EXAMPLE_MEAN_DIV), {"mean_op": "recip"}),
        (EXAMPLE_RSQRT, [0x3F80] * len(EXAMPLE_RSQRT), {"inv_op": "rsqrt"}),
    ]
    for xb, wb, alt in cases:
        x = np.array([xb], np.uint16)
        w = np.array(wb, np.uint16)
        stated = refs.row_exact(xb, [0] * len(xb), wb, 1e-6)
        other = refs.row_exact(xb, [0] * len(xb), wb, 1e-6, **alt)
        assert stated["out"] != other["out"], alt  # the example discriminates
        out, _ = o.add_rmsnorm_fwd(x, np.zeros_like(x), w, 1e-6)
        assert list(out[0]) == stated["out"], alt
    xb, wb = EXAMPLE_QUANT_DIV, [0x3F80] * len(EXAMPLE_QUANT_DIV)
    stated = refs.row_exact(xb, [0] * 8, wb, 1e-6, quant=True)
    other = refs.row_exact(xb, [0] * 8, wb, 1e-6, quant=True, quant_op="recip")
    assert stated["q"] != other["q"]
    x = np.array([xb], np.uint16)
    q, scale, _ = o.add_rmsnorm_quant_fwd(x, np.zeros_like(x), np.array(wb, np.uint16), 1e-6)
    assert list(q[0].astype(int)) == stated["q"] and scale[0] == stated["scale"]
    xb = EXAMPLE_FP8_DIV
    stated, sc = refs.e4m3_row_exact(xb, None, [0x3F80] * 8, 1e-6)
    other, _ = refs.e4m3_row_exact(xb, None, [0x3F80] * 8, 1e-6, quant_op="recip")
    assert stated != other
    q, scale = o.rmsnorm_fp8_fwd(np.array([xb], np.uint16), np.full(8, 0x3F80, np.uint16), 1e-6)
    assert list(q[0]) == stated and scale[0] == sc


# ------------------------------------------------------------------ quant
def pin_quant(o, seed: int = 13):
    """int8 variant: |q| <= 127 with 127 reached on every nonzero row,
    |q - q64| <= 1 and |scale / scale64 - 1| <= 2^-20 against fp64, q*scale
    within half a step of y, zero rows give scale 0 and q 0, residual_out
    equal to the bf16 variant's, and bitwise agreement with the exact-
    rational evaluation on small rows."""
    g = inputs.generator(seed)
    for n, h, sr in [(16, 1024, 4.0), (4, 24, 1.0), (2, 16384, 4.0)]:
        x = inputs.normal_bf16(g, (n, h), 0.0, 1.0)
        r = inputs.normal_bf16(g, (n, h), 0.0, sr)
        w = inputs.normal_bf16(g, (h,), 1.0, 0.1)
        q, scale, ro = o.add_rmsnorm_quant_fwd(x, r, w, 1e-6)
        _, ro_b = o.add_rmsnorm_fwd(x, r, w, 1e-6)
        assert np.array_equal(ro, ro_b)
        qa = np.abs(q.astype(np.int64))
        assert qa.max() <= 127 and np.all(qa.max(axis=1) == 127)
        y64, _ = refs.add_rmsnorm_f64(x, r, w, 1e-6)
        q64, s64 = refs.quant_f64(y64)
        assert np.abs(q.astype(np.int64) - q64).max() <= 1
        assert np.all(np.abs(scale.astype(np.float64) / s64 - 1) <= 2.0 ** -20)
        deq = q.astype(np.float64) * scale.astype(np.float64)[:, None]
        assert np.all(np.abs(deq - y64) <= 0.5 * scale.astype(np.float64)[:, None] * (1 + 1e-5)
                      + np.abs(y64) * 2.0 ** -20)
    z = np.zeros((2, 64), np.uint16)
    q, scale, ro = o.add_rmsnorm_quant_fwd(z, z, np.full(64, 0x3F80, np.uint16), 1e-6)
    assert np.all(q == 0) and np.all(scale == 0) and np.all(ro == 0)
    for i in range(8):
        h = (8, 24)[i % 2]
        x = refs.u16(inputs.normal_bf16(g, (1, h), 0.0, 1.0))
        r = refs.u16(inputs.normal_bf16(g, (1, h), 0.0, 2.0))
        w = refs.u16(inputs.normal_bf16(g, (h,), 1.0, 0.3))
        q, scale, ro = o.add_rmsnorm_quant_fwd(x, r, w, 1e-6)
        ex = refs.row_exact(x[0], r[0], w, 1e-6, quant=True)
        assert list(q[0].astype(int)) == ex["q"] and scale[0] == ex["scale"], i


# ------------------------------------------------------- the two halves
def pin_rmsnorm(o, seed: int = 17):
    """Plain RMSNorm (acc = x): within 1 bf16 ulp of fp64; constant rows give
    the weight back; equal to the residual-add form with a zero residual on
    rows without -0 (a special case that reduces to the pinned function);
    and a -0 input keeps its sign (acc = -0, so out = -0 * inv * w), which a
    zero residual would have turned into +0."""
    g = inputs.generator(seed)
    for n, h, sx in [(6, 1024, 1.0), (4, 24, 2.0), (3, 3000, 0.5), (8, 64, 1e-3), (1, 32768, 1.0)]:
        x = inputs.normal_bf16(g, (n, h), 0.0, sx)
        w = inputs.normal_bf16(g, (h,), 1.0, 0.5)
        out = o.rmsnorm_fwd(x, w, 1e-6)
        y64, _ = refs.add_rmsnorm_f64(x, torch.zeros_like(x), w, 1e-6)
        assert float((np.abs(refs.bf16_value(out) - y64) / refs.ulp_bf16(y64)).max()) <= 1.0
        out_add, _ = o.add_rmsnorm_fwd(x, torch.zeros_like(x), w, 1e-6)
        assert np.array_equal(out, out_add)
    h = 256
    w = refs.u16(inputs.normal_bf16(g, (h,), 0.0, 1.0))
    x = np.array([[0x4040] * h, [0xC0A0] * h], np.uint16)  # constant 3 and -5
    out = o.rmsnorm_fwd(x, w, 1e-6)
    assert np.array_equal(out[0], w) and np.array_equal(out[1], w ^ np.uint16(0x8000))
    x = np.zeros((1, h), np.uint16)
    x[0, ::2] = 0x8000                                       # -0 at even positions
    x[0, 1] = 0x3F80                                         # one nonzero keeps inv finite
    out = o.rmsnorm_fwd(x, np.full(h, 0x3F80, np.uint16), 1e-6)
    assert np.all(out[0, 2::2] == 0x8000) and np.all(out[0, 3::2] == 0x0000)
    out_add, _ = o.add_rmsnorm_fwd(x, np.zeros_like(x), np.full(h, 0x3F80, np.uint16), 1e-6)
    assert np.all(out_add[0, 2::2] == 0x0000)                # -0 + +0 = +0 in the add form
    for i in range(6):
        hh = (8, 24, 16)[i % 3]
        xb = refs.u16(inputs.normal_bf16(g, (1, hh), 0.0, 1.0))
        wb = refs.u16(inputs.normal_bf16(g, (hh,), 1.0, 0.3))
        out = o.rmsnorm_fwd(xb, wb, 1e-6)
        assert list(out[0]) == refs.row_exact(xb[0], [0] * hh, wb, 1e-6)["out"], i


def pin_rmsnorm_quant(o, seed: int = 19):
    """Plain RMSNorm, int8 out: the int8 variant's invariants, and equal to the
    residual-add int8 form with a zero residual."""
    g = inputs.generator(seed)
    for n, h in [(8, 1024), (3, 24), (2, 16384)]:
        x = inputs.normal_bf16(g, (n, h), 0.0, 2.0)
        w = inputs.normal_bf16(g, (h,), 1.0, 0.1)
        q, scale = o.rmsnorm_quant_fwd(x, w, 1e-6)
        q2, s2, _ = o.add_rmsnorm_quant_fwd(x, torch.zeros_like(x), w, 1e-6)
        assert np.array_equal(q, q2) and np.array_equal(scale.view(np.uint32), s2.view(np.uint32))
        assert np.all(np.abs(q.astype(np.int64)).max(axis=1) == 127)
        y64, _ = refs.add_rmsnorm_f64(x, torch.zeros_like(x), w, 1e-6)
        q64, _ = refs.quant_f64(y64)
        assert np.abs(q.astype(np.int64) - q64).max() <= 1


def pin_residual_add(o, seed: int = 23):
    """The residual update alone: torch's cast of the fp32 sum, the residual-add
    form's residual_out, and the page's truncation in trunc mode."""
    for c in [inputs.WORKLOADS["tiny"].make(), inputs.edge_rows(16, 1024)]:
        ro = o.residual_add_fwd(c["x"], c["residual"])
        exp = refs.u16((c["x"].float() + c["residual"].float()).to(torch.bfloat16))
        assert np.array_equal(ro, exp)
        _, ro2 = o.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"])
        assert np.array_equal(ro, ro2)
        acc = c["x"].float() + c["residual"].float()
        trunc = refs.u16((acc.view(torch.int32) >> 16).to(torch.int16))
        assert np.array_equal(o.residual_add_fwd(c["x"], c["residual"], "trunc"), trunc)


# ---------------------------------------------------------------- fp8 e4m3
def pin_e4m3_encoder(o, seed: int = 29):
    """The e4m3 encoder: hand-derived codes (ties to the even code, the
    subnormal range, saturation at 448), every finite code decodes and
    re-encodes to itself, and agreement with torch's cast to float8_e4m3fn on
    values clamped to the finite range (torch rounds to nearest even there)."""
    table = [(1.0, 0x38), (448.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E), (-448.0, 0xFE),
             (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (1.5 * 2.0 ** -10, 0x01), (3 * 2.0 ** -10, 0x02),
             (1.0625, 0x38), (1.1875, 0x3A), (432.0, 0x7E), (240.0, 0x77), (-0.0, 0x80),
             (0.0, 0x00), (2.0 ** -6, 0x08), (7 * 2.0 ** -9, 0x07), (15 * 2.0 ** -10, 0x08)]
    for f, code in table:
        assert o.e4m3_scalar(f) == code, (f, hex(code), hex(o.e4m3_scalar(f)))
    for c in list(range(0x7F)) + [c | 0x80 for c in range(0x7F)]:
        v = -0.0 if c == 0x80 else float(refs.e4m3_value(c))
        assert o.e4m3_scalar(v) == c, hex(c)
    rng = np.random.default_rng(seed)
    f = np.concatenate([rng.standard_normal(1 << 18).astype(np.float32) * 50,
                        (rng.standard_normal(1 << 16) * 2.0 ** -8).astype(np.float32),
                        np.array([refs.e4m3_value(c) for c in range(0x7F)], dtype=np.float64).astype(np.float32)
                        * np.float32(1.0625)])
    f = np.clip(f, -448.0, 448.0).astype(np.float32)
    got = o.e4m3_convert(f)
    exp = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, (bad.size, float(f[bad[0]]), hex(got[bad[0]]), hex(exp[bad[0]]))


def pin_fp8_rows(o, seed: int = 31):
    """Per-row e4m3 out: 448 reached on every nonzero row, dequantisation
    within half an e4m3 step of the fp64 value (plus the fp32 path's error),
    equal to the exact-rational evaluation on small rows, zero rows give
    scale 0 and code 0, and the residual form's residual_out is the bf16
    variant's."""
    g = inputs.generator(seed)
    vals = np.array([float(refs.e4m3_value(c)) for c in range(0x7F)] + [float("nan")])
    for n, h, with_res in [(8, 1024, True), (4, 24, False), (2, 16384, True), (6, 3000, False)]:
        x = inputs.normal_bf16(g, (n, h), 0.0, 1.0)
        r = inputs.normal_bf16(g, (n, h), 0.0, 2.0) if with_res else None
        w = inputs.normal_bf16(g, (h,), 1.0, 0.1)
        res = o.rmsnorm_fp8_fwd(x, w, 1e-6, residual=r)
        q, scale = res[0], res[1]
        if with_res:
            _, ro_b = o.add_rmsnorm_fwd(x, r, w, 1e-6)
            assert np.array_equal(res[2], ro_b)
        assert np.all((q & 0x7F).max(axis=1) == 0x7E)
        mag = vals[q & 0x7F] * np.where(q & 0x80, -1.0, 1.0)
        y64, _ = refs.add_rmsnorm_f64(x, r if with_res else torch.zeros_like(x), w, 1e-6)
        deq = mag * scale.astype(np.float64)[:, None]
        # half an e4m3 step at the value's binade (2^-4 relative), or half the
        # subnormal step 2^-10 times the scale
        step = np.maximum(np.abs(mag) * 2.0 ** -4, 2.0 ** -10) * scale.astype(np.float64)[:, None]
        assert np.all(np.abs(deq - y64) <= step + np.abs(y64) * 2.0 ** -20)
    z = np.zeros((2, 64), np.uint16)
    q, scale = o.rmsnorm_fp8_fwd(z, np.full(64, 0x3F80, np.uint16), 1e-6)
    assert np.all(q == 0) and np.all(scale == 0)
    for i in range(6):
        hh = (8, 16)[i % 2]
        xb = refs.u16(inputs.normal_bf16(g, (1, hh), 0.0, 1.0))
        rb = refs.u16(inputs.normal_bf16(g, (1, hh), 0.0, 1.0))
        wb = refs.u16(inputs.normal_bf16(g, (hh,), 1.0, 0.3))
        plain = i % 3 == 0
        res = o.rmsnorm_fp8_fwd(xb, wb, 1e-6, residual=None if plain else rb)
        codes, sc = refs.e4m3_row_exact(xb[0], None if plain else rb[0], wb, 1e-6)
        assert list(res[0][0]) == codes and res[1][0] == sc, i


# ---------------------------------------------------------------- fp4 e2m1
def pin_e2m1_encoder(o):
    """Every interval and every tie of the eight e2m1 magnitudes, by hand:
    ties go to the even code; past 6 saturates; the sign is bit 3."""
    table = [(0.0, 0x0), (0.2, 0x0), (0.25, 0x0), (0.3, 0x1), (0.5, 0x1), (0.75, 0x2), (0.8, 0x2),
             (1.0, 0x2), (1.25, 0x2), (1.3, 0x3), (1.5, 0x3), (1.75, 0x4), (2.0, 0x4), (2.5, 0x4),
             (2.6, 0x5), (3.0, 0x5), (3.5, 0x6), (4.0, 0x6), (5.0, 0x6), (5.1, 0x7), (6.0, 0x7),
             (7.0, 0x7), (1e30, 0x7), (-0.0, 0x8), (-0.75, 0xA), (-6.0, 0xF), (-100.0, 0xF)]
    for f, code in table:
        assert o.e2m1_scalar(f) == code, (f, code, o.e2m1_scalar(f))
    for c in range(16):
        v = float(refs.E2M1[c & 7]) * (-1.0 if c & 8 else 1.0)
        if c == 8:
            v = -0.0
        assert o.e2m1_scalar(v) == c, c
    f = np.linspace(-7, 7, 20001, dtype=np.float32)
    got = o.e2m1_convert(f)
    exp = np.array([refs.e2m1_rne_exact(refs.frac(v), bool(np.float32(v).view(np.uint32) >> 31)) for v in f])
    assert np.array_equal(got, exp)


def pin_fp4_rows(o, seed: int = 37):
    """Per-row e2m1 out: 6 reached on every nonzero row, dequantisation within
    half an e2m1 step of fp64 (plus the fp32 path's error), exact-rational
    rows, zero rows, and residual_out equal to the bf16 variant's."""
    g = inputs.generator(seed)
    mags = np.array([float(v) for v in refs.E2M1])
    for n, h, with_res in [(8, 1024, True), (4, 24, False), (2, 16384, True)]:
        x = inputs.normal_bf16(g, (n, h), 0.0, 1.0)
        r = inputs.normal_bf16(g, (n, h), 0.0, 2.0) if with_res else None
        w = inputs.normal_bf16(g, (h,), 1.0, 0.1)
        res = o.rmsnorm_fp4_fwd(x, w, 1e-6, residual=r)
        codes = refs.unpack_fp4(res[0])
        scale = res[1].astype(np.float64)
        if with_res:
            _, ro_b = o.add_rmsnorm_fwd(x, r, w, 1e-6)
            assert np.array_equal(res[2], ro_b)
        assert np.all((codes & 7).max(axis=1) == 7)
        val = mags[codes & 7] * np.where(codes & 8, -1.0, 1.0) * scale[:, None]
        y64, _ = refs.add_rmsnorm_f64(x, r if with_res else torch.zeros_like(x), w, 1e-6)
        # e2m1 steps are 0.5 up to 2, 1 up to 4 and 2 up to 6: half the step
        # of the interval holding the larger of the value and its code
        m = np.maximum(np.abs(val), np.abs(y64)) / scale[:, None]
        half = np.where(m > 4, 1.0, np.where(m > 2, 0.5, 0.25))
        assert np.all(np.abs(val - y64) <= half * scale[:, None] * (1 + 1e-6) + np.abs(y64) * 2.0 ** -20)
    z = np.zeros((2, 64), np.uint16)
    q, scale = o.rmsnorm_fp4_fwd(z, np.full(64, 0x3F80, np.uint16), 1e-6)
    assert np.all(q == 0) and np.all(scale == 0)
    for i in range(6):
        hh = (8, 16)[i % 2]
        xb = refs.u16(inputs.normal_bf16(g, (1, hh), 0.0, 1.0))
        rb = refs.u16(inputs.normal_bf16(g, (1, hh), 0.0, 1.0))
        wb = refs.u16(inputs.normal_bf16(g, (hh,), 1.0, 0.3))
        plain = i % 3 == 0
        res = o.rmsnorm_fp4_fwd(xb, wb, 1e-6, residual=None if plain else rb)
        codes, sc = refs.fp4_row_exact(xb[0], None if plain else rb[0], wb, 1e-6)
        assert list(refs.unpack_fp4(res[0])[0]) == codes and res[1][0] == sc, i


# ------------------------------------------------------ fused q/k RMSNorm
def pin_qk_rows(o, seed: int = 41):
    """Fused q/k RMSNorm with per-group e4m3 out.  Against the exact-rational
    evaluation on small rows (each group its own scale; k plain bf16 with
    its own weight and eps); 448 reached in every nonzero group; every
    group dequantised within half an e4m3 step of fp64; group size =
    q_hidden gives the per-row e4m3 output, group size 0 the bf16 output of
    the residual-add (or plain) RMSNorm; zero groups give scale 0, code 0;
    either side may be empty."""
    g = inputs.generator(seed)
    vals = np.array([float(refs.e4m3_value(c)) for c in range(0x7F)] + [float("nan")])
    for i, (hq, hk, gs, with_res) in enumerate([(16, 8, 8, True), (32, 16, 8, False), (24, 8, 8, True),
                                                (64, 24, 16, True), (32, 32, 32, False)]):
        qb = refs.u16(inputs.normal_bf16(g, (2, hq), 0.0, 1.0))
        rb = refs.u16(inputs.normal_bf16(g, (2, hq), 0.0, 3.0)) if with_res else None
        qw = refs.u16(inputs.normal_bf16(g, (hq,), 1.0, 0.3))
        kb = refs.u16(inputs.normal_bf16(g, (3, hk), 0.5, 2.0))
        kw = refs.u16(inputs.normal_bf16(g, (hk,), 1.0, 0.3))
        q_eps, k_eps = 1e-6, 0.25
        res = o.qk_rmsnorm_fwd(qb, qw, kb, kw, q_eps, k_eps, group_size=gs, q_residual=rb)
        for r in range(2):
            codes, scales = refs.e4m3_group_exact(qb[r], None if rb is None else rb[r], qw, q_eps, gs)
            assert list(res["q_out"][r]) == codes, (i, r)
            assert [np.float32(s) for s in res["q_scale"][r]] == [np.float32(s) for s in scales], (i, r)
            if with_res:
                ro = refs.row_exact(qb[r], rb[r], qw, q_eps)["ro"]
                assert list(res["q_residual_out"][r]) == ro, (i, r)
        for r in range(3):
            assert list(res["k_out"][r]) == refs.plain_bf16_exact(kb[r], kw, k_eps), (i, r)

    for n, hq, gs, with_res in [(6, 1536, 128, True), (5, 4096, 64, False), (4, 200, 8, True)]:
        q = inputs.normal_bf16(g, (n, hq), 0.0, 1.0)
        r = inputs.normal_bf16(g, (n, hq), 0.0, 2.0) if with_res else None
        qw = inputs.normal_bf16(g, (hq,), 1.0, 0.1)
        k = inputs.normal_bf16(g, (n, 512), 0.0, 1.0)
        kw = inputs.normal_bf16(g, (512,), 1.0, 0.1)
        res = o.qk_rmsnorm_fwd(q, qw, k, kw, 1e-6, 1e-5, group_size=gs, q_residual=r)
        codes = res["q_out"].reshape(n, hq // gs, gs)
        assert np.all((codes & 0x7F).max(axis=2) == 0x7E)
        y64, _ = refs.add_rmsnorm_f64(q, r if with_res else torch.zeros_like(q), qw, 1e-6)
        mag = vals[codes & 0x7F] * np.where(codes & 0x80, -1.0, 1.0)
        sc = res["q_scale"].astype(np.float64)[:, :, None]
        deq = (mag * sc).reshape(n, hq)
        step = (np.maximum(np.abs(mag) * 2.0 ** -4, 2.0 ** -10) * sc).reshape(n, hq)
        assert np.all(np.abs(deq - y64) <= step + np.abs(y64) * 2.0 ** -20)
        whole = o.qk_rmsnorm_fwd(q, qw, k, kw, 1e-6, 1e-5, group_size=hq, q_residual=r)
        per_row = o.rmsnorm_fp8_fwd(q, qw, 1e-6, residual=r)
        assert np.array_equal(whole["q_out"], per_row[0])
        assert np.array_equal(whole["q_scale"][:, 0], per_row[1])
        bf = o.qk_rmsnorm_fwd(q, qw, k, kw, 1e-6, 1e-5, group_size=0, q_residual=r)
        if with_res:
            out, ro = o.add_rmsnorm_fwd(q, r, qw, 1e-6)
            assert np.array_equal(bf["q_residual_out"], ro)
            assert np.array_equal(res["q_residual_out"], ro)
        else:
            out = o.rmsnorm_fwd(q, qw, 1e-6)
        assert np.array_equal(bf["q_out"], out)
        assert np.array_equal(bf["k_out"], o.rmsnorm_fwd(k, kw, 1e-5))
        assert np.array_equal(res["k_out"], bf["k_out"])

    # zero groups inside a nonzero row; an empty side
    q = np.zeros((2, 64), np.uint16)
    q[:, 16:32] = refs.u16(inputs.normal_bf16(g, (2, 16), 0.0, 1.0))
    one = np.full(64, 0x3F80, np.uint16)
    res = o.qk_rmsnorm_fwd(q, one, np.zeros((0, 8), np.uint16), np.full(8, 0x3F80, np.uint16),
                           1e-6, 1e-6, group_size=16)
    assert np.all(res["q_scale"][:, [0, 2, 3]] == 0) and np.all(res["q_scale"][:, 1] > 0)
    assert np.all(res["q_out"][:, :16] == 0) and np.all(res["q_out"][:, 32:] == 0)
    assert res["k_out"].shape == (0, 8)
    res = o.qk_rmsnorm_fwd(np.zeros((0, 64), np.uint16), one, q, one, 1e-6, 1e-6, group_size=16)
    assert res["q_out"].shape == (0, 64) and np.array_equal(res["k_out"], o.rmsnorm_fwd(q, one, 1e-6))


FAST_PINS = [
    pin_rne_edge_table,
    pin_tree_worked_examples,
    pin_tree_integer_rows,
    pin_tree_error_bound,
    pin_row_sum_worked_example,
    pin_residual_out_is_torch_cast,
    pin_out_within_one_ulp_of_f64,
    pin_closed_forms,
    pin_rows_independent,
    pin_rows_exact_rational,
    pin_reading_examples,
    pin_quant,
    pin_rmsnorm,
    pin_rmsnorm_quant,
    pin_residual_add,
    pin_e4m3_encoder,
    pin_fp8_rows,
    pin_e2m1_encoder,
    pin_fp4_rows,
    pin_qk_rows,
]
