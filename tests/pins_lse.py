"""Pins of the log-sum-exp oracle (oracle/lse_oracle.c) to things other than
itself: exact special values, the definition log(e^a + e^b) evaluated with
50-digit decimal arithmetic, and identities of the merge.  Each pin takes
an ``oracle.lse.LseOracle``; the mutation test plants slips in copies of the
C source and requires one of these to fail."""
from __future__ import annotations

import math
from decimal import Decimal, getcontext

import numpy as np

getcontext().prec = 50
INF = float("inf")


def _dec_merge(*vals) -> float:
    """log(sum e^v) of fp32 values, to 50 digits, as a float."""
    finite = [Decimal(float(v)) for v in vals if v != -INF]
    if not finite:
        return -INF
    top = max(finite)
    s = sum(((v - top).exp() for v in finite), Decimal(0))
    return float(top + s.ln())


def pin_special_values(o):
    """Hand-derived values: merge(0, 0) = ln 2, merge(1, 0) = ln(e + 1),
    merge(a, -inf) = a, both -inf gives -inf, +inf wins, NaN propagates, and
    the order of the operands does not matter."""
    assert o.merge1(0.0, 0.0) == math.log(2.0)
    assert abs(o.merge1(1.0, 0.0) - math.log(math.e + 1.0)) <= 4e-16
    assert abs(o.merge1(0.0, 1.0) - math.log(math.e + 1.0)) <= 4e-16
    for a in (-3.5, 0.0, 7.25, 1e30, -1e30):
        assert o.merge1(a, -INF) == np.float32(a) and o.merge1(-INF, a) == np.float32(a)
    assert o.merge1(-INF, -INF) == -INF
    assert o.merge1(INF, 3.0) == INF and o.merge1(-INF, INF) == INF
    nan = float("nan")
    for other in (1.0, INF, -INF, nan):
        assert math.isnan(o.merge1(nan, other)) and math.isnan(o.merge1(other, nan)), other
    # a gap beyond the double exponent range: the smaller term vanishes
    assert o.merge1(1e30, -1e30) == np.float32(1e30)


def pin_definition_decimal(o, seed: int = 1):
    """Random pairs (softmax-lse-like magnitudes, small and huge gaps, equal
    values) against log(e^a + e^b) in 50-digit decimal arithmetic."""
    rng = np.random.default_rng(seed)
    a = np.concatenate([rng.normal(10, 3, 400), rng.normal(0, 50, 200), rng.uniform(-1, 1, 100)]).astype(np.float32)
    b = np.concatenate([a[:400] + rng.normal(0, 1, 400), rng.normal(0, 50, 200), a[600:700]]).astype(np.float32)
    got = o.merge(a, b)
    for x, y, g in zip(a, b, got):
        ref = _dec_merge(x, y)
        assert abs(g - ref) <= 2 ** -50 * max(1.0, abs(ref)), (x, y, g, ref)


def pin_identities(o, seed: int = 2):
    """merge(a, a) = a + ln 2; merge(a + t, b + t) = merge(a, b) + t for an
    exactly representable shift; three-way merges in either grouping equal
    log(e^a + e^b + e^c)."""
    rng = np.random.default_rng(seed)
    a = rng.normal(0, 20, 300).astype(np.float32)
    b = (a + rng.normal(0, 2, 300)).astype(np.float32)
    same = o.merge(a, a)
    assert np.all(np.abs(same - (a.astype(np.float64) + math.log(2.0))) <= 4e-15 * np.maximum(1, np.abs(same)))
    t = np.float32(64.0)
    shifted = o.merge((a + t).astype(np.float32), (b + t).astype(np.float32))
    ok = ((a + t) - t == a) & ((b + t) - t == b)
    assert np.all(np.abs(shifted - (o.merge(a, b) + 64.0))[ok] <= 1e-13)
    c = rng.normal(0, 20, 300).astype(np.float32)
    for x, y, z in list(zip(a, b, c))[:60]:
        ref = _dec_merge(x, y, z)
        ab = o.merge1(x, y)
        # merging through an fp32 intermediate rounds it once
        left = o.merge1(np.float32(ab), z)
        assert abs(left - ref) <= 2 ** -23 * max(1.0, abs(ab)) + 1e-15 * max(1.0, abs(ref))


def pin_merge_2d(o, seed: int = 3):
    """The row-strided form equals the flat form on the gathered rows; the
    second half of each row merged with a half-width step tensor."""
    rng = np.random.default_rng(seed)
    rows, S = 7, 24
    lse = rng.normal(5, 2, rows * S).astype(np.float32)
    step = rng.normal(5, 2, rows * (S // 2)).astype(np.float32)
    got = o.merge_2d(lse[S // 2:], S, step, S // 2, rows, S // 2)
    ref = o.merge(lse.reshape(rows, S)[:, S // 2:].copy(), step.reshape(rows, S // 2))
    assert np.array_equal(got, ref)
    assert got.shape == (rows, S // 2)


def pin_unary(o, seed: int = 4):
    """log1p, cosh and exp against 50-digit decimal evaluations of
    ln(1 + x), (e^x + e^-x) / 2 and e^x; the page's log1p inputs are uniform
    in [0, 1)."""
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.uniform(0, 1, 300), rng.uniform(-0.999, 5, 100), [0.0, -0.5, 1e-30, 3e-8]])
    x = x.astype(np.float32)
    got = o.unary(x, "log1p")
    for v, g in zip(x, got):
        ref = float((Decimal(1) + Decimal(float(v))).ln())
        assert abs(g - ref) <= 2.5e-16 * max(abs(ref), 1e-300), (v, g, ref)
    y = np.concatenate([rng.uniform(-10, 10, 300), [0.0, 88.0, -88.0]]).astype(np.float32)
    gc, ge = o.unary(y, "cosh"), o.unary(y, "exp")
    for v, c, e in zip(y, gc, ge):
        d = Decimal(float(v))
        assert abs(c - float((d.exp() + (-d).exp()) / 2)) <= 4.5e-16 * c
        assert abs(e - float(d.exp())) <= 2.5e-16 * e


LSE_PINS = [pin_special_values, pin_definition_decimal, pin_identities, pin_merge_2d, pin_unary]
