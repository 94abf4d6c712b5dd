"""Log-sum-exp merge and launch-invariant unary functions on the GPU,
through the C ABI, against the double-precision oracle: within
ulp(result) + 2^-22 for the merge (the bound the merge's arithmetic gives:
expf's error scaled by at most 1/2, the series log1p's 2.95 x 2^-24
relative of a value below ln 2, the rounding of lo - hi, and the final
rounding) and within the CUDA math library's documented ulp bounds for the
unary functions (coshf: its measured maximum, below 3 ulp); special
values exactly; and one result, bit for bit, under
every launch configuration (the page's reproducer: log1p of 225,280 uniform
values under many configurations gives a single result group here)."""
import numpy as np
import pytest
import torch

import oracle.lse as lse_oracle
import deterministic_residual_add_gb300 as dr
from gpu_util import dev

pytestmark = pytest.mark.gpu

INF = float("inf")


def ulp32(v: np.ndarray) -> np.ndarray:
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 23)


@pytest.fixture(scope="module")
def lo():
    return lse_oracle.lib()


def lse_pairs(n, seed):
    rng = np.random.default_rng(seed)
    a = rng.normal(8.0, 3.0, n).astype(np.float32)
    kind = rng.integers(0, 6, n)
    b = np.where(kind == 0, a + rng.normal(0, 1, n),
        np.where(kind == 1, a,
        np.where(kind == 2, a - rng.exponential(20, n),
        np.where(kind == 3, rng.normal(-5, 40, n),
        np.where(kind == 4, a + rng.normal(0, 1e-5, n), rng.normal(0, 1, n)))))).astype(np.float32)
    return a, b


def check_merge(got: np.ndarray, a: np.ndarray, b: np.ndarray, lo):
    ref = lo.merge(a, b).ravel()
    got = got.ravel().astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])
    err = np.abs(got[fin] - ref[fin])
    bound = ulp32(ref[fin]) + 2.0 ** -22
    bad = np.flatnonzero(err > bound)
    assert bad.size == 0, (a.ravel()[fin][bad[:3]], b.ravel()[fin][bad[:3]], got[fin][bad[:3]], ref[fin][bad[:3]])
    return float((err / ulp32(ref[fin])).max()) if err.size else 0.0


@pytest.mark.parametrize("n", [1, 7, 1000, 225280, 1 << 22])
def test_merge_parity(lo, n):
    a, b = lse_pairs(n, n)
    d = dev()
    out = dr.lse_merge_fwd(torch.from_numpy(a).to(d), torch.from_numpy(b).to(d))
    torch.cuda.synchronize()
    check_merge(out.cpu().numpy(), a, b, lo)


def test_merge_special_values(lo):
    nan = float("nan")
    vals = [0.0, -0.0, 1.0, -1.0, 88.0, -88.0, 1e30, -1e30, 3e38, -3e38, 1e-40, INF, -INF, nan, 0.6931472]
    a = np.array([x for x in vals for _ in vals], np.float32)
    b = np.array([y for _ in vals for y in vals], np.float32)
    d = dev()
    out = dr.lse_merge_fwd(torch.from_numpy(a).to(d), torch.from_numpy(b).to(d)).cpu().numpy()
    check_merge(out, a, b, lo)
    assert out[(a == -INF) & (b == -INF)].tolist() == [-INF]


CONFIGS = [None] + [dr.LaunchConfig(threads_per_row=T, blocks_per_thread=V, grid_ctas=G)
                    for T in (32, 128, 256, 1024) for V in (1, 2, 4, 8) for G in (0, 1, 7)] + \
          [dr.LaunchConfig(serialize=1)]


def test_merge_launch_invariance(lo):
    a, b = lse_pairs(100003, 5)
    d = dev()
    ta, tb = torch.from_numpy(a).to(d), torch.from_numpy(b).to(d)
    digests = set()
    for cfg in CONFIGS:
        out = dr.lse_merge_fwd(ta, tb, config=cfg)
        torch.cuda.synchronize()
        digests.add(out.cpu().numpy().tobytes())
    assert len(digests) == 1
    check_merge(np.frombuffer(digests.pop(), np.float32), a, b, lo)


def test_merge_every_difference(lo):
    """merge(0, d) for every fp32 d in [-104, 0] (below -104, e^d is under
    2^-150 and the correction is 0): the exp, the division and the series on
    every argument they can meet with the larger operand 0, where the final
    addition is exact.  The bound there is 2^-22 absolute: the series'
    2.95 x 2^-24 relative of a value below ln 2, plus the exp's error
    (at most 2 + floor(1.173 |d|) ulp of u = e^d) scaled by 1 / (1 + u)."""
    from concurrent.futures import ThreadPoolExecutor
    first, last = 0x80000000, 0xC2D00000
    chunk = 1 << 26
    d = dev()
    worst = 0.0
    with ThreadPoolExecutor(8) as ex:
        for c0 in range(first, last + 1, chunk):
            c1 = min(last + 1, c0 + chunk)
            bits = np.arange(c0, c1, dtype=np.uint64).astype(np.uint32)
            x = bits.view(np.float32)
            zeros = np.zeros_like(x)
            got = dr.lse_merge_fwd(torch.zeros(x.size, device=d), torch.from_numpy(x).to(d)).cpu().numpy()
            parts = np.array_split(np.arange(x.size), 8)
            ref = np.concatenate(list(ex.map(lambda ix: lo.merge(zeros[ix], x[ix]), parts)))
            err = np.abs(got.astype(np.float64) - ref)
            bad = np.flatnonzero(err > 2.0 ** -22)
            assert bad.size == 0, (x[bad[:3]], got[bad[:3]], ref[bad[:3]])
            worst = max(worst, float(err.max()))
    assert worst > 0.0


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_merge_alignment_invariance(lo, offset):
    """Views that start off a 16-byte boundary, or whose row stride is not
    a multiple of 4 elements, take the element-at-a-time path; the bits
    equal those of the aligned (16-byte vector) path on the same values."""
    rows, cols, stride = 33, 3000, 3001 + offset
    a, b = lse_pairs(rows * cols, 40 + offset)
    a, b = a.reshape(rows, cols), b.reshape(rows, cols)
    d = dev()
    ref = dr.lse_merge_fwd(torch.from_numpy(a).to(d), torch.from_numpy(b).to(d)).cpu().numpy()
    flat_a = torch.zeros(offset + rows * stride, device=d)
    flat_b = torch.zeros(offset + rows * stride, device=d)
    va = flat_a[offset:].view(rows, stride)[:, :cols]
    vb = flat_b[offset:].view(rows, stride)[:, :cols]
    va.copy_(torch.from_numpy(a))
    vb.copy_(torch.from_numpy(b))
    got = dr.lse_merge_fwd(va, vb).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    out = torch.zeros(offset + rows * stride, device=d)[offset:].view(rows, stride)[:, :cols]
    dr.lse_merge_fwd(torch.from_numpy(a).to(d), torch.from_numpy(b).to(d), out=out)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    check_merge(ref, a, b, lo)


def test_second_half_in_place(lo):
    """A running [rows x S] lse merged, in place, with a [rows x S/2] step
    lse on the second half of each row; the first half is untouched."""
    rows, S = 96, 4096
    rng = np.random.default_rng(9)
    run = rng.normal(8, 3, (rows, S)).astype(np.float32)
    step = rng.normal(8, 3, (rows, S // 2)).astype(np.float32)
    d = dev()
    t = torch.from_numpy(run).to(d)
    half = t[:, S // 2:]
    dr.lse_merge_fwd(half, torch.from_numpy(step).to(d), out=half)
    torch.cuda.synchronize()
    got = t.cpu().numpy()
    assert np.array_equal(got[:, :S // 2], run[:, :S // 2])
    check_merge(got[:, S // 2:], run[:, S // 2:], step, lo)
    ref2d = lo.merge_2d(run.ravel()[S // 2:], S, step.ravel(), S // 2, rows, S // 2)
    assert np.array_equal(ref2d, lo.merge(run[:, S // 2:], step))


def test_flat_in_place(lo):
    a, b = lse_pairs(5000, 11)
    d = dev()
    ta = torch.from_numpy(a).to(d)
    dr.lse_merge_fwd(ta, torch.from_numpy(b).to(d), out=ta)
    torch.cuda.synchronize()
    check_merge(ta.cpu().numpy(), a, b, lo)


# log1pf and expf are held to the bounds CUDA documents (1 and 2 ulp);
# coshf measured up to 2.27 ulp on these inputs (at x = -8.956692), so it
# is held to 3.
UNARY_BOUND_ULP = {"log1p": 1.0, "cosh": 3.0, "exp": 2.0}


@pytest.mark.parametrize("op", ["log1p", "cosh", "exp"])
def test_unary_bounds_and_invariance(lo, op):
    rng = np.random.default_rng(2)
    if op == "log1p":
        x = rng.random(225280, dtype=np.float32)  # the page's reproducer inputs
        x = np.concatenate([x, rng.uniform(-0.999, 100, 20000).astype(np.float32),
                            np.array([0, -0.0, 1e-30, -0.5, 3e38], np.float32)])
    else:
        x = np.concatenate([rng.uniform(-10, 10, 200000), rng.uniform(-88, 88, 20000), [0, 1e-20]]).astype(np.float32)
    d = dev()
    tx = torch.from_numpy(x).to(d)
    digests = set()
    for cfg in CONFIGS:
        out = dr.invariant_unary_fwd(tx, op, config=cfg)
        torch.cuda.synchronize()
        digests.add(out.cpu().numpy().tobytes())
    assert len(digests) == 1
    got = np.frombuffer(digests.pop(), np.float32).astype(np.float64)
    ref = lo.unary(x, op)
    # ulps of the larger magnitude's binade (a result that rounds up to a
    # power of two is measured in that binade's units)
    err_ulp = np.abs(got - ref) / ulp32(np.maximum(np.abs(ref), np.abs(got)))
    worst = int(np.argmax(err_ulp))
    assert err_ulp.max() <= UNARY_BOUND_ULP[op], (op, err_ulp.max(), x[worst], got[worst], ref[worst])


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unary_alignment_invariance(offset):
    x = np.random.default_rng(offset).uniform(-0.9, 50, 100003).astype(np.float32)
    d = dev()
    ref = dr.invariant_unary_fwd(torch.from_numpy(x).to(d), "log1p").cpu().numpy()
    buf = torch.zeros(offset + x.size, device=d)
    view = buf[offset:]
    view.copy_(torch.from_numpy(x))
    got = dr.invariant_unary_fwd(view, "log1p").cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_unary_in_place(lo):
    x = np.linspace(-3, 3, 4097, dtype=np.float32)
    d = dev()
    t = torch.from_numpy(x).to(d)
    ref = dr.invariant_unary_fwd(t.clone(), "cosh")
    dr.invariant_unary_fwd(t, "cosh", out=t)
    torch.cuda.synchronize()
    assert torch.equal(t, ref)
