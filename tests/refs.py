"""Independent references for the tests: fp64 closed forms, exact rational
rounding, ULP helpers and the page's bias metric.

None of this is the oracle; it exists to pin the oracle (and, through it,
the CUDA path) to something other than itself.
"""
from __future__ import annotations

import math
from fractions import Fraction
from pathlib import Path

import numpy as np
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


def load_golden(name: str) -> dict:
    vals = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        vals[k] = float(v)
    return vals


# ---------------------------------------------------------------- bit views
def u16(t) -> np.ndarray:
    """bf16 tensor / uint16-compatible array -> numpy uint16 bit patterns."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        return t.numpy().view(np.uint16)
    a = np.asarray(t)
    return a.view(np.uint16) if a.dtype == np.int16 else a.astype(np.uint16, copy=False)


def bf16_value(b) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    b = u16(b)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_bits(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float32).view(np.uint32)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values around |v|: 2^(floor(log2|v|) - 7), never below
    the subnormal spacing 2^-133."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    u = np.exp2(e - 7)
    return np.where(a > 0, np.maximum(u, 2.0 ** -133), 2.0 ** -133)


# ------------------------------------------------------- fp64 closed forms
def add_rmsnorm_f64(x, residual, weight, eps: float):
    """The page's reference() evaluated in fp64 with no intermediate rounding
    except eps, taken as the fp32 value the kernels receive."""
    acc = bf16_value(x) + bf16_value(residual)
    var = np.mean(acc * acc, axis=-1, keepdims=True)
    inv = 1.0 / np.sqrt(var + float(np.float32(eps)))
    y = acc * inv * bf16_value(weight)
    return y, acc


def quant_f64(y64: np.ndarray):
    amax = np.max(np.abs(y64), axis=-1)
    scale = amax / 127.0
    safe = np.where(scale > 0, scale, 1.0)
    q = np.clip(np.rint(y64 / safe[..., None]), -127, 127)
    q = np.where(scale[..., None] > 0, q, 0)
    return q.astype(np.int64), scale


# ------------------------------------------------ exact rational rounding
def rn32(q: Fraction) -> np.float32:
    """Round a rational to the nearest fp32 value, ties to even, with
    subnormals and overflow to infinity (IEEE 754 binary32)."""
    if q == 0:
        return np.float32(0.0)
    neg = q < 0
    a = -q if neg else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum_exp = max(e, -126) - 23
    scaled = a / (Fraction(2) ** quantum_exp)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    val = Fraction(m) * Fraction(2) ** quantum_exp
    if val >= Fraction(2) ** 128:
        r = np.float32(np.inf)
    else:
        r = np.float32(float(val))  # exact: val is an fp32 value
        assert Fraction(float(r)) == val
    return np.float32(-r) if neg else r


def frac(v) -> Fraction:
    return Fraction(float(v))


def sqrt_rn32(v) -> np.float32:
    """Correctly rounded fp32 square root of a non-negative rational (or fp32
    value), computed with integer square roots (no floating point)."""
    q = v if isinstance(v, Fraction) else frac(v)
    assert q >= 0
    if q == 0:
        return np.float32(0.0)
    k = 400
    num = q.numerator << (2 * k)
    s = math.isqrt(num // q.denominator)
    # sqrt(q) lies in [s, s+1) / 2^k.  The square root of a binary32 value is
    # never a midpoint between two binary32 values, and 2^-400 resolution is
    # far below half an ulp of any binary32 result.
    lo = rn32(Fraction(s, 1 << k))
    hi = rn32(Fraction(s + 1, 1 << k))
    assert lo == hi, "sqrt too close to a rounding boundary for this resolution"
    return lo


def rne_bf16_exact(v: np.float32) -> int:
    """Nearest bf16 to an fp32 value, ties to even, decided with rationals."""
    f = frac(v)
    if f == 0:
        return int(np.float32(v).view(np.uint32)) >> 16
    neg = f < 0
    a = -f if neg else f
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum_exp = max(e, -126) - 7
    scaled = a / (Fraction(2) ** quantum_exp)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    val = Fraction(m) * Fraction(2) ** quantum_exp
    if val >= Fraction(2) ** 128:
        bits = 0x7F80
    else:
        bits = int(np.float32(float(val)).view(np.uint32)) >> 16
    return bits | (0x8000 if neg else 0)


def row_exact(x_bits, r_bits, w_bits, eps: float, *, mul_order: str = "left",
              mean_op: str = "div", inv_op: str = "recip_of_sqrt", quant: bool = False,
              quant_op: str = "div"):
    """One row of the method with every operation rounded by rn32.

    Defaults are the readings the oracle states: pairwise tree over the
    zero-padded row, mean = S / hidden, inv = 1 / sqrt(mean + eps) with both
    operations rounded, y = (acc * inv) * w.  The keyword options evaluate
    the alternative readings (mul_order="right": acc * (inv * w);
    mean_op="recip": S * (1 / hidden); inv_op="rsqrt": 1/sqrt rounded once;
    quant_op="recip": y * (1 / scale))
    so a test can show an input tells the readings apart.

    Returns dict(ro, out, y, S, inv) and, with quant, also q and scale."""
    xs = [frac(bf16_value(np.uint16(b))) for b in x_bits]
    rs = [frac(bf16_value(np.uint16(b))) for b in r_bits]
    ws = [frac(bf16_value(np.uint16(b))) for b in w_bits]
    h = len(xs)
    acc = [rn32(a + b) for a, b in zip(xs, rs)]
    sq = [rn32(frac(a) * frac(a)) for a in acc]
    p = 1
    while p < h:
        p *= 2
    level = [frac(s) for s in sq] + [Fraction(0)] * (p - h)
    while len(level) > 1:
        level = [frac(rn32(level[i] + level[i + 1])) for i in range(0, len(level), 2)]
    S = rn32(level[0])
    if mean_op == "div":
        mean = rn32(frac(S) / h)
    else:
        mean = rn32(frac(S) * frac(rn32(Fraction(1, h))))
    v = rn32(frac(mean) + frac(np.float32(eps)))
    if inv_op == "recip_of_sqrt":
        inv = rn32(Fraction(1) / frac(sqrt_rn32(v)))
    else:
        inv = sqrt_rn32(Fraction(1) / frac(v))
    if mul_order == "left":
        ys = [rn32(frac(rn32(frac(a) * frac(inv))) * w) for a, w in zip(acc, ws)]
    else:
        ys = [rn32(frac(a) * frac(rn32(frac(inv) * w))) for a, w in zip(acc, ws)]
    res = {"ro": [rne_bf16_exact(a) for a in acc], "out": [rne_bf16_exact(y) for y in ys],
           "y": ys, "S": S, "inv": inv}
    if quant:
        amax = max((abs(frac(y)) for y in ys), default=Fraction(0))
        scale = rn32(amax / 127)
        qs = []
        for y in ys:
            if scale == 0:
                qs.append(0)
                continue
            if quant_op == "div":
                t = frac(rn32(frac(y) / frac(scale)))
            else:
                t = frac(rn32(frac(y) * frac(rn32(Fraction(1) / frac(scale)))))
            n = math.floor(t)
            rem = t - n
            if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
                n += 1
            qs.append(max(-127, min(127, n)))
        res["q"], res["scale"] = qs, scale
    return res


# ---------------------------------------------------------------- e4m3
def e4m3_value(code: int) -> Fraction:
    """Exact value of an e4m3 (e4m3fn) code; NaN codes are not accepted."""
    sign = -1 if code & 0x80 else 1
    e, m = (code >> 3) & 0xF, code & 7
    assert not (e == 15 and m == 7), "NaN"
    mag = Fraction(m, 8) * Fraction(1, 2 ** 6) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return sign * mag


def e4m3_rne_exact(q: Fraction) -> int:
    """Nearest e4m3 code to a rational, ties to the even code, saturating at
    448; the sign of zero follows the sign of q."""
    neg = q < 0
    a = -q if neg else q
    if a >= 448:
        return 0x7E | (0x80 if neg else 0)
    best = min(range(0x7F), key=lambda c: (abs(e4m3_value(c) - a), c & 1))
    return best | (0x80 if neg else 0)


def e4m3_row_exact(x_bits, r_bits, w_bits, eps: float, quant_op: str = "div"):
    """Exact-rational e4m3 quantisation of one row (residual None: plain):
    scale = RN32(amax / 448), q = e4m3 of RN32(y / scale) (quant_op="recip":
    of RN32(y * RN32(1 / scale)), the alternative reading)."""
    xs = list(x_bits)
    rs = list(r_bits) if r_bits is not None else [0] * len(xs)
    ys = row_exact(xs, rs, w_bits, eps)["y"] if r_bits is not None else _plain_row_y(xs, w_bits, eps)
    return _e4m3_codes(ys, quant_op)


def e4m3_group_exact(x_bits, r_bits, w_bits, eps: float, group: int):
    """Exact-rational per-group e4m3 quantisation of one row: y as in
    e4m3_row_exact, then every run of `group` consecutive elements gets its
    own scale = RN32(amax / 448) over that run.  Returns (codes, scales)."""
    xs = list(x_bits)
    rs = list(r_bits) if r_bits is not None else [0] * len(xs)
    ys = row_exact(xs, rs, w_bits, eps)["y"] if r_bits is not None else _plain_row_y(xs, w_bits, eps)
    codes, scales = [], []
    for lo in range(0, len(ys), group):
        c, s = _e4m3_codes(ys[lo:lo + group], "div")
        codes += c
        scales.append(s)
    return codes, scales


def plain_bf16_exact(x_bits, w_bits, eps: float):
    """bf16 bit patterns of plain RMSNorm of one row by exact rational steps."""
    return [rne_bf16_exact(y) for y in _plain_row_y(list(x_bits), w_bits, eps)]


def _e4m3_codes(ys, quant_op):
    amax = max((abs(frac(y)) for y in ys), default=Fraction(0))
    scale = rn32(amax / 448)
    if scale == 0:
        return [0] * len(ys), scale
    codes = []
    for y in ys:
        if quant_op == "div":
            t = rn32(frac(y) / frac(scale))
        else:
            t = rn32(frac(y) * frac(rn32(Fraction(1) / frac(scale))))
        c = e4m3_rne_exact(frac(t))
        if frac(t) == 0 and np.float32(t).view(np.uint32) >> 31:
            c |= 0x80
        codes.append(c)
    return codes, scale


E2M1 = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
        Fraction(4), Fraction(6)]


def e2m1_rne_exact(q: Fraction, negative_zero: bool = False) -> int:
    """Nearest e2m1 code to a rational, ties to the even code, saturating at
    6; bit 3 is the sign."""
    neg = q < 0 or (q == 0 and negative_zero)
    a = abs(q)
    code = 7 if a >= 6 else min(range(8), key=lambda c: (abs(E2M1[c] - a), c & 1))
    return code | (8 if neg else 0)


def fp4_row_exact(x_bits, r_bits, w_bits, eps: float):
    """Exact-rational e2m1 codes (one per element, unpacked) and scale of one
    row: scale = RN32(amax / 6), code = e2m1 of RN32(y / scale)."""
    xs = list(x_bits)
    ys = row_exact(xs, list(r_bits), w_bits, eps)["y"] if r_bits is not None else _plain_row_y(xs, w_bits, eps)
    amax = max((abs(frac(y)) for y in ys), default=Fraction(0))
    scale = rn32(amax / 6)
    if scale == 0:
        return [0] * len(ys), scale
    codes = []
    for y in ys:
        t = rn32(frac(y) / frac(scale))
        codes.append(e2m1_rne_exact(frac(t), bool(np.float32(t).view(np.uint32) >> 31)))
    return codes, scale


def unpack_fp4(q: np.ndarray) -> np.ndarray:
    """[..., h/2] bytes -> [..., h] codes (even element in the low nibble)."""
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def _plain_row_y(x_bits, w_bits, eps):
    """fp32 y of plain RMSNorm (acc = x exactly) by exact rational steps."""
    acc = [np.float32(bf16_value(np.uint16(b))) for b in x_bits]
    h = len(acc)
    sq = [rn32(frac(a) * frac(a)) for a in acc]
    p = 1
    while p < h:
        p *= 2
    level = [frac(s) for s in sq] + [Fraction(0)] * (p - h)
    while len(level) > 1:
        level = [frac(rn32(level[i] + level[i + 1])) for i in range(0, len(level), 2)]
    S = rn32(level[0])
    v = rn32(frac(rn32(frac(S) / h)) + frac(np.float32(eps)))
    inv = rn32(Fraction(1) / frac(sqrt_rn32(v)))
    ws = [frac(bf16_value(np.uint16(b))) for b in w_bits]
    return [rn32(frac(rn32(frac(a) * frac(inv))) * w) for a, w in zip(acc, ws)]


# ------------------------------------------------------------- metrics
def magnitude_bias(got_bits, exp_bits) -> float:
    """The page's magnitude_bias(): mean over e != 0 of (|g| - |e|) / |e|;
    negative means shrunk toward zero."""
    g, e = bf16_value(got_bits), bf16_value(exp_bits)
    nz = e != 0
    return float(((np.abs(g[nz]) - np.abs(e[nz])) / np.abs(e[nz])).mean())


def magnitude_bias_values(got_bits, exp_values: np.ndarray) -> float:
    """Same metric against real-valued expectations (e.g. fp64 or fp32 acc)."""
    g = bf16_value(got_bits)
    e = np.asarray(exp_values, dtype=np.float64)
    nz = e != 0
    return float(((np.abs(g[nz]) - np.abs(e[nz])) / np.abs(e[nz])).mean())


def rms(v: np.ndarray) -> float:
    v = np.asarray(v, dtype=np.float64)
    return float(np.sqrt(np.mean(v * v)))


def cos_sim(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / math.sqrt((a @ a) * (b @ b)))
