"""Seeded synthetic inputs shared by the CUDA path's tests and the oracle's.

This module only draws numbers: it holds none of the method's arithmetic.
Every tensor is made on the CPU with torch's CPU generator, in fp32, scaled
by a standard deviation and shifted by a mean, then narrowed to bf16 by
torch's own round-to-nearest-even cast.  The distributions follow the
ROCm/aiter issue #5151 page ("Steps to Reproduce": randn(...) * std, weight
randn * 0.05 + 1.0, per-step deltas from generators seeded 1000 + step); the
bits do not match the page's, whose numbers came from a GPU generator.

Workloads (n_rows x hidden, distributions as N(mean, std)):

  tiny            64 x 1024   x N(0,1)     residual N(0,1)  weight N(1,0.1)  seed 0
  2048x4096     2048 x 4096   x N(0,1)     residual N(0,4)  weight N(1,0.1)  seed 1
  4096x8192     4096 x 8192   x N(0,1)     residual N(0,4)  weight N(1,0.1)  seed 2
  chain4096     4096 x 4096   residual0 N(0,1) and weight N(1,0.1) from seed 3;
                              x_k N(0,0.05) from seed 1000 + k, k = 0..71
  quant2048x16384 2048 x 16384 x N(0,1)    residual N(0,4)  weight N(1,0.1)  seed 4

Within one workload the draws come from one generator in the order
x, residual, weight.  eps is 1e-6 everywhere.

Fused q/k RMSNorm workloads (QK_WORKLOADS; the page names the kernel but
gives no shapes, so these are the two common layouts and a wider
low-rank one, with the main workloads' distributions): per token, q rows
N(0,1) with a residual N(0,4), k rows N(0,1); both weights N(1,0.1);
draws in the order q, residual, q weight, k, k weight.

  qk_lowrank4096  4096 tokens: q 1 x 1536 (+ residual, e4m3 groups of 128),
                  k 1 x 512                                           seed 5
  qk_heads4096    4096 tokens: q 32 heads x 128, k 8 heads x 128, bf16 out,
                  no residual                                         seed 6
  qk_wide4096     4096 tokens: q 1 x 3072 (+ residual, e4m3 groups of 128),
                  k 1 x 1024                                          seed 8

Log-sum-exp merge and elementwise workloads (ELEM_WORKLOADS; fp32):
softmax log-sum-exps of attention rows are values of about log(S) plus a
score scale, drawn as N(8, 3) for the running lse and the step lse (seed 7);
log1p inputs are uniform in [0, 1) as in the TransformerEngine page's
reproducer (N = 225,280; seed 0), plus a 16M-element case.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

EPS = 1e-6


def normal_bf16(gen: torch.Generator, shape, mean: float, std: float) -> torch.Tensor:
    """N(mean, std) drawn in fp32 on the CPU, cast to bf16."""
    t = torch.randn(shape, generator=gen, dtype=torch.float32)
    return (t * std + mean).to(torch.bfloat16)


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


@dataclass(frozen=True)
class Workload:
    name: str
    n_rows: int
    hidden: int
    x_std: float
    residual_std: float
    seed: int
    weight_mean: float = 1.0
    weight_std: float = 0.1
    eps: float = EPS
    quant: bool = False

    def make(self, n_rows: int | None = None):
        """Return dict(x, residual, weight, eps) as CPU bf16 tensors.

        n_rows < self.n_rows draws the full-size tensors' leading rows
        (same bits as the full workload's first rows); n_rows > self.n_rows
        draws that many rows from the same distributions and seed."""
        g = generator(self.seed)
        rows = self.n_rows if n_rows is None or n_rows <= self.n_rows else n_rows
        x = normal_bf16(g, (rows, self.hidden), 0.0, self.x_std)
        r = normal_bf16(g, (rows, self.hidden), 0.0, self.residual_std)
        w = normal_bf16(g, (self.hidden,), self.weight_mean, self.weight_std)
        if n_rows is not None and n_rows < rows:
            x, r = x[:n_rows].contiguous(), r[:n_rows].contiguous()
        return {"x": x, "residual": r, "weight": w, "eps": self.eps}


WORKLOADS = {
    "tiny": Workload("tiny", 64, 1024, 1.0, 1.0, seed=0),
    "2048x4096": Workload("2048x4096", 2048, 4096, 1.0, 4.0, seed=1),
    # the same distributions and seed over more rows (the launch-boundary fit)
    "8192x4096": Workload("8192x4096", 8192, 4096, 1.0, 4.0, seed=1),
    "16384x4096": Workload("16384x4096", 16384, 4096, 1.0, 4.0, seed=1),
    "4096x8192": Workload("4096x8192", 4096, 8192, 1.0, 4.0, seed=2),
    # the remaining shape of the aiter page's "Cost of fixing" table
    "8192x2048": Workload("8192x2048", 8192, 2048, 1.0, 4.0, seed=1),
    "quant2048x16384": Workload("quant2048x16384", 2048, 16384, 1.0, 4.0, seed=4, quant=True),
}


@dataclass(frozen=True)
class Chain:
    """Chained calls: residual_out of call k is the residual of call k + 1."""
    name: str = "chain4096"
    n_rows: int = 4096
    hidden: int = 4096
    depth: int = 72
    residual0_std: float = 1.0
    x_std: float = 0.05
    seed: int = 3
    delta_seed0: int = 1000
    weight_mean: float = 1.0
    weight_std: float = 0.1
    eps: float = EPS

    def initial(self):
        """(residual_0, weight) as CPU bf16 tensors."""
        g = generator(self.seed)
        r0 = normal_bf16(g, (self.n_rows, self.hidden), 0.0, self.residual0_std)
        w = normal_bf16(g, (self.hidden,), self.weight_mean, self.weight_std)
        return r0, w

    def delta(self, k: int) -> torch.Tensor:
        """x_k for call k, from its own generator seeded delta_seed0 + k."""
        return normal_bf16(generator(self.delta_seed0 + k), (self.n_rows, self.hidden),
                           0.0, self.x_std)


CHAIN4096 = Chain()

# The page's own reproducer settings ("Steps to Reproduce", part 2): m = 256
# rows, hidden 4096, initial state N(0,1) and weight N(1,0.05) from seed 1,
# deltas N(0,0.5) from seeds 1000 + step, 72 calls.
P3_CHAIN = Chain(name="p3chain", n_rows=256, hidden=4096, depth=72, residual0_std=1.0,
                 x_std=0.5, seed=1, delta_seed0=1000, weight_mean=1.0, weight_std=0.05)


def p3_rounding_probe_inputs():
    """The page's part 1: three (m, x std, residual std) settings drawn in order
    from one generator seeded 0, weight N(1, 0.05) each time, hidden 4096."""
    g = generator(0)
    cases = []
    for m, xs, rs in [(512, 1.0, 1.0), (512, 1.0, 30.0), (4096, 3.0, 3.0)]:
        x = normal_bf16(g, (m, 4096), 0.0, xs)
        r = normal_bf16(g, (m, 4096), 0.0, rs)
        w = normal_bf16(g, (4096,), 1.0, 0.05)
        cases.append({"m": m, "x_std": xs, "residual_std": rs, "x": x, "residual": r,
                      "weight": w, "eps": EPS})
    return cases


# Rounding edge patterns as bf16 bit pairs (x, residual).  With x = 1.0
# (0x3F80) and a residual of 2^-8 the fp32 sum has exactly half a bf16 ulp
# below the cut; the four pairs hit: tie with even kept bit, tie with odd
# kept bit, just below half, just above half.
EDGE_PAIRS = [
    (0x3F80, 0x3B80),  # 1.0 + 2^-8           -> 0x3F808000 (tie, even)
    (0x3F81, 0x3B80),  # (1 + 2^-7) + 2^-8    -> 0x3F818000 (tie, odd)
    (0x3F80, 0x3B7F),  # 1.0 + (2^-8 - 2^-16) -> 0x3F807F80 (below half)
    (0x3F80, 0x3B81),  # 1.0 + (2^-8 + 2^-15) -> 0x3F808100 (above half)
]


def edge_rows(n_rows: int = 16, hidden: int = 1024, seed: int = 0):
    """Rows whose elements cycle through EDGE_PAIRS and their negatives.

    Element (i, j) takes pattern (i + j) mod 8; patterns 4..7 are 0..3 with
    both signs flipped.  Weight N(1, 0.1) from `seed`."""
    pats = [(x, r) for x, r in EDGE_PAIRS] + [(x | 0x8000, r | 0x8000) for x, r in EDGE_PAIRS]
    xs = np.array([p[0] for p in pats], dtype=np.uint16)
    rs = np.array([p[1] for p in pats], dtype=np.uint16)
    idx = (np.arange(n_rows)[:, None] + np.arange(hidden)[None, :]) % len(pats)
    x = torch.from_numpy(xs[idx].view(np.int16).copy()).view(torch.bfloat16)
    r = torch.from_numpy(rs[idx].view(np.int16).copy()).view(torch.bfloat16)
    w = normal_bf16(generator(seed), (hidden,), 1.0, 0.1)
    return {"x": x.contiguous(), "residual": r.contiguous(), "weight": w, "eps": EPS}


def bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor -> int16 view of its bits (no arithmetic)."""
    return t.view(torch.int16)


@dataclass(frozen=True)
class QkWorkload:
    """Fused q/k RMSNorm inputs: q is n_tokens * q_heads rows of q_head
    elements, k is n_tokens * k_heads rows of k_head."""
    name: str
    n_tokens: int
    q_heads: int
    q_head: int
    k_heads: int
    k_head: int
    group_size: int
    residual: bool
    seed: int
    residual_std: float = 4.0

    def make(self, n_tokens: int | None = None):
        """dict(q, residual (or None), q_weight, k, k_weight) as CPU bf16
        tensors; n_tokens < self.n_tokens keeps the leading tokens."""
        g = generator(self.seed)
        nq, nk = self.n_tokens * self.q_heads, self.n_tokens * self.k_heads
        q = normal_bf16(g, (nq, self.q_head), 0.0, 1.0)
        r = normal_bf16(g, (nq, self.q_head), 0.0, self.residual_std) if self.residual else None
        qw = normal_bf16(g, (self.q_head,), 1.0, 0.1)
        k = normal_bf16(g, (nk, self.k_head), 0.0, 1.0)
        kw = normal_bf16(g, (self.k_head,), 1.0, 0.1)
        if n_tokens is not None:
            q = q[:n_tokens * self.q_heads].contiguous()
            k = k[:n_tokens * self.k_heads].contiguous()
            r = r[:n_tokens * self.q_heads].contiguous() if r is not None else None
        return {"q": q, "residual": r, "q_weight": qw, "k": k, "k_weight": kw}


QK_WORKLOADS = {
    "qk_lowrank4096": QkWorkload("qk_lowrank4096", 4096, 1, 1536, 1, 512, group_size=128, residual=True, seed=5),
    "qk_heads4096": QkWorkload("qk_heads4096", 4096, 32, 128, 8, 128, group_size=0, residual=False, seed=6),
    # a wider low-rank layout (q rows wider than one warp takes well)
    "qk_wide4096": QkWorkload("qk_wide4096", 4096, 1, 3072, 1, 1024, group_size=128, residual=True, seed=8),
}


def hashed_bf16_rows(rows: torch.Tensor, hidden: int, salt: int) -> torch.Tensor:
    """bf16 bit patterns (as int16) for the given row indices, a fixed hash of
    (row, column, salt) on whatever device `rows` lives on: random sign,
    exponent 2^-4..2^3, 7 random mantissa bits.  Any subset of rows of a
    huge tensor can be rebuilt exactly without materialising the rest, so
    inputs past 2^31 elements can be made on the device and checked on
    sampled rows.  Every intermediate stays below 2^63."""
    cols = torch.arange(hidden, device=rows.device, dtype=torch.int64)
    hsh = (rows.to(torch.int64)[:, None] * 131 + cols[None, :] * 7 + salt * 977) * 739982445
    hsh = hsh & 0xFFFFFFFF
    hsh = hsh ^ (hsh >> 13)
    mant = hsh & 0x7F
    expo = 0x7B + ((hsh >> 7) & 0x7)
    sign = ((hsh >> 10) & 1) << 15
    return (sign | (expo << 7) | mant).to(torch.int16)


@dataclass(frozen=True)
class ElemWorkload:
    """fp32 elementwise workloads: kind "merge" (rows x cols running lse and
    a step lse of rows x step_cols, merged into the last step_cols columns
    of each row, in place) or "log1p" (n values)."""
    name: str
    kind: str
    rows: int
    cols: int
    step_cols: int
    seed: int

    def make(self):
        g = generator(self.seed)
        if self.kind == "log1p":
            return {"x": torch.rand((self.rows * self.cols,), generator=g, dtype=torch.float32)}
        run = torch.randn((self.rows, self.cols), generator=g, dtype=torch.float32) * 3.0 + 8.0
        step = torch.randn((self.rows, self.step_cols), generator=g, dtype=torch.float32) * 3.0 + 8.0
        return {"lse": run, "step": step}


ELEM_WORKLOADS = {
    "lse_merge8x32x32768": ElemWorkload("lse_merge8x32x32768", "merge", 8 * 32, 32768, 32768, seed=7),
    "lse_merge_half8x32x32768": ElemWorkload("lse_merge_half8x32x32768", "merge", 8 * 32, 32768, 16384, seed=7),
    "log1p225280": ElemWorkload("log1p225280", "log1p", 1, 225280, 0, seed=0),
    "log1p16M": ElemWorkload("log1p16M", "log1p", 1, 1 << 24, 0, seed=0),
}
