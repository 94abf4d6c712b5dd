"""Negative controls: the oracle's truncating store reproduces the one-sided
bias and the residual shrink printed on the ROCm/aiter issue #5151 page
("Steps to Reproduce" output block; golden file tests/golden/
p3_reproducer_output.txt), while round-to-nearest-even shows none.

The page's numbers came from a GPU random generator; these runs use torch's
CPU generator with the same seeds and distributions, so the comparisons are
statistical, with tolerances far below the effect sizes."""
import numpy as np
import pytest
import torch

import oracle
import refs
from deterministic_residual_add_gb300 import inputs

GOLD = refs.load_golden("p3_reproducer_output.txt")
THREADS = oracle.default_threads()


def page_truncate(x, r):
    """The page's bf16_truncate() applied to fp32(x) + fp32(residual), in torch."""
    acc = x.float() + r.float()
    return refs.u16((acc.view(torch.int32) >> 16).to(torch.int16))


def test_rounding_probe_matches_page(orc):
    for c in inputs.p3_rounding_probe_inputs():
        _, ro_t = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"], "trunc",
                                      threads=THREADS)
        _, ro_r = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"], "rne",
                                      threads=THREADS)
        torch_rne = refs.u16((c["x"].float() + c["residual"].float()).to(torch.bfloat16))
        assert np.array_equal(ro_t, page_truncate(c["x"], c["residual"]))  # trunc_bitexact=True
        assert np.array_equal(ro_r, torch_rne)                              # rne_bitexact=True
        assert refs.magnitude_bias(ro_r, torch_rne) == GOLD["rne.bias"]
        key = f"probe.{c['m']}.{c['x_std']:g}.{c['residual_std']:g}.bias"
        bias = refs.magnitude_bias(ro_t, torch_rne)
        assert bias < 0
        assert abs(bias / GOLD[key] - 1) < 0.01, (key, bias)
        pct = round(100 * float((ro_t != torch_rne).mean()))
        assert GOLD["probe.differ_percent_min"] <= pct <= GOLD["probe.differ_percent_max"]


def torch_reference(x, r, w, eps):
    """The page's reference() with the round-to-nearest-even cast, on the CPU."""
    acc = x.float() + r.float()
    var = acc.pow(2).mean(-1, keepdim=True)
    return ((acc * torch.rsqrt(var + eps)) * w.float()).to(torch.bfloat16), acc.to(torch.bfloat16)


@pytest.mark.slow
def test_chain_shrink_matches_page(orc):
    ch = inputs.P3_CHAIN
    h0, w = ch.initial()
    res_t = refs.u16(h0).copy()
    res_r = res_t.copy()
    res_ref = h0.clone()
    for step in range(ch.depth):
        d = ch.delta(step)
        out_t, res_t = orc.add_rmsnorm_fwd(d, res_t, w, ch.eps, "trunc", threads=THREADS)
        out_r, res_r = orc.add_rmsnorm_fwd(d, res_r, w, ch.eps, "rne", threads=THREADS)
        out_ref, res_ref = torch_reference(d, res_ref, w, ch.eps)
        # residual_out does not depend on the norm, so the RNE chain is the
        # torch reference chain bit for bit ("shrink +0.000%")
        assert np.array_equal(res_r, refs.u16(res_ref)), step
        if (step + 1) % 24 == 0:
            shrink = 100 * (1 - refs.rms(refs.bf16_value(res_t)) / refs.rms(refs.bf16_value(res_r)))
            cos = refs.cos_sim(refs.bf16_value(out_t), refs.bf16_value(out_r))
            assert abs(shrink - GOLD[f"chain.{step + 1}.shrink_percent"]) < 0.02, (step, shrink)
            assert abs(cos - GOLD[f"chain.{step + 1}.out_cos"]) < 1e-5, (step, cos)
            cos_rne = refs.cos_sim(refs.bf16_value(out_r), refs.bf16_value(refs.u16(out_ref)))
            assert round(cos_rne, 8) == 1.0


@pytest.mark.slow
def test_chain4096_drift_and_bias(orc):
    """The 72-call chain at 4096 x 4096: round-to-nearest-even stays within
    0.05% of the unrounded (fp64) residual norm, truncation shrinks it by
    more than 1%, ties-away grows it; the step-0 magnitude bias against the
    fp32 sum is ~0 for RNE, < -1e-3 for truncation, > +5e-5 for ties-away."""
    ch = inputs.CHAIN4096
    r0, w = ch.initial()
    res = {m: refs.u16(r0).copy() for m in ("rne", "trunc", "ties_away")}
    res64 = refs.bf16_value(r0)
    drift = {}
    for k in range(ch.depth):
        d = ch.delta(k)
        if k == 0:
            acc32 = (d.float() + r0.float()).numpy().astype(np.float64)
        for m in res:
            _, res[m] = orc.add_rmsnorm_fwd(d, res[m], w, ch.eps, m, threads=THREADS)
            if k == 0:
                b = refs.magnitude_bias_values(res[m], acc32)
                if m == "rne":
                    assert abs(b) < 2e-5, b
                elif m == "trunc":
                    assert b < -1e-3, b
                else:
                    assert b > 5e-5, b
        res64 = res64 + refs.bf16_value(d)
        if (k + 1) % 24 == 0:
            n64 = refs.rms(res64)
            drift[k + 1] = {m: refs.rms(refs.bf16_value(res[m])) / n64 - 1 for m in res}
    assert abs(drift[72]["rne"]) < 5e-4, drift
    assert drift[72]["trunc"] < -1e-2, drift
    assert drift[72]["ties_away"] > drift[72]["rne"], drift
