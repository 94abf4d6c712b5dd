"""The log-sum-exp oracle against its pins (tests/pins_lse.py), and planted
slips in copies of its C source that the pins must catch."""
import pytest

import oracle.lse as lse
import pins_lse

S = lse.SOURCE.read_text()


@pytest.fixture(scope="module")
def o():
    return lse.lib()


@pytest.mark.parametrize("pin", pins_lse.LSE_PINS, ids=lambda p: p.__name__)
def test_pin(o, pin):
    pin(o)


MUTANTS = {
    "gap_sign_flipped": ("return hi + log1p(exp(lo - hi));", "return hi + log1p(exp(hi - lo));"),
    "log_instead_of_log1p": ("return hi + log1p(exp(lo - hi));", "return hi + log(exp(lo - hi));"),
    "base_is_min": ("return hi + log1p(exp(lo - hi));", "return lo + log1p(exp(lo - hi));"),
    "log1p_term_dropped": ("return hi + log1p(exp(lo - hi));", "return hi;"),
    "both_minus_inf_gives_nan": ("        return hi; /* +inf, or -inf when both are -inf */",
                                 "        return hi > 0 ? hi : NAN;"),
    "nan_ignored": ("    if (isnan(a) || isnan(b))\n        return NAN;", ""),
    "unary_cosh_is_sinh": ("op == LSE_UNARY_COSH ? cosh(v)", "op == LSE_UNARY_COSH ? sinh(v)"),
    "unary_log1p_is_log": ("op == LSE_UNARY_LOG1P ? log1p(v)", "op == LSE_UNARY_LOG1P ? log(v)"),
    "strided_rows_ignore_stride": ("a[r * a_stride + c], b[r * b_stride + c]", "a[r * n_cols + c], b[r * b_stride + c]"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    assert S.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(S.replace(old, new))
    so = lse.compile_source(src, tmp_path / f"lib{name}.so")
    o = lse.LseOracle(so)
    caught = []
    for pin in pins_lse.LSE_PINS:
        try:
            pin(o)
        except Exception:  # noqa: BLE001 - any failure of a pin counts
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
