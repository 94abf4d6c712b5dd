"""The CPU oracle against its pins (page values, closed forms, exact
arithmetic, library casts); see tests/pins.py for what each pin checks."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.FAST_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rne_matches_torch_cast(orc):
    pins.pin_rne_vs_torch_sample(orc, n_random=1 << 22)
