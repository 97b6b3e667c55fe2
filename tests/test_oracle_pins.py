"""The CPU oracle against its pins (see oracle_pins.py for what each pin is)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("name,fn,needs_pin", P.ALL_CHECKS, ids=[c[0] for c in P.ALL_CHECKS])
def test_oracle_pin(orc, pin, name, fn, needs_pin):
    fn(orc, pin) if needs_pin else fn(orc)
