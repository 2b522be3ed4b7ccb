"""The oracle against its pins (CPU only): hand-worked examples, closed forms, exact arithmetic,
invariants and library special cases. See ``oracle_pins.py`` for what each pin checks."""

import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)
