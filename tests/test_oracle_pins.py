"""The CPU oracle against closed forms, exact enumeration, library special
cases, brute force and the pages' worked example (see ``_pins.py``)."""
import pytest

import _pins


@pytest.mark.parametrize("name", sorted(_pins.ALL_PINS))
def test_pin_holds(name):
    errs = _pins.ALL_PINS[name]()
    assert not errs, errs
