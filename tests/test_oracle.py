"""The CPU oracle against its pins (format definitions, exact arithmetic,
invariants, library routines).  No GPU needed."""
import pytest

from tests import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()
