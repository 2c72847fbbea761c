"""The CPU oracle against its pins (no GPU)."""
import pytest

from tests import oracle_pins

pytestmark = pytest.mark.timeout(300) if hasattr(pytest.mark, "timeout") else []


@pytest.mark.parametrize("name", sorted(oracle_pins.ALL_PINS))
def test_pin(name):
    oracle_pins.ALL_PINS[name]()
