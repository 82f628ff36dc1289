"""CPU pins of the fp64 oracle (see tests/oracle_pins.py for what each pins)."""
import os

import pytest

import oracle_pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_golden_two_keys_file_matches_pin():
    """The printed hand-worked values and the ones the pin asserts agree."""
    path = os.path.join(os.path.dirname(__file__), "golden", "two_keys.txt")
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, value = line.split()
                vals[name] = float(value)
    assert vals == {"o0": -0.1931757358900147, "o1": 1.642391233933647,
                    "lse0": 1.8132616875182228, "lse1": -0.8730719889570275}
