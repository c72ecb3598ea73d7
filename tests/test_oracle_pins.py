"""The CPU oracle against its pins (no GPU needed)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(0)


# Each planted mistake is a plausible error somewhere in the oracle; at least
# one pin must reject it.
PLANTS = {
    1: "dequantisation drops the zero term",
    2: "codes truncated instead of rounded half-to-even",
    3: "query heads grouped interleaved instead of contiguously",
    4: "bit order inside a packed word reversed",
    5: "protected heads quantised anyway",
    6: "visual range end treated as inclusive",
    7: "binary16 conversion truncates",
    8: "softmax scale dropped",
    9: "scale uses 2^b steps instead of 2^b - 1",
    10: "2-bit K storage slots of a register pair swapped",
    11: "K-only protected head keeps its V in bf16 too",
    12: "sensitivity divergence taken in the other direction",
    13: "sensitivity probe quantises V where it should quantise K",
}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda p: PLANTS[p])
def test_pins_catch_planted_mistake(plant):
    caught = []
    for pin in ALL_PINS:
        try:
            pin(plant)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin caught planted mistake {plant}: {PLANTS[plant]}"


def test_oracle_reports_cores():
    assert oracle.online_cores() >= 1
