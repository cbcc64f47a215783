"""Each planted mistake in the oracle must trip at least one pin (CPU only).

The plants are compile-time variants of oracle.c (ORACLE_PLANT=n): a dropped
causal mask, a causal mask off by one, a wrong exponent sign, a missing
normalisation, a transposed K operand, and a log-normaliser without its
row maximum.
"""
import pytest

import oracle
from tests import oracle_pins

PLANTS = {1: "causal mask dropped", 2: "mask off by one", 3: "exponent sign",
          4: "no normalisation", 5: "transposed K", 6: "LSE without max",
          7: "grouped K/V heads mapped round-robin",
          8: "backward: softmax row correction dropped", 9: "backward: scale missing from dK"}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda p: PLANTS[p])
def test_plant_is_caught(plant, tmp_path):
    path = oracle.build(str(tmp_path / f"liboracle_plant{plant}.so"), plant=plant)
    lib = oracle.load(path)
    assert lib.oracle_plant() == plant
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:
            caught.append((pin.__name__, str(e)[:80]))
    assert caught, f"planted mistake '{PLANTS[plant]}' passed every pin"
