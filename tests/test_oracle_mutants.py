"""Each planted mistake in the oracle (a dropped term, a wrong sign, index or
operand order) must make at least one pin fail."""
import pytest

import oracle
from tests import oracle_pins

PLANTS = {
    1: "nibble order reversed",
    2: "dequant bias dropped",
    3: "wrong quantisation group index",
    4: "silu replaced by sigmoid",
    5: "ties broken toward the higher index",
    6: "top-k weights not renormalised",
    7: "gate and up swapped",
    8: "scatter not stable in token order",
    9: "router bias sign flipped",
    10: "down matrix transposed",
    11: "shared expert dropped",
    12: "rms norm without square root",
    13: "NaN logit ranked above every number",
}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda p: f"{p}-{PLANTS[p]}")
def test_planted_mistake_is_caught(plant, tmp_path):
    orc = oracle.Oracle(plant, out_dir=str(tmp_path))
    assert orc.lib.oracle_planted() == plant
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught planted mistake {plant} ({PLANTS[plant]})"
