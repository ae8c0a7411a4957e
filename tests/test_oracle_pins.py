"""The CPU oracle against its pins (no GPU), and proof that the pins bite:
each deliberately wrong build of the oracle fails at least one pin."""
import os
import tempfile

import pytest

from oracle import build_oracle, oracle as O
from tests import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check, orc):
    check(orc)


PLANTS = {1: "gate and up swapped", 2: "shared branch dropped",
          3: "ties to the higher index", 4: "SiLU sign flipped",
          5: "gate weight paired with the wrong j", 6: "unstable bucket order",
          7: "rows read from the wrong peer", 8: "logits as one sequential chain"}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda p: PLANTS[p].replace(" ", "_"))
def test_planted_mistake_is_caught(plant):
    with tempfile.TemporaryDirectory() as d:
        path = build_oracle.build(os.path.join(d, f"liborc_plant{plant}.so"), plant=plant)
        lib = O.load(path)
        failed = []
        for check in P.ALL_CHECKS:
            try:
                check(lib)
            except AssertionError:
                failed.append(check.__name__)
        assert failed, f"no pin caught planted mistake {plant} ({PLANTS[plant]})"
