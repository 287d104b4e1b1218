"""The oracle's row-parallel projection against its pins (no GPU)."""
import numpy as np
import pytest

import gemv_pins as pins
import oracle


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check()


def test_rejects_bad_arguments():
    with pytest.raises(TypeError):
        oracle.gemv(np.zeros((2, 4), np.float32), np.zeros((2, 4, 8), np.float32))
    with pytest.raises(ValueError):
        oracle.gemv(np.zeros((2, 4), np.uint16), np.zeros((2, 5, 8), np.uint16))


MUTANTS = {18: "rows folded from the last", 19: "last row dropped", 20: "weights read transposed",
           21: "rows summed in 8 segments, then the segment sums"}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant):
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(mutant=mutant)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {mutant} ({MUTANTS[mutant]})"
