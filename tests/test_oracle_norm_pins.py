"""The oracle's residual-add + RMS normalisation against its pins (no GPU)."""
import numpy as np
import pytest

import norm_pins as pins
import oracle


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check()


def test_rejects_bad_arguments():
    x = np.zeros((2, 16), np.float32)
    with pytest.raises(ValueError):
        oracle.add_rmsnorm(x, x, np.zeros(5, np.float32), 0.0, 5)
    with pytest.raises(TypeError):
        oracle.add_rmsnorm(x, x.astype(np.float64), np.zeros(8, np.float32), 0.0, 8)


# Each planted mistake in the normalisation must be caught by at least one pin.
MUTANTS = {
    12: "residual dropped",
    13: "mean over h - 1",
    14: "eps added outside the square root",
    15: "weight dropped",
    16: "mean square of the unrounded z",
    17: "fixed point 8 bits coarser",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant):
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(mutant=mutant)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {mutant} ({MUTANTS[mutant]})"
