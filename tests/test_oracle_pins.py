"""The CPU oracle against its pins (no GPU needed)."""
import numpy as np
import pytest
import torch

import exact_ref
import oracle
import oracle_pins as pins
from barrier_free_message_gb300 import inputs


def test_all_ones_gives_R():
    pins.check_all_ones()


def test_every_rank_gets_the_same_bits():
    pins.check_identical_ranks()


def test_power_of_two_scaling_is_exact():
    pins.check_power_of_two_scaling()


def test_small_integers_exact_and_additive():
    pins.check_small_integers()


def test_hand_derived_cases():
    pins.check_golden()


@pytest.mark.parametrize("R", [2, 3, 4])
def test_brute_force_against_exact_arithmetic(R):
    pins.check_brute_force(ranks=(R,))


def test_fp32_brute_force_against_exact_arithmetic():
    vals = [0x00000000, 0x80000000, 0x3F800000, 0xBF800000, 0x00000001, 0x80000001,
            0x4B800000, 0xCB800000, 0x33800000, 0xB3800000, 0x7F7FFFFF, 0xFF7FFFFF,
            0x00800000, 0x3F800001]
    import itertools
    tuples = list(itertools.product(vals, repeat=3))
    x = np.array(tuples, dtype=np.uint32).T.copy().view(np.float32)
    out = oracle.allreduce(x).view(np.uint32)
    for j, t in enumerate(tuples):
        assert int(out[0, j]) == exact_ref.fold_fp32(list(t)), [hex(v) for v in t]


def test_narrowing_matches_torch():
    pins.check_narrowing_vs_torch()


def test_threaded_oracle_gives_identical_bits():
    x = inputs.to_bits(inputs.draw(15, 0, 8, 100_003, "normal", 1.0, "bf16"))
    assert np.array_equal(oracle.allreduce(x), oracle.allreduce(x, threads=4))
    xf = inputs.to_bits(inputs.draw(15, 1, 4, 50_001, "uniform", 1.0, "fp32"))
    assert np.array_equal(oracle.allreduce(xf).view(np.uint32),
                          oracle.allreduce(xf, threads=3).view(np.uint32))


def test_exact_ref_encodings_roundtrip():
    # the exact reference's own encoders invert its decoders on every bf16 value
    for b in range(0, 1 << 16):
        if (b >> 7) & 0xFF == 0xFF:
            continue
        assert exact_ref.units_to_bf16_bits(*exact_ref.bf16_bits_to_units(b)) == b


def test_oracle_rejects_bad_arguments():
    with pytest.raises(TypeError):
        oracle.allreduce(np.zeros((2, 4), np.float64))
    out = oracle.allreduce(np.zeros((3, 0), np.uint16))
    assert out.shape == (3, 0)


# Each planted mistake in the oracle must be caught by at least one pin.
MUTANTS = {
    1: "reversed rank order",
    2: "bf16 accumulator",
    3: "fold starts from +0",
    4: "last rank dropped",
    5: "truncating narrowing",
    6: "only rank 0 written",
    7: "pairwise tree",
    8: "neighbouring element read",
    9: "last rank subtracted",
    10: "subnormal inputs flushed",
    11: "ties away from zero",
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
