"""The oracle's admissible interval for the order-free (atomic) AllReduce
against its pins (no GPU needed):

* hand-derived intervals, worked out on paper from the bound's formula, that
  fail if a factor, the unit roundoff, the R - 1 or the flush term is wrong;
* brute force: every order of every tiny case, simulated add by add in
  binary32 with and without flush-to-zero, lands inside the interval;
* small integers: every order gives the same bits, and they are the
  fixed-order oracle's;
* the vectorised narrowing against the scalar one, and the checks of
  non-finite elements.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import atomic
from barrier_free_message_gb300 import inputs


def f32(*vals):
    return np.array(vals, dtype=np.float32)


def column(*vals, dtype="fp32"):
    x = f32(*vals)[:, None]
    return x if dtype == "fp32" else oracle.narrow_bf16_array(x)


def bf16_bits(v):
    return oracle.narrow_bf16(float(v))


# ------------------------------------------------------------- hand-derived
def test_two_ranks_hand_derived():
    # x = (1, 2^-30): A = s = 1 + 2^-30, B ~ 2 * 2^-24 * A = 2^-23.
    # s - B = 1 - 2^-23 + 2^-30 - ..., binary32 spacing below 1 is 2^-24, so
    # rounding down gives 1 - 2^-23; s + B = 1 + 2^-23 + 2^-30 + ..., spacing
    # above 1 is 2^-23, so rounding up gives 1 + 2^-22.
    lo, hi = atomic.interval(column(1.0, 2.0 ** -30))
    assert lo[0] == 1 - 2.0 ** -23 and hi[0] == 1 + 2.0 ** -22
    # in bf16 both ends round back to 1
    lo, hi = atomic.interval(column(1.0, 2.0 ** -30, dtype="bf16"))
    assert lo[0] == 1.0 and hi[0] == 1.0


def test_four_ranks_hand_derived():
    # x = (1, 2^-30, 2^-30, 2^-30): B ~ 2 * 3 * 2^-24 = 3 * 2^-23.
    # s - B = 1 - 6 * 2^-24 + 3 * 2^-30 -> down: 1 - 3 * 2^-23
    # s + B = 1 + 3 * 2^-23 + 3 * 2^-30 -> up:   1 + 4 * 2^-23
    lo, hi = atomic.interval(column(1.0, 2.0 ** -30, 2.0 ** -30, 2.0 ** -30))
    assert lo[0] == 1 - 3 * 2.0 ** -23 and hi[0] == 1 + 4 * 2.0 ** -23


def test_flushed_subnormals_are_admissible():
    # two subnormal inputs: a flushing adder returns 0, a gradual one 2^-129
    lo, hi = atomic.interval(column(2.0 ** -130, 2.0 ** -130))
    assert lo[0] <= 0.0 <= 2.0 ** -129 <= hi[0]
    assert hi[0] < 2.0 ** -122           # and not much more (B ~ 4 * 2^-126)


def test_sixteen_ones_hand_derived():
    # R = 16 copies of 1: s = A = 16, B = 2 * 15 * 2^-24 * 16 + ... =
    # 15 * 2^-19 + ...; binary32 spacing is 2^-20 below 16 and 2^-19 above,
    # so s - B rounds down to 16 - 31 * 2^-20 and s + B up to 16 + 16 * 2^-19;
    # in bf16 (spacing 2^-4 below 16, 2^-3 above) both ends round to 16
    lo, hi = atomic.interval(column(*([1.0] * 16)))
    assert lo[0] == 16 - 31 * 2.0 ** -20 and hi[0] == 16 + 16 * 2.0 ** -19
    lo, hi = atomic.interval(column(*([1.0] * 16), dtype="bf16"))
    assert lo[0] == hi[0] == 16.0


def test_check_rejects_values_outside():
    x = column(1.0, 2.0 ** -30)
    for good in (1.0, 1 + 2.0 ** -22, 1 - 2.0 ** -23):
        assert atomic.check(x, f32(good)).all(), good
    for bad in (1 + 2.0 ** -21, 1 - 2.0 ** -22, np.nan, np.inf):
        assert not atomic.check(x, f32(bad)).any(), bad


# -------------------------------------------------------------- brute force
def simulate(values, order, ftz):
    """Binary32 accumulation from +0 in `order`, optionally flushing subnormal
    operands and results to zero (sign kept)."""
    acc = np.float32(0.0)
    for q in order:
        v = np.float32(values[q])
        if ftz and v != 0 and abs(v) < np.float32(2.0 ** -126):
            v = np.float32(np.copysign(0.0, v))
        acc = np.float32(acc + v)
        if ftz and acc != 0 and abs(acc) < np.float32(2.0 ** -126):
            acc = np.float32(np.copysign(0.0, acc))
    return acc


def awkward_cases(seed, R, cases):
    rng = np.random.default_rng(seed)
    out = np.empty((R, cases), dtype=np.float32)
    for j in range(cases):
        kind = j % 5
        if kind == 0:      # wide magnitude spread
            v = rng.standard_normal(R) * 2.0 ** rng.integers(-24, 25, R)
        elif kind == 1:    # cancellation
            b = rng.standard_normal() * 2.0 ** rng.integers(0, 20)
            v = np.concatenate([[b, -b], rng.standard_normal(R - 2) * 2.0 ** -20])
        elif kind == 2:    # subnormals and tiny normals
            v = rng.standard_normal(R) * 2.0 ** rng.integers(-150, -120, R)
        elif kind == 3:    # values close to each other
            v = 1.0 + rng.integers(-8, 8, R) * 2.0 ** -23
        else:              # plain normal
            v = rng.standard_normal(R)
        out[:, j] = rng.permutation(v)
    return out


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("R", [2, 3, 4, 5])
def test_every_order_is_admissible(R, dtype):
    x32 = awkward_cases(100 + R, R, 400)
    x = x32 if dtype == "fp32" else oracle.narrow_bf16_array(x32)
    xw = atomic.widen(x).astype(np.float32)
    lo, hi = atomic.interval(x)
    fold = atomic.widen(oracle.allreduce(x)[:1])[0]
    assert ((lo <= fold) & (fold <= hi)).all(), "the fixed-order fold must be admissible"
    for j in range(x.shape[1]):
        for order in itertools.permutations(range(R)):
            for ftz in (False, True):
                acc = simulate(xw[:, j], order, ftz)
                v = float(acc) if dtype == "fp32" else oracle.widen_bf16(oracle.narrow_bf16(float(acc)))
                assert lo[j] <= v <= hi[j], (j, order, ftz, xw[:, j], v, lo[j], hi[j])


def test_small_integers_are_order_free():
    x = inputs.to_bits(inputs.draw(21, 0, 5, 300, "int", 64.0, "bf16"))
    xw = atomic.widen(x).astype(np.float32)
    want = oracle.allreduce(x)[0]
    for j in range(x.shape[1]):
        got = {bf16_bits(simulate(xw[:, j], order, ftz))
               for order in itertools.permutations(range(5)) for ftz in (False, True)}
        assert got == {int(want[j])}, (j, got, int(want[j]))


# ------------------------------------------------------ helpers and specials
def test_array_narrowing_matches_scalar():
    pats = np.array([0x3F808000, 0x3F818000, 0x3F80FFFF, 0x3F807FFF, 0x7F7FFFFF, 0xFF7FFFFF, 0x00000001,
                     0x80000001, 0x7FC00001, 0xFF800001, 0x7F800000, 0x00008000, 0x00018000],
                    dtype=np.uint32)
    rng = np.random.default_rng(5)
    pats = np.concatenate([pats, rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32)])
    f = pats.view(np.float32)
    got = oracle.narrow_bf16_array(f)
    want = np.array([oracle.narrow_bf16(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_non_finite_classes():
    x = np.array([[np.nan, np.inf, np.inf, -np.inf, 1.0],
                  [1.0, -np.inf, 2.0, 3.0, 2.0]], dtype=np.float32)
    good = np.array([np.nan, np.nan, np.inf, -np.inf, 3.0], dtype=np.float32)
    assert atomic.check(x, good).all()
    bad = np.array([1.0, np.inf, -np.inf, np.inf, np.nan], dtype=np.float32)
    assert not atomic.check(x, bad).any()


def test_check_refuses_possible_overflow():
    x = np.array([[3e38], [3e38]], dtype=np.float32)
    with pytest.raises(ValueError):
        atomic.check(x, np.array([np.inf], dtype=np.float32))
