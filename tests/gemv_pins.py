"""Pins of the oracle's row-parallel projection (``oracle.gemv``).

Each ``check_*`` takes the oracle variant (0 = the oracle, other numbers = a
copy with one planted mistake) and raises AssertionError when the variant
breaks what the pin fixes:

* small integers: every partial sum is exact, so the result is the integer
  product x W (numpy int64) rounded once to bf16;
* hand-derived order witnesses: rows 2^24, 1, -2^24 inside one segment, and
  the same three values as three segment sums, both give 0 (a left fold);
  any other order gives 1;
* an independent float64 product within the bound of the summation's
  roundings;
* one row (k = 1): the exact product rounded once.
"""
import numpy as np

import oracle
from barrier_free_message_gb300 import inputs


def f64(a):
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16(vals):
    return oracle.narrow_bf16_array(np.asarray(vals, dtype=np.float32))


def check_small_integers(mutant=0):
    rng = np.random.default_rng(11)
    for R, k, h in ((2, 24, 40), (3, 1000, 72), (1, 3584, 16)):
        xi = rng.integers(-8, 9, (R, k))
        Wi = rng.integers(-8, 9, (R, k, h))
        y = oracle.gemv(bf16(xi), bf16(Wi), mutant=mutant)
        want = bf16(np.einsum("rk,rkh->rh", xi, Wi).astype(np.float32))
        assert np.array_equal(y, want), f"integer product R={R} k={k} h={h}"


def check_order_witnesses(mutant=0):
    # within segment 0 (k = 24, c = 3): rows 0, 1, 2 = 2^24, 1, -2^24
    x = np.zeros((1, 24), np.float32)
    W = np.zeros((1, 24, 2), np.float32)
    x[0, :3] = 1.0
    W[0, :3, 0] = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    # across segments: segment sums 2^24, 1, -2^24 (rows 0, 3, 6), column 1
    x2 = np.zeros((1, 24), np.float32)
    x2[0, [0, 3, 6]] = 1.0
    W2 = np.zeros((1, 24, 2), np.float32)
    W2[0, [0, 3, 6], 1] = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    y = oracle.gemv(bf16(x), bf16(W), mutant=mutant)
    y2 = oracle.gemv(bf16(x2), bf16(W2), mutant=mutant)
    assert f64(y)[0, 0] == 0.0, "rows of a segment must be added in row order"
    assert f64(y2)[0, 1] == 0.0, "segment sums must be folded from segment 0"


def check_vs_float64(mutant=0):
    """|y - y64| <= 2 (c + 8) 2^-24 sum_i |x_i W_ij| + 2^-8 |y64|: at most c - 1
    additions inside a segment and 7 across segments, each rounding by 2^-24
    of a partial sum bounded by sum |x W| (doubled for second-order terms),
    then the final rounding to bf16 (2^-9, doubled for a near-tie flip)."""
    R, k, h = 4, 1024, 512
    x = inputs.to_bits(inputs.draw(60, 0, R, k, "normal", 1.0, "bf16"))
    W = inputs.to_bits(inputs.draw(60, 1, R, k * h, "normal", 0.05, "bf16")).reshape(R, k, h)
    y = f64(oracle.gemv(x, W, mutant=mutant))
    xf, Wf = f64(x), f64(W)
    y64 = np.einsum("rk,rkh->rh", xf, Wf)
    mag = np.einsum("rk,rkh->rh", np.abs(xf), np.abs(Wf))
    c = (k + 7) // 8
    bad = np.abs(y - y64) > 2 * (c + 8) * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(y64)
    assert not bad.any(), f"{int(bad.sum())} outputs off the float64 product"


def check_single_row(mutant=0):
    x = bf16([[1.5], [-3.0]])
    W = bf16([[[2.0 ** -3, -7.0, 1.0 + 2.0 ** -7]], [[0.25, 3.0, -(2.0 ** 100)]]])
    y = oracle.gemv(x, W, mutant=mutant)
    want = bf16((f64(x)[:, :, None] * f64(W)).sum(axis=1).astype(np.float32))
    assert np.array_equal(y, want), "one row: the product rounded once"


ALL_CHECKS = [check_small_integers, check_order_witnesses, check_vs_float64, check_single_row]
