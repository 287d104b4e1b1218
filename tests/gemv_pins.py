"""Pins of the oracle's row-parallel projection (``oracle.gemv``).

Each ``check_*`` takes the oracle variant (0 = the oracle, other numbers = a
copy with one planted mistake) and raises AssertionError when the variant
breaks what the pin fixes:

* small integers: every partial sum is exact, so the result is the integer
  product x W (numpy int64) rounded once to bf16;
* hand-derived order witnesses, each 0 only for a left fold in row order:
  rows 2^24, 1, -2^24 (any other order of the three gives 1), and rows
  2^24 at 0, 1 at 3 and 4, -2^24 at 23 (a sum of blocks of rows, for
  instance segments of consecutive rows or pairs, keeps the two ones: 2);
* an independent float64 product within the bound of the k - 1 roundings
  of a left fold;
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
    # column 0: rows 0, 1, 2 = 2^24, 1, -2^24.  From the left, 2^24 + 1 is a
    # tie that rounds to the even 2^24, so the ones vanish and the sum is 0;
    # from the right, -2^24 + 1 is exact and the sum is 1.
    k = 24
    x = np.zeros((1, k), np.float32)
    W = np.zeros((1, k, 2), np.float32)
    x[0, :] = 1.0
    W[0, :3, 0] = [2.0 ** 24, 1.0, -(2.0 ** 24)]
    # column 1: rows 0, 3, 4, 23 = 2^24, 1, 1, -2^24.  A left fold in row
    # order loses each one against 2^24 (0); any order that adds rows 3 and 4
    # to each other first -- segments of 3 rows, pairs, a tree -- keeps 2.
    W[0, [0, 3, 4, 23], 1] = [2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)]
    y = f64(oracle.gemv(bf16(x), bf16(W), mutant=mutant))
    assert y[0, 0] == 0.0, "rows must be added in row order, from row 0"
    assert y[0, 1] == 0.0, "rows must be added one at a time to one running sum"


def check_vs_float64(mutant=0):
    """|y - y64| <= 2 (k + 1) 2^-24 sum_i |x_i W_ij| + 2^-8 |y64|: k - 1
    additions of the left fold, each rounding by 2^-24 of a partial sum
    bounded by sum |x W| (doubled for second-order terms), then the final
    rounding to bf16 (2^-9, doubled for a near-tie flip)."""
    R, k, h = 4, 1024, 512
    x = inputs.to_bits(inputs.draw(60, 0, R, k, "normal", 1.0, "bf16"))
    W = inputs.to_bits(inputs.draw(60, 1, R, k * h, "normal", 0.05, "bf16")).reshape(R, k, h)
    y = f64(oracle.gemv(x, W, mutant=mutant))
    xf, Wf = f64(x), f64(W)
    y64 = np.einsum("rk,rkh->rh", xf, Wf)
    mag = np.einsum("rk,rkh->rh", np.abs(xf), np.abs(Wf))
    bad = np.abs(y - y64) > 2 * (k + 1) * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(y64)
    assert not bad.any(), f"{int(bad.sum())} outputs off the float64 product"


def check_single_row(mutant=0):
    x = bf16([[1.5], [-3.0]])
    W = bf16([[[2.0 ** -3, -7.0, 1.0 + 2.0 ** -7]], [[0.25, 3.0, -(2.0 ** 100)]]])
    y = oracle.gemv(x, W, mutant=mutant)
    want = bf16((f64(x)[:, :, None] * f64(W)).sum(axis=1).astype(np.float32))
    assert np.array_equal(y, want), "one row: the product rounded once"


ALL_CHECKS = [check_small_integers, check_order_witnesses, check_vs_float64, check_single_row]
