"""Pins of the oracle's residual-add + RMS normalisation (``oracle.add_rmsnorm``).

Each ``check_*`` takes the oracle variant (0 = the oracle, other numbers = a
copy with one planted mistake) and raises AssertionError when the variant
breaks what the pin fixes:

* closed form: a row of equal powers of two +-2^k normalises to +-1, so the
  output is +-w exactly (eps = 0), and z is the input;
* an independent float64 RMS normalisation, y = z / sqrt(mean(z^2) + eps) w,
  with z = T(a + res) computed here from numpy's binary32 add; the tolerance
  follows from the definition's roundings (see ``check_vs_float64``);
* invariants: scaling a row by 2^k leaves y unchanged bit for bit and scales
  z by 2^k (eps = 0); permuting the elements of a row (weights with them)
  permutes y; normalising the returned z again (residual 0, no AllReduce)
  gives the same y;
* special rows: all zeros give 0; a NaN makes the row NaN; an infinity
  makes every finite element 0 and itself NaN.
"""
import numpy as np

import oracle
from barrier_free_message_gb300 import inputs


def f64(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def to_type(f32, dtype):
    return oracle.narrow_bf16_array(f32) if dtype == "bf16" else np.asarray(f32, np.float32)


def draw(seed, R, rows, h, dtype, sigma=1.0):
    g = [inputs.to_bits(inputs.draw(seed, c, R, rows * h, "normal", sigma, dtype)) for c in range(2)]
    w = inputs.to_bits(inputs.draw(seed, 2, 1, h, "normal", 1.0, dtype))[0]
    return g[0], g[1], w


def check_power_of_two_rows(mutant=0):
    for dtype in ("bf16", "fp32"):
        R, rows, h = 2, 6, 48
        k = np.array([0, 3, -5, 20, -30, 7])
        sign = np.array([1, -1, 1, -1, 1, 1])
        a32 = np.repeat((sign * np.ldexp(1.0, k)).astype(np.float32)[:, None], h, axis=1).reshape(-1)
        a = np.stack([to_type(a32, dtype)] * R)
        res = np.zeros_like(a)
        w = to_type(np.linspace(-2, 3, h).astype(np.float32), dtype)
        out, z = oracle.add_rmsnorm(a, res, w, 0.0, h, allreduce_first=False, mutant=mutant)
        want = np.concatenate([to_type(f64(w).astype(np.float32) * s, dtype) for s in sign])
        for r in range(R):
            assert np.array_equal(z[r], a[r]), "z of a zero residual must be the input"
            assert np.array_equal(out[r], want), f"{dtype}: rows of +-2^k must give +-w"


def check_vs_float64(mutant=0):
    """Tolerance.  Against the exact normalisation the definition's roundings
    give a relative error below 8 * 2^-24 before the final store: in ms the
    truncated sum of squares (< 2^-25 here, h <= 4096), float(S), the
    division by h and the eps add (2^-24 each), halved through the square
    root; then sqrt, the reciprocal and the two products (2^-24 each).
    fp32 output: |y - y64| <= 2^-21 |y64| + 2^-140; bf16 output adds the
    final rounding (2^-9 relative) and a possible flip at a near-tie:
    |y - y64| <= 2^-8 |y64| + 2^-130."""
    for dtype, rel in (("fp32", 2.0 ** -21), ("bf16", 2.0 ** -8)):
        R, rows, h = 4, 5, 4096
        x, res, w = draw(40, R, rows, h, dtype)
        eps = 0.5
        out, z = oracle.add_rmsnorm(x, res, w, eps, h, mutant=mutant)
        a = oracle.allreduce(x)                         # pinned on its own
        z_want = to_type((f64(a).astype(np.float32) + f64(res).astype(np.float32)).astype(np.float32), dtype)
        assert np.array_equal(z, z_want), "z must be T(a + res) in binary32"
        zz = f64(z_want).reshape(R, rows, h)
        rstd = 1.0 / np.sqrt((zz * zz).mean(axis=2, keepdims=True) + np.float64(np.float32(eps)))
        y64 = (zz * rstd * f64(w)[None, None, :]).reshape(R, rows * h)
        y = f64(out)
        bad = np.abs(y - y64) > rel * np.abs(y64) + 2.0 ** -130
        assert not bad.any(), f"{dtype}: {int(bad.sum())} elements off the float64 normalisation"


def check_scaling_and_order(mutant=0):
    for dtype in ("bf16", "fp32"):
        R, rows, h = 2, 3, 1000
        x, res, w = draw(41, R, rows, h, dtype)
        a = oracle.allreduce(x)
        out, z = oracle.add_rmsnorm(a, res, w, 0.0, h, allreduce_first=False, mutant=mutant)
        for k in (-12, 9):
            s = lambda t: to_type((f64(t) * 2.0 ** k).astype(np.float32), dtype)
            out2, z2 = oracle.add_rmsnorm(s(a), s(res), w, 0.0, h, allreduce_first=False, mutant=mutant)
            assert np.array_equal(out2, out), f"{dtype}: scaling by 2^{k} changed y"
            assert np.array_equal(z2, s(z)), f"{dtype}: scaling by 2^{k} must scale z"
        perm = np.random.default_rng(3).permutation(h)
        p = lambda t: t.reshape(R, rows, h)[:, :, perm].reshape(R, rows * h)
        out3, _ = oracle.add_rmsnorm(p(a), p(res), w[perm], 0.0, h, allreduce_first=False, mutant=mutant)
        assert np.array_equal(out3, p(out)), f"{dtype}: the order within a row changed y"


def check_renormalise_z(mutant=0):
    for dtype in ("bf16", "fp32"):
        R, rows, h = 3, 4, 2048
        x, res, w = draw(42, R, rows, h, dtype, sigma=3.0)
        out, z = oracle.add_rmsnorm(x, res, w, 1e-3, h, mutant=mutant)
        out2, z2 = oracle.add_rmsnorm(z, np.zeros_like(z), w, 1e-3, h, allreduce_first=False, mutant=mutant)
        assert np.array_equal(z2, z) and np.array_equal(out2, out), f"{dtype}: y is not the normalisation of z"


def check_special_rows(mutant=0):
    R, h = 2, 16
    a = np.zeros((R, 3 * h), np.float32)
    a[:, h:] = 1.0
    a[:, h + 3] = np.nan
    a[:, 2 * h + 5] = np.inf
    res = np.zeros_like(a)
    w = np.full(h, 2.0, np.float32)
    out, _ = oracle.add_rmsnorm(a, res, w, 1e-6, h, allreduce_first=False, mutant=mutant)
    assert (out[:, :h] == 0).all(), "an all-zero row normalises to 0"
    assert np.isnan(out[:, h:2 * h]).all(), "a NaN makes the row NaN"
    row = out[:, 2 * h:]
    assert np.isnan(row[:, 5]).all() and (np.delete(row, 5, axis=1) == 0).all(), "an infinity gives rstd = 0"


ALL_CHECKS = [check_power_of_two_rows, check_vs_float64, check_scaling_and_order, check_renormalise_z,
              check_special_rows]
