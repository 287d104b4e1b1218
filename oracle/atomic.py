"""Admissible results of the AllReduce whose additions run in any order.

TEST INFRASTRUCTURE ONLY, under the same rule as the rest of this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import it, and it shares nothing with the GPU library.

What it follows.  "Every Microsecond Counts" (page 1), section "Four
barrier-free mechanisms", part 4 (the LL128 atomic algorithm): every rank
adds its data into a shared 128-byte line with hardware atomic adds and bumps
the line's counter; the line is complete when the counter equals the number
of ranks.  The pages fix neither the order of those adds (it is whatever
order the memory system performs them in) nor their precision.  Reading
taken: binary32 accumulators starting from zero, one binary32 add per rank,
round to nearest even, subnormal operands and results possibly flushed to
zero (the hardware float atomics do), then one rounding to the output type.

So the result is not one value but a set.  This module returns, per
element, an interval of the output type that contains every result any order
and either flush behaviour can give:

* s = the exact sum of the widened inputs, A = the sum of their magnitudes;
* recursive summation of R terms in any order, each add rounded with unit
  roundoff u = 2^-24, is within gamma_{R-1} A of s, gamma_k = k u / (1 - k u)
  (N. J. Higham, *Accuracy and Stability of Numerical Algorithms*, 2nd ed.,
  section 4.2); for k u <= 1/2 that is at most 2 (R - 1) u A;
* flushing moves an operand or a result by less than 2^-126, at most R
  operands and R results: 2 R 2^-126 more;
* s and A are evaluated here in binary64 in rank order, which is off by at
  most (R - 1) 2^-53 A; 2^-48 A covers it for every R this library takes.

With B the sum of the three terms, every binary32 accumulator value lies in
[s - B, s + B]; that interval is widened outward to binary32 values, and
both ends are rounded to the output type with the oracle's own narrowing.
Rounding to nearest is monotone, so every admissible result lies between the
two rounded ends.

Non-finite inputs: an element with a NaN, or with both +inf and -inf, is NaN
in every order; otherwise one with +inf (-inf) is +inf (-inf).  The interval
assumes no partial sum overflows, which holds when A is below the largest
binary32 value; ``check`` refuses elements where it does not.
"""
import numpy as np

from . import narrow_bf16_array

U32 = 2.0 ** -24          # unit roundoff of binary32, round to nearest
TINY = 2.0 ** -126        # smallest normal binary32
FLT_MAX = float(np.finfo(np.float32).max)


def widen(x: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) or float32 [R, n] -> exact float64 values."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if x.dtype == np.float32:
        return x.astype(np.float64)
    raise TypeError(f"takes uint16 (bf16 bits) or float32 arrays, got {x.dtype}")


def bound(xw: np.ndarray) -> np.ndarray:
    """B per element for widened inputs xw[R, n] (see the module docstring)."""
    R = xw.shape[0]
    A = np.abs(xw).sum(axis=0)
    return 2.0 * (R - 1) * U32 * A + 2.0 * R * TINY + 2.0 ** -48 * A


def _down32(v: np.ndarray) -> np.ndarray:
    """Largest binary32 <= v (elementwise, v finite float64)."""
    f = v.astype(np.float32)
    return np.where(f.astype(np.float64) > v, np.nextafter(f, np.float32(-np.inf)), f)


def _up32(v: np.ndarray) -> np.ndarray:
    """Smallest binary32 >= v."""
    f = v.astype(np.float32)
    return np.where(f.astype(np.float64) < v, np.nextafter(f, np.float32(np.inf)), f)


def interval(x: np.ndarray):
    """(lo, hi) float64 arrays [n]: the values of the output type (x's type)
    between which every admissible result of the element lies.  Finite
    inputs only (see ``check`` for the others)."""
    xw = widen(np.ascontiguousarray(x))
    s = xw.sum(axis=0)
    B = bound(xw)
    with np.errstate(over="ignore"):
        lo32, hi32 = _down32(s - B), _up32(s + B)
    if x.dtype == np.uint16:
        lo = widen(narrow_bf16_array(lo32)[None, :])[0]
        hi = widen(narrow_bf16_array(hi32)[None, :])[0]
        return lo, hi
    return lo32.astype(np.float64), hi32.astype(np.float64)


def check(x: np.ndarray, out: np.ndarray) -> np.ndarray:
    """Boolean [n]: out[i] (same dtype as x, one rank's result) is an
    admissible result for inputs x[:, i].  Raises ValueError if an element's
    magnitudes could overflow binary32 (the interval does not apply)."""
    x = np.ascontiguousarray(x)
    xw = widen(x)
    v = widen(np.ascontiguousarray(out)[None, :])[0]
    finite = np.isfinite(xw).all(axis=0)
    with np.errstate(invalid="ignore", over="ignore"):
        A = np.where(finite, np.abs(np.where(np.isfinite(xw), xw, 0.0)).sum(axis=0), 0.0)
    if (A >= FLT_MAX / 2).any():
        raise ValueError("partial sums may overflow binary32; the interval does not apply")
    ok = np.zeros(x.shape[1], dtype=bool)
    if finite.any():
        lo, hi = interval(x[:, finite])
        vf = v[finite]
        ok[finite] = (lo <= vf) & (vf <= hi)
    nf = ~finite
    if nf.any():
        xn = xw[:, nf]
        is_nan = np.isnan(xn).any(axis=0) | ((xn == np.inf).any(axis=0) & (xn == -np.inf).any(axis=0))
        pos = (xn == np.inf).any(axis=0)
        vn = v[nf]
        ok[nf] = np.where(is_nan, np.isnan(vn), np.where(pos, vn == np.inf, vn == -np.inf))
    return ok
