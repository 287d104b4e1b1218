"""The arithmetic lemma behind the bf16 row statistics of the fused kernels.

The normalisation's sum of squares is an exact integer: every square is
truncated to whole units of 2^(2E - F), where 2^E is the smallest power of two
above every |z| of the row and F = 53 - ceil(log2 hidden).  For elements of at
most 8 significant bits (bf16) the kernels form each term in binary32 instead
of 64-bit integers: v is scaled by 2^k, k = floor(F/2) - E, in two steps
(2^floor(k/2), then 2^(k - floor(k/2))), squared, doubled when F is odd, and
truncated to an integer.  This test checks, on the CPU with numpy's binary32
(round to nearest even, subnormals kept), that the result equals
floor(v^2 2^(F - 2E)) computed exactly with integers, for every positive finite
bf16 value and a spread of admissible E and F.  No kernel code runs here.
"""
import numpy as np


def bf16_values():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)                 # every positive finite bf16
    return (bits << 16).view(np.float32)


def exp_above(v):
    """Smallest E with v < 2^E (v > 0), from the binary32 fields."""
    b = v.view(np.uint32).astype(np.int64)
    eb = b >> 23
    sub = 31 - np.floor(np.log2(np.maximum(b, 1))).astype(np.int64)   # leading zeros of the subnormal field
    return np.where(eb > 0, eb - 126, (31 - sub) - 148)


def exact_terms(v, E, F):
    """floor(v^2 2^(F - 2E)) with integers: v = m 2^e exactly."""
    b = v.view(np.uint32).astype(np.int64)
    eb, fr = b >> 23, b & 0x7FFFFF
    m = np.where(eb > 0, fr | 0x800000, fr)
    e = np.where(eb > 0, eb - 150, -149)
    # m has its low 16 bits zero (bf16): use the 8-bit significand to stay in int64
    m8, e8 = m >> 16, e + 16
    sh = 2 * e8 + F - 2 * E
    sq = m8 * m8
    out = np.zeros_like(sq)
    pos = sh >= 0
    out[pos] = sq[pos] << sh[pos]
    neg = ~pos & (sh > -64)
    out[neg] = sq[neg] >> (-sh[neg])
    return out


def narrow_terms(v, E, F):
    """The binary32 formulation of the kernels."""
    k = F // 2 - E
    k1 = k >> 1
    k2 = k - k1
    s1 = ((127 + k1) << 23).astype(np.uint32).view(np.float32)
    s2 = ((127 + k2) << 23).astype(np.uint32).view(np.float32)
    with np.errstate(under="ignore"):
        vs = (v * s1).astype(np.float32) * s2
        vs = vs.astype(np.float32)
        t = (vs * vs).astype(np.float32)
        t = np.where((F & 1) == 1, (t * np.float32(2.0)).astype(np.float32), t)
    assert (t < 2.0 ** 53).all()
    return np.trunc(t.astype(np.float64)).astype(np.int64)


def test_exp_above_is_the_smallest_bound():
    v = bf16_values().astype(np.float64)
    E = exp_above(bf16_values())
    assert (v < np.ldexp(1.0, E)).all() and (v >= np.ldexp(1.0, E - 1)).all()


def test_narrow_terms_equal_the_exact_truncated_squares():
    v = bf16_values()
    E0 = exp_above(v)
    checked = 0
    for F in (36, 37, 40, 45, 52, 53):                     # hidden from 2^17 down to 1
        for dE in (0, 1, 2, 7, 19, 40, 90, 200):           # rows whose largest |z| is 2^dE above v
            E = E0 + dE
            keep = E <= 128
            vv, EE = v[keep], E[keep]
            got = narrow_terms(vv, EE, np.full_like(EE, F))
            want = exact_terms(vv, EE, np.full_like(EE, F))
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, (F, dE, float(vv[bad[0]]), int(EE[bad[0]]), int(got[bad[0]]), int(want[bad[0]]))
            checked += vv.size
    assert checked > 1_000_000


def test_a_planted_mistake_is_caught():
    """Without the doubling for odd F the formulation is wrong: the check sees it."""
    v = bf16_values()[::97]
    E = exp_above(v) + 1
    F = np.full_like(E, 37)
    k = F // 2 - E
    s = ((127 + (k >> 1)) << 23).astype(np.uint32).view(np.float32)
    s2 = ((127 + k - (k >> 1)) << 23).astype(np.uint32).view(np.float32)
    with np.errstate(under="ignore"):
        vs = ((v * s).astype(np.float32) * s2).astype(np.float32)
        t = (vs * vs).astype(np.float32)
    wrong = np.trunc(t.astype(np.float64)).astype(np.int64)
    assert (wrong != exact_terms(v, E, F)).any()


def floor_by_shift(t):
    """The kernels' floor of a binary32 t in [0, 2^53): the significand with its
    implicit bit, as m 2^32, shifted right by 182 - (exponent field), amounts
    above 63 giving 0 (PTX shr.b64 clamps them)."""
    b = t.view(np.uint32).astype(np.uint64)
    m = ((b & np.uint64(0x7FFFFF)) | np.uint64(0x800000)) << np.uint64(32)
    amt = np.uint64(182) - (b >> np.uint64(23))
    out = np.zeros_like(m)
    ok = amt < np.uint64(64)
    out[ok] = m[ok] >> amt[ok]
    return out.astype(np.int64)


def test_floor_by_shift_is_the_floor():
    # every exponent field a t in [0, 2^53) can have, with edge and random significands
    rng = np.random.default_rng(5)
    fields = np.arange(0, 127 + 53, dtype=np.uint32)
    mant = np.concatenate([np.array([0, 1, 2, 0x400000, 0x7FFFFE, 0x7FFFFF], dtype=np.uint32),
                           rng.integers(0, 0x800000, 4000, dtype=np.uint32)])
    t = ((fields[:, None] << np.uint32(23)) | mant[None, :]).reshape(-1).view(np.float32)
    want = np.floor(t.astype(np.float64)).astype(np.int64)
    assert np.array_equal(floor_by_shift(t), want)
    # and on every square the narrow path forms for the bf16 values
    v = bf16_values()
    for F in (36, 40, 53):
        for dE in (0, 1, 5, 30):
            E = exp_above(v) + dE
            keep = E <= 128
            k = F // 2 - E[keep]
            k1 = k >> 1
            s1 = ((127 + k1) << 23).astype(np.uint32).view(np.float32)
            s2 = ((127 + k - k1) << 23).astype(np.uint32).view(np.float32)
            with np.errstate(under="ignore"):
                vs = ((v[keep] * s1).astype(np.float32) * s2).astype(np.float32)
                tt = (vs * vs).astype(np.float32)
                if F & 1:
                    tt = (tt * np.float32(2.0)).astype(np.float32)
            assert np.array_equal(floor_by_shift(tt), np.floor(tt.astype(np.float64)).astype(np.int64))
