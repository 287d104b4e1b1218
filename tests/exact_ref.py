"""Exact-arithmetic reference for pinning the CPU oracle on tiny inputs.

Every binary32 and bf16 value is an integer multiple of 2**-149, so this
module holds each value as a sign and a Python integer count of 2**-149 units.
Sums are then exact, and each rounding step is written out explicitly:
round to nearest, ties to even, to 24 significant bits (binary32) or 8
significant bits (bf16), with the subnormal quantum of each format.  Nothing
here uses hardware floating point, so it is independent of the C oracle it
checks.

The fold it evaluates is the one the AllReduce is held to: widen each rank's
value, add them in rank order 0..R-1 rounding to binary32 after every add, and
round the total once to the output type.
"""

FP32_MAX_UNITS = ((1 << 24) - 1) << 253        # (2 - 2**-23) * 2**127 in 2**-149 units
INF = "inf"


def bf16_bits_to_units(b):
    """bf16 bit pattern -> (negative, magnitude in 2**-149 units)."""
    neg = bool(b & 0x8000)
    exp = (b >> 7) & 0xFF
    frac = b & 0x7F
    if exp == 0xFF:
        raise ValueError("inf/nan not handled")
    if exp == 0:
        return neg, frac << 16                      # frac * 2**-133
    return neg, (128 + frac) << (exp + 15)          # (1.frac) * 2**(exp-127)


def fp32_bits_to_units(u):
    neg = bool(u & 0x80000000)
    exp = (u >> 23) & 0xFF
    frac = u & 0x7FFFFF
    if exp == 0xFF:
        raise ValueError("inf/nan not handled")
    if exp == 0:
        return neg, frac
    return neg, ((1 << 23) + frac) << (exp - 1)


def _round_to_quantum(m, qe):
    """Round the non-negative integer m to a multiple of 2**qe, ties to even."""
    if qe <= 0:
        return m
    q, r = divmod(m, 1 << qe)
    half = 1 << (qe - 1)
    if r > half or (r == half and (q & 1)):
        q += 1
    return q << qe


def round_fp32(neg, m):
    """Round an exact value to binary32 (result still in units)."""
    qe = max(0, m.bit_length() - 24)
    m = _round_to_quantum(m, qe)
    if m > FP32_MAX_UNITS:
        return neg, INF
    return neg, m


def add_exact_then_round_fp32(a, b):
    """binary32 a + b, rounded to nearest even (IEEE sign rules for zeros)."""
    (na, ma), (nb, mb) = a, b
    if ma == 0 and mb == 0:
        return (na and nb), 0                       # -0 + -0 = -0, otherwise +0
    s = (-ma if na else ma) + (-mb if nb else mb)
    if s == 0:
        return False, 0                             # exact zero sum rounds to +0
    return round_fp32(s < 0, abs(s))


def units_to_bf16_bits(neg, m):
    """Round a binary32 value (in units) once to bf16 and encode it."""
    sign = 0x8000 if neg else 0
    if m == INF:
        return sign | 0x7F80
    qe = max(16, m.bit_length() - 8)
    M = _round_to_quantum(m, qe)
    if M == 0:
        return sign
    if M < (1 << 23):                                # subnormal: multiples of 2**-133
        return sign | (M >> 16)
    bl = M.bit_length()
    exp = bl - 23                                    # leading bit 2**(bl-1-149), bias 127
    if exp >= 0xFF:
        return sign | 0x7F80
    sig = M >> (bl - 8)
    return sign | (exp << 7) | (sig - 128)


def units_to_fp32_bits(neg, m):
    sign = 0x80000000 if neg else 0
    if m == INF:
        return sign | 0x7F800000
    if m < (1 << 23):
        return sign | m
    bl = m.bit_length()
    exp = bl - 23
    sig = m >> (bl - 24)
    return sign | (exp << 23) | (sig - (1 << 23))


def fold_bf16(bits_per_rank):
    """The AllReduce of one element: bf16 inputs (one per rank) -> bf16 output bits."""
    acc = bf16_bits_to_units(bits_per_rank[0])
    for b in bits_per_rank[1:]:
        if acc[1] == INF:
            break
        acc = add_exact_then_round_fp32(acc, bf16_bits_to_units(b))
    return units_to_bf16_bits(*acc)


def fold_fp32(bits_per_rank):
    acc = fp32_bits_to_units(bits_per_rank[0])
    for b in bits_per_rank[1:]:
        if acc[1] == INF:
            break
        acc = add_exact_then_round_fp32(acc, fp32_bits_to_units(b))
    return units_to_fp32_bits(*acc)
