"""The fused kernels' largest magnitude of a bf16 vector (max_mag_bf16 in
fused_common.cuh), restated on the CPU: the 16-byte vector's words masked to
the magnitudes of the first n elements, pairwise unsigned 16-bit maxima of
the halves, the larger of the two halves left, moved to the upper half.  It
must equal the largest binary32 magnitude bits of those n elements (a bf16's
bits are the upper half of its binary32 bits).  No kernel code runs here."""
import numpy as np


def packed_max(words, n):
    """words: [N, 4] uint32 (8 bf16 each, element 2i in the low half of word i)."""
    w = words.copy()
    for i in range(4):
        keep = np.uint32(0x7FFF7FFF) if 2 * i + 1 < n else np.uint32(0x00007FFF) if 2 * i < n else np.uint32(0)
        w[:, i] &= keep
    lo, hi = w & np.uint32(0xFFFF), w >> np.uint32(16)
    a_lo, a_hi = np.maximum(lo[:, 0], lo[:, 1]), np.maximum(hi[:, 0], hi[:, 1])
    b_lo, b_hi = np.maximum(lo[:, 2], lo[:, 3]), np.maximum(hi[:, 2], hi[:, 3])
    m_lo, m_hi = np.maximum(a_lo, b_lo), np.maximum(a_hi, b_hi)
    return np.maximum(m_hi, m_lo) << np.uint32(16)


def elementwise_max(words, n):
    halves = np.stack([words & np.uint32(0xFFFF), words >> np.uint32(16)], axis=2).reshape(-1, 8)
    mags = (halves[:, :n].astype(np.uint32) << np.uint32(16)) & np.uint32(0x7FFFFFFF)
    return mags.max(axis=1) if n else np.zeros(len(words), np.uint32)


def test_packed_max_equals_the_elementwise_max():
    rng = np.random.default_rng(12)
    words = rng.integers(0, 1 << 32, size=(20000, 4), dtype=np.uint64).astype(np.uint32)
    # special patterns: zeros, negative zero, infinities, NaN, subnormals, the largest finite
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFFF, 0x0001, 0x807F, 0x7F7F, 0xFF7F],
                        dtype=np.uint32)
    pick = rng.integers(0, len(specials), size=(4000, 8))
    sp = specials[pick]
    words = np.concatenate([words, (sp[:, 0::2] | (sp[:, 1::2] << np.uint32(16)))])
    for n in (4, 8):                       # 8-byte and 16-byte units
        assert np.array_equal(packed_max(words, n), elementwise_max(words, n)), n
