"""The select kernel classifies a score against the level-1 bin [kcand, kw]
of the order-preserving key (negative floats bit-inverted, others with the
sign bit set).  When that bin lies at or above the key of +0 it compares the
raw float bits instead: a signed compare for winners (key > kw) and an
unsigned range test for candidates (kcand <= key <= kw).  This pins that
the two rules agree for every bin of the upper half, on random bit patterns
and on the edge values (+-0, +-inf, NaNs, the bin edges themselves)."""

import numpy as np


def _order_key(u):
    return np.where(u & 0x80000000, ~u & 0xFFFFFFFF, u | 0x80000000).astype(np.uint64)


def _as_int32(u):
    s = u.astype(np.int64)
    return np.where(s >= 2**31, s - 2**32, s)


def test_raw_bit_classification_matches_the_order_key():
    rng = np.random.default_rng(0)
    edges = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 1, 0x80000001,
                      0x7FFFFFFF, 0xFFFFFFFF], np.uint64)
    for b1 in list(range(1024, 2048, 5)) + [2047]:
        kcand = b1 << 21
        kw = 0xFFFFFFFF if b1 == 2047 else ((b1 + 1) << 21) - 1
        crange = kw - kcand
        tw, tc = kw & 0x7FFFFFFF, kcand & 0x7FFFFFFF
        near = np.arange(-3, 4, dtype=np.int64)
        u = np.concatenate([rng.integers(0, 2**32, 4000, dtype=np.uint64), edges,
                            ((tc + near) & 0x7FFFFFFF).astype(np.uint64),
                            ((tw + near) & 0x7FFFFFFF).astype(np.uint64),
                            (((tc + near) & 0x7FFFFFFF) | 0x80000000).astype(np.uint64)]) & 0xFFFFFFFF
        key = _order_key(u)
        winners = key > kw
        candidates = ((key - kcand) & 0xFFFFFFFF) <= crange
        assert np.array_equal(winners, _as_int32(u) > tw), b1
        assert np.array_equal(candidates, ((u - tc) & 0xFFFFFFFF) <= crange), b1
