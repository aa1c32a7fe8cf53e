"""The comparators of the GPU parity tests, on the CPU: they accept what the
tolerance rule allows (FP32 logits within max(1e-3 |o|, 1e-4) of the oracle;
top-k sets equal up to positions tied with the k-th score within that
tolerance, in any order) and reject everything else."""

import numpy as np
import pytest

from dsa_case import TOL_ABS, TOL_REL, check_logits, check_topk


def _scores(seed=0, rows=3, width=300):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((rows, width)) * 10
    ends = np.array([width, width - 17, 40])[:rows]
    for r in range(rows):
        s[r, ends[r]:] = -np.inf
    return s, ends


def test_logits_within_the_tolerance_pass():
    want, ends = _scores()
    got = want.astype(np.float32)
    fin = np.isfinite(want)
    nudge = np.where(fin, np.maximum(TOL_REL * np.abs(want), TOL_ABS) * 0.9, 0.0)
    check_logits((want + nudge).astype(np.float32), want, ends, range(3))
    check_logits(got, want, ends, range(3))


def test_logits_past_the_tolerance_fail():
    want, ends = _scores()
    got = want.astype(np.float32).copy()
    o = want[1, 5]
    got[1, 5] = np.float32(o + max(TOL_REL * abs(o), TOL_ABS) * 1.5)
    with pytest.raises(AssertionError):
        check_logits(got, want, ends, range(3))


def test_logits_past_the_bound_must_be_minus_infinity():
    want, ends = _scores()
    got = want.astype(np.float32).copy()
    got[2, ends[2]] = 0.0
    with pytest.raises(AssertionError):
        check_logits(got, want, ends, range(3))


def _oracle_topk(s, ends, k):
    out = np.full((s.shape[0], k), -1, np.int32)
    for r in range(s.shape[0]):
        n = int(ends[r])
        order = np.lexsort((np.arange(n), -s[r, :n]))[:k]
        out[r, :order.size] = order
    return out


def test_topk_in_any_order_passes():
    s, ends = _scores(1)
    k = 32
    got = _oracle_topk(s, ends, k)
    rng = np.random.default_rng(2)
    for r in range(2):
        rng.shuffle(got[r])
    check_topk(got, s, ends, k, range(3))


def test_topk_swap_of_a_tie_at_the_kth_score_passes():
    s, ends = _scores(3)
    k = 16
    r = 0
    n = int(ends[r])
    order = np.lexsort((np.arange(n), -s[r, :n]))
    inside, outside = order[k - 1], order[k]
    s[r, outside] = s[r, inside] - TOL_ABS * 0.5          # within the tolerance of the k-th score
    got = _oracle_topk(s, ends, k)
    got[r, list(got[r]).index(inside)] = outside
    check_topk(got, s, ends, k, range(3))


@pytest.mark.parametrize("mistake", ["low score", "duplicate", "out of range", "short row order"])
def test_topk_mistakes_fail(mistake):
    s, ends = _scores(4)
    k = 16
    got = _oracle_topk(s, ends, k)
    r = 0
    n = int(ends[r])
    if mistake == "low score":
        got[r, 0] = int(np.argmin(s[r, :n]))                  # far below the k-th score
    elif mistake == "duplicate":
        got[r, 1] = got[r, 0]
    elif mistake == "out of range":
        got[r, 0] = n                                           # at the row's bound
    else:
        k = 50                                                  # row 2 holds 40 keys: all of them, in order
        got = _oracle_topk(s, ends, k)
        got[2, [0, 1]] = got[2, [1, 0]]
    with pytest.raises(AssertionError):
        check_topk(got, s, ends, k, range(3))
