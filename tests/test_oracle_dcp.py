"""Pins of the DCP oracle (page *amd.ops.fp4_indexer*, ``decode_layout``'s DCP
branch; page *cutedsl.dsa.overlap*, the top-k merge) against brute force."""

import numpy as np
import pytest

from oracle import dcp as D
from oracle import indexer as O


def test_rank_local_ends_count_the_owned_keys():
    rng = np.random.default_rng(0)
    for _ in range(400):
        world = int(rng.integers(1, 9))
        inter = int(rng.choice([1, 2, 3, 16, 64]))
        E = int(rng.integers(0, 3000))
        t = np.arange(E)
        own = D.owner(t, world, inter)
        for rank in range(world):
            mine = t[own == rank]
            assert D.rank_local_ends(E, rank, world, inter) == mine.size
            # their local positions are exactly 0 .. count-1, in global order
            assert np.array_equal(D.global_to_local(mine, world, inter), np.arange(mine.size))
            assert np.array_equal(D.local_to_global(np.arange(mine.size), rank, world, inter), mine)


def test_hand_case():
    # world 2, interleave 2: keys 0,1 4,5 8,9 on rank 0; 2,3 6,7 on rank 1
    assert D.rank_local_ends(10, 0, 2, 2) == 6 and D.rank_local_ends(10, 1, 2, 2) == 4
    assert list(D.local_to_global(np.arange(4), 1, 2, 2)) == [2, 3, 6, 7]


def test_layout_dcp_reduces_to_the_plain_layout():
    rng = np.random.default_rng(1)
    for _ in range(30):
        R = int(rng.integers(0, 40))
        qlen = rng.integers(0, 5, R).astype(np.int32)
        seq = rng.integers(0, 9000, R).astype(np.int32)
        rows = int(qlen.sum()) + 2
        s0, e0 = O.decode_layout(seq, qlen, rows)
        s1, e1 = D.decode_layout_dcp(seq, qlen, rows, 0, 1, 7)
        assert np.array_equal(s0, s1) and np.array_equal(e0, e1)
        world, inter = int(rng.integers(2, 6)), int(rng.integers(1, 70))
        parts = [D.decode_layout_dcp(seq, qlen, rows, r, world, inter)[1].astype(np.int64) for r in range(world)]
        assert np.array_equal(sum(parts), e0)


def test_invalid_geometry():
    for rank, world, inter in ((2, 2, 1), (-1, 2, 1), (0, 2, 0)):
        with pytest.raises(ValueError):
            D.decode_layout_dcp(np.array([5], np.int32), np.array([1], np.int32), 1, rank, world, inter)


def test_merge_of_local_topks_is_the_global_topk():
    rng = np.random.default_rng(2)
    for trial in range(60):
        world = int(rng.integers(1, 6))
        inter = int(rng.choice([1, 4, 64]))
        rows = 3
        E = rng.integers(0, 2500, rows)
        k = int(rng.integers(1, 300))
        full = np.round(rng.standard_normal((rows, int(E.max(initial=1)) + 1)), 1).astype(np.float32)   # ties
        want = O.topk(full, E, k)
        # every rank: its own keys in local order, its local top-k with scores
        sc = np.full((rows, world, k), -np.inf, np.float32)
        ix = np.full((rows, world, k), -1, np.int32)
        for rank in range(world):
            n_loc = D.rank_local_ends(E, rank, world, inter)
            local = np.full((rows, int(n_loc.max(initial=0)) + 1), -np.inf, np.float32)
            for r in range(rows):
                g = D.local_to_global(np.arange(n_loc[r]), rank, world, inter)
                local[r, :n_loc[r]] = full[r, g]
            top = O.topk(local, n_loc, k)
            for r in range(rows):
                m = top[r] >= 0
                ix[r, rank, :m.sum()] = top[r][m]
                sc[r, rank, :m.sum()] = local[r, top[r][m]]
        got = D.topk_merge(sc, ix, world, inter, k)
        assert np.array_equal(got, want), trial
        # local slots: each selected key is reported by exactly its owner
        cover = np.zeros_like(got, dtype=np.int64)
        for rank in range(world):
            ls = D.local_slots(got, rank, world, inter)
            has = ls >= 0
            cover += has
            assert np.array_equal(D.local_to_global(ls[has], rank, world, inter), got[has])
        assert np.array_equal(cover, (got >= 0).astype(np.int64))
