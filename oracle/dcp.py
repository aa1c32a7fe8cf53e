"""Plain CPU oracle of the decode-context-parallel (DCP) pieces of the step.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA path.

Page *amd.ops.fp4_indexer*, ``decode_layout`` (its ``dcp_world_size > 1``
branch): the key space of a request is dealt out to D ranks in runs of I
(``interleave``) consecutive positions, run n going to rank n mod D; each
rank scores only its own keys, numbered consecutively in rank-local space,
so a row's global bound E becomes the number of its keys below E.

Page *cutedsl.dsa.overlap*: under DCP the indexer path ends with "the top-k
merge and the local slots".  The merge is not printed; the reading taken
here is the plain one: every rank contributes its local top-k
candidates (score, rank-local position), the k best of all of them by
(score desc, global position asc) are the row's top-k, and a rank's local
slots are the rank-local positions of the selected keys it owns.
"""

from __future__ import annotations

import numpy as np

from .indexer import decode_layout


def owner(t, world: int, interleave: int):
    """Rank that holds global key position t: run t // I goes to rank (t // I) mod D."""
    return (np.asarray(t, np.int64) // interleave) % world


def global_to_local(t, world: int, interleave: int):
    """Rank-local position of global key t on its owner: its runs are numbered
    consecutively, (t // (D I)) full rounds of I keys before it, plus t mod I."""
    t = np.asarray(t, np.int64)
    return (t // (world * interleave)) * interleave + t % interleave


def local_to_global(l, rank: int, world: int, interleave: int):
    """Global position of rank-local key l of ``rank`` (inverse of global_to_local)."""
    l = np.asarray(l, np.int64)
    return (l // interleave) * (world * interleave) + rank * interleave + l % interleave


def rank_local_ends(ends, rank: int, world: int, interleave: int) -> np.ndarray:
    """The DCP branch of ``decode_layout``: full = E // (D I) * I keys come from
    complete rounds; the partial round gives the rank min(I, max(0, E - full D - r I))
    more."""
    e = np.asarray(ends, np.int64)
    full = e // (world * interleave) * interleave
    return (full + np.clip(e - full * world - rank * interleave, 0, interleave)).astype(np.int32)


def decode_layout_dcp(seq_lens, query_lens, num_rows: int, rank: int, world: int, interleave: int):
    """``decode_layout`` with the DCP geometry: starts as without DCP, row bounds
    in rank-local key space, padding rows 0."""
    if not (0 <= rank < world) or interleave < 1 or num_rows < 0:
        raise ValueError("Invalid DCP geometry or query row count")
    starts, ends = decode_layout(seq_lens, query_lens, num_rows)
    if world > 1:
        ends = rank_local_ends(ends, rank, world, interleave)
    return starts, ends


def topk_merge(scores, idx, world: int, interleave: int, k_out: int) -> np.ndarray:
    """scores FP32 [rows, world, k], idx int32 [rows, world, k] (rank w's
    candidates, rank-local positions, -1 empty) -> int32 [rows, k_out] global
    positions ordered by (score desc, global position asc), -1 filled."""
    scores = np.asarray(scores, np.float64)
    idx = np.asarray(idx, np.int64)
    rows = scores.shape[0]
    out = np.full((rows, k_out), -1, np.int32)
    ranks = np.broadcast_to(np.arange(world)[None, :, None], idx.shape)
    for r in range(rows):
        keep = idx[r] >= 0
        g = local_to_global(idx[r][keep], 0, world, interleave) + ranks[r][keep] * interleave
        s = scores[r][keep]
        order = np.lexsort((g, -s))
        m = min(k_out, order.size)
        out[r, :m] = g[order[:m]]
    return out


def local_slots(global_idx, rank: int, world: int, interleave: int) -> np.ndarray:
    """Rank-local positions of the selected keys that ``rank`` owns, -1 elsewhere."""
    g = np.asarray(global_idx, np.int64)
    mine = (g >= 0) & (owner(np.maximum(g, 0), world, interleave) == rank)
    return np.where(mine, global_to_local(np.maximum(g, 0), world, interleave), -1).astype(np.int32)
