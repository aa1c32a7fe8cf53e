"""The seeded workload recipe: the shapes and structure every test, the bench
and the oracle share (lengths in their ranges, block tables drawn as a
permutation of the page pool, the step's rows at the last positions of their
requests, padding rows and the one slot -1 of long_mxfp4)."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import make_workload  # noqa: E402
from synth.workloads import CONFIGS, PAGE  # noqa: E402


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_recipe_structure(name):
    spec = CONFIGS[name]
    wl = make_workload(name)
    assert wl.fmt == spec["fmt"] and wl.topk == spec["topk"] and wl.R == spec["R"]
    lo, hi = spec["seq"]
    assert np.all((wl.seq_lens >= lo) & (wl.seq_lens <= hi))
    qlo, qhi = spec["qlen"]
    assert np.all((wl.query_lens >= qlo) & (wl.query_lens <= qhi))
    real = int(wl.query_lens.sum())
    assert wl.num_rows == real + spec["pad_rows"]

    # block table: each request's ceil(seq/64) pages, all pages of the pool exactly once
    pages = [(int(s) + PAGE - 1) // PAGE for s in wl.seq_lens]
    assert wl.num_pages == sum(pages) and wl.max_pages == max(pages)
    used = np.concatenate([wl.block_table[q, :n] for q, n in enumerate(pages)])
    assert np.array_equal(np.sort(used), np.arange(wl.num_pages))
    for q, n in enumerate(pages):
        assert np.all(wl.block_table[q, n:] == -1)

    # rows: request order, each request's rows at its last query_len positions
    r = 0
    for q in range(wl.R):
        for i in range(int(wl.query_lens[q])):
            assert wl.row_request[r] == q
            assert wl.row_position[r] == int(wl.seq_lens[q]) - int(wl.query_lens[q]) + i
            r += 1
    assert np.all(wl.row_request[real:] == -1) and np.all(wl.step_slots[real:] == -1)

    # the step's new keys go to the slots of their positions (except the rows named in the recipe)
    for r in range(real):
        q, t = int(wl.row_request[r]), int(wl.row_position[r])
        want = -1 if q in spec["no_slot_rows"] else int(wl.block_table[q, t // PAGE]) * PAGE + t % PAGE
        assert wl.step_slots[r] == want

    # prefill covers positions 0 .. seq - qlen - 1 of each request, at their own slots
    for q in range(min(wl.R, 3)):
        bits, slots = wl.prefill(q)
        n = int(wl.seq_lens[q]) - int(wl.query_lens[q])
        assert bits.shape == (n, 128) and slots.shape == (n,)
        t = np.arange(n)
        assert np.array_equal(slots, wl.block_table[q, t // PAGE].astype(np.int64) * PAGE + t % PAGE)


def test_long_mxfp4_has_one_padding_slot():
    wl = make_workload("long_mxfp4")
    assert int((wl.step_slots < 0).sum()) == 1 and wl.step_slots[7] == -1


def test_same_seed_same_inputs_and_overrides_apply():
    a, b = make_workload("spec_verify"), make_workload("spec_verify")
    assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.prefill(5)[0], b.prefill(5)[0])
    c = make_workload("spec_verify", fmt="mxfp4_rg", seed=9)
    assert c.fmt == "mxfp4_rg" and not np.array_equal(c.q_bits, a.q_bits)


def test_values_are_bf16_patterns_of_the_stated_draws():
    """q, wv and the key projections are BF16 bit patterns of N(0, 1) draws;
    mxfp4_decode scales about 1 % of its query elements by 20."""
    from synth import bf16_bits_to_f32
    wl = make_workload("fp8_decode")
    q = bf16_bits_to_f32(wl.q_bits).ravel()
    assert abs(float(q.mean())) < 0.01 and abs(float(q.std()) - 1.0) < 0.01
    big = np.abs(bf16_bits_to_f32(make_workload("mxfp4_decode").q_bits)).ravel()
    share = float((big > 6.0).mean())   # |N(0,1)| > 6 is ~2e-9; x20 outliers exceed 6 about 77 % of the time
    assert 0.005 < share < 0.01


@pytest.mark.parametrize("name,unique,scored,rows", [
    ("fp8_decode", 393_216, 393_216, 64),            # 64 x mean(U[4096, 8192])
    ("mxfp4_decode", 1_572_864, 1_572_864, 64),      # 64 x mean(U[16384, 32768])
    ("spec_verify", 4_456_448, 11_141_120, 324),     # 128 x mean(U[4096, 65536]); 2.5 rows a request + 4 padding
    ("long_mxfp4", 1_048_576, 1_048_576, 8),         # 8 x 131072
])
def test_sizes_are_those_of_the_stated_configurations(name, unique, scored, rows):
    """Keys read (the requests' lengths), keys scored (each row to its own
    causal bound) and rows come out within 5 % of the configurations'
    expected sizes."""
    wl = make_workload(name)
    got_scored = sum(int(wl.seq_lens[q]) - int(wl.query_lens[q]) + i + 1
                     for q in range(wl.R) for i in range(int(wl.query_lens[q])))
    assert abs(int(wl.seq_lens.sum()) / unique - 1) < 0.05
    assert abs(got_scored / scored - 1) < 0.05
    assert abs(wl.num_rows / rows - 1) < 0.05
