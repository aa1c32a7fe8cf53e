"""The no-allocation top-k entry point against the workspace one.

``dsa_topk_noalloc`` is for callers that cannot allocate device memory when
they call the library (an engine that reserved its HBM up front, a plugin host
without an allocator); it keeps its scratch in a static device array.  This
file runs last so that a run stopping at the first failure has already run
every other test; it passes alone in a fresh process as well.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _scores(rng, rows, width):
    x = np.round(rng.standard_normal((rows, width)), 2).astype(np.float32)   # ties at the boundary
    x[0, :] = 0.5                                                            # one row of equal values
    return x


def _check_against_both(got, want, vals, ends, k, tag):
    """Rows with at most k entries list 0..n-1 then -1 exactly; longer rows
    hold k distinct valid positions whose values are those of the workspace
    entry point's set and of the oracle's top k (ties at the k-th value may
    pick different positions, never different values)."""
    from oracle import indexer as O
    ref = O.topk(vals, ends, k)
    for r in range(got.shape[0]):
        n = int(ends[r])
        if n <= k:
            assert np.array_equal(got[r], want[r]), (tag, r)
            assert list(got[r, :n]) == list(range(n)) and np.all(got[r, n:] == -1), (tag, r)
            continue
        assert len(set(got[r].tolist())) == k and np.all((got[r] >= 0) & (got[r] < n)), (tag, r)
        sel = np.sort(vals[r, got[r]])
        assert np.array_equal(sel, np.sort(vals[r, want[r]])), (tag, r)
        assert np.array_equal(sel, np.sort(vals[r, ref[r]])), (tag, r)


def _call(dsa, logits, ends_t, k):
    import torch
    rows, width = logits.shape
    out = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    rc = dsa.lib().dsa_topk_noalloc(logits.data_ptr(), logits.stride(0), ends_t.data_ptr(), rows, width, k,
                                    out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    return out


def test_topk_noalloc_matches_workspace_topk_twice(cuda_lib):
    import torch
    dsa = cuda_lib
    rng = np.random.default_rng(21)
    rows, width, k = dsa.TOPK_NOALLOC_MAX_ROWS, 30000, 2048
    for call in range(2):                                   # two calls in a row share the static scratch
        vals = _scores(rng, rows, width)
        logits = torch.from_numpy(vals).cuda()
        ends = rng.integers(0, width + 1, rows).astype(np.int32)
        ends[1], ends[2], ends[3] = width, 0, k            # full row, empty row, exactly k
        ends_t = torch.from_numpy(ends).cuda()
        out = _call(dsa, logits, ends_t, k)
        ref = dsa.topk(logits, ends_t, k)                   # the workspace entry point
        torch.cuda.synchronize()
        _check_against_both(out.cpu().numpy(), ref.cpu().numpy(), vals, ends, k, call)


def test_topk_noalloc_more_winners_than_shared_memory_holds(cuda_lib):
    """k = 5000 is past the 4096 winners a CTA buffers on chip: split rows
    place winners straight through the shared counters of the static array."""
    import torch
    dsa = cuda_lib
    rng = np.random.default_rng(22)
    rows, width, k = 6, 40000, 5000
    vals = _scores(rng, rows, width)
    ends = np.array([width, 39000, 5000, 4999, 20000, 0], np.int32)
    logits, ends_t = torch.from_numpy(vals).cuda(), torch.from_numpy(ends).cuda()
    out = _call(dsa, logits, ends_t, k)
    ref = dsa.topk(logits, ends_t, k)
    torch.cuda.synchronize()
    _check_against_both(out.cpu().numpy(), ref.cpu().numpy(), vals, ends, k, "k5000")


def test_topk_noalloc_few_rows_after_many(cuda_lib):
    """A 3-row call right after a 64-row one: each call clears only its own
    rows' histograms and counters, which must be enough."""
    import torch
    dsa = cuda_lib
    rng = np.random.default_rng(23)
    width, k = 30000, 2048
    for rows in (dsa.TOPK_NOALLOC_MAX_ROWS, 3):
        vals = _scores(rng, rows, width)
        ends = np.full(rows, width, np.int32)
        logits, ends_t = torch.from_numpy(vals).cuda(), torch.from_numpy(ends).cuda()
        out = _call(dsa, logits, ends_t, k)
        ref = dsa.topk(logits, ends_t, k)
        torch.cuda.synchronize()
        _check_against_both(out.cpu().numpy(), ref.cpu().numpy(), vals, ends, k, rows)


def test_topk_noalloc_rejects_too_many_rows(cuda_lib):
    import torch
    L = cuda_lib.lib()
    rows = cuda_lib.TOPK_NOALLOC_MAX_ROWS + 1
    logits = torch.zeros((rows, 64), dtype=torch.float32, device="cuda")
    ends = torch.full((rows,), 64, dtype=torch.int32, device="cuda")
    out = torch.empty((rows, 8), dtype=torch.int32, device="cuda")
    rc = L.dsa_topk_noalloc(logits.data_ptr(), 64, ends.data_ptr(), rows, 64, 8, out.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    assert rc == -2
    with pytest.raises(ValueError):
        cuda_lib.topk_noalloc(logits, ends, 8)
