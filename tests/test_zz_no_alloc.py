"""The no-allocation top-k entry point against the workspace one.

``dsa_topk_noalloc`` is for callers that cannot allocate device memory when
they call the library (an engine that reserved its HBM up front, a plugin host
without an allocator); it keeps its scratch in a static device array.  This
file runs last so that a run stopping at the first failure has already run
every other test; it passes alone in a fresh process as well.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _scores(rng, rows, width):
    x = np.round(rng.standard_normal((rows, width)), 2).astype(np.float32)   # ties at the boundary
    x[0, :] = 0.5                                                            # one row of equal values
    return x


def test_topk_noalloc_matches_workspace_topk_twice(cuda_lib):
    import torch
    dsa = cuda_lib
    L = dsa.lib()
    rng = np.random.default_rng(21)
    rows, width, k = dsa.TOPK_NOALLOC_MAX_ROWS, 30000, 2048
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):                                   # two calls in a row share the static scratch
        logits = torch.from_numpy(_scores(rng, rows, width)).cuda()
        ends = rng.integers(0, width + 1, rows).astype(np.int32)
        ends[1], ends[2], ends[3] = width, 0, k            # full row, empty row, exactly k
        ends_t = torch.from_numpy(ends).cuda()
        out = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
        rc = L.dsa_topk_noalloc(logits.data_ptr(), logits.stride(0), ends_t.data_ptr(), rows, width, k,
                                out.data_ptr(), stream)
        assert rc == 0
        ref = dsa.topk(logits, ends_t, k)                   # the workspace entry point
        torch.cuda.synchronize()
        got, want, vals = out.cpu().numpy(), ref.cpu().numpy(), logits.cpu().numpy()
        for r in range(rows):
            n = int(ends[r])
            if n <= k:
                assert np.array_equal(got[r], want[r]), (call, r)
                continue
            assert len(set(got[r].tolist())) == k and np.all((got[r] >= 0) & (got[r] < n)), (call, r)
            # equal sets up to ties at the k-th value: the selected values agree exactly
            assert np.array_equal(np.sort(vals[r, got[r]]), np.sort(vals[r, want[r]])), (call, r)


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
