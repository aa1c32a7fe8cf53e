"""DCP on GB300 through the C ABI: rank-local row bounds bit-exact against the
oracle, and the top-k merge against the oracle's merge (page
*amd.ops.fp4_indexer* ``decode_layout``; page *cutedsl.dsa.overlap*)."""

import numpy as np
import pytest

from oracle import dcp as D
from oracle import indexer as O

pytestmark = pytest.mark.gpu


def test_decode_layout_dcp_bit_exact(cuda_lib):
    import torch
    rng = np.random.default_rng(0)
    for _ in range(60):
        R = int(rng.integers(0, 600))
        qlen = rng.integers(0, 5, R).astype(np.int32)
        seq = rng.integers(0, 200000, R + int(rng.integers(0, 3))).astype(np.int32)
        rows = int(qlen.sum()) + int(rng.integers(0, 4))
        world = int(rng.integers(1, 9))
        rank = int(rng.integers(0, world))
        inter = int(rng.choice([1, 2, 64, 4096]))
        st, en = cuda_lib.decode_layout_dcp(torch.from_numpy(seq).cuda(), torch.from_numpy(qlen).cuda(), rows,
                                            rank, world, inter)
        ws, we = D.decode_layout_dcp(seq, qlen, rows, rank, world, inter)
        assert np.array_equal(st.cpu().numpy(), ws) and np.array_equal(en.cpu().numpy(), we)


def _candidates(rng, rows, world, inter, k, width):
    full = np.round(rng.standard_normal((rows, width)), 2).astype(np.float32)
    E = rng.integers(0, width + 1, rows)
    sc = np.full((rows, world, k), -np.inf, np.float32)
    ix = np.full((rows, world, k), -1, np.int32)
    for rank in range(world):
        n_loc = D.rank_local_ends(E, rank, world, inter)
        local = np.full((rows, int(n_loc.max(initial=0)) + 1), -np.inf, np.float32)
        for r in range(rows):
            local[r, :n_loc[r]] = full[r, D.local_to_global(np.arange(n_loc[r]), rank, world, inter)]
        top = O.topk(local, n_loc, k)
        for r in range(rows):
            m = top[r] >= 0
            ix[r, rank, :m.sum()] = top[r][m]
            sc[r, rank, :m.sum()] = local[r, top[r][m]]
    return full, E, sc, ix


@pytest.mark.parametrize("world,inter,k,k_out", [(1, 1, 64, 64), (2, 64, 2048, 2048), (4, 16, 512, 300),
                                                  (3, 1, 40, 100), (8, 4, 1024, 2048)])
def test_topk_merge(cuda_lib, world, inter, k, k_out):
    import torch
    rng = np.random.default_rng(world * 100 + k)
    rows, width = 6, 9000
    full, E, sc, ix = _candidates(rng, rows, world, inter, k, width)
    want = D.topk_merge(sc, ix, world, inter, k_out)
    rank = world - 1
    got, loc = cuda_lib.topk_merge(torch.from_numpy(sc.reshape(rows, world * k)).cuda(),
                                   torch.from_numpy(ix.reshape(rows, world * k)).cuda(), world, k, inter, k_out,
                                   rank=rank)
    got, loc = got.cpu().numpy(), loc.cpu().numpy()
    for r in range(rows):
        w = want[r][want[r] >= 0]
        g = got[r][got[r] >= 0]
        assert len(set(g.tolist())) == g.size == w.size, r
        assert np.all(g < E[r])
        # the selected scores are the same multiset (ties at the boundary are exchangeable)
        assert np.array_equal(np.sort(full[r, g]), np.sort(full[r, w])), r
        mine = loc[r] >= 0
        assert np.array_equal(D.local_to_global(loc[r][mine], rank, world, inter), got[r][mine])
        owned = (got[r] >= 0) & (D.owner(np.maximum(got[r], 0), world, inter) == rank)
        assert np.array_equal(mine, owned)


def test_topk_merge_argument_errors(cuda_lib):
    import torch
    lib = cuda_lib.lib()
    s = torch.cuda.current_stream().cuda_stream
    ws = cuda_lib.new_workspace(cuda_lib.topk_workspace_size(2, 8), "cuda")
    sc = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    ix = torch.zeros((2, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((2, 8), dtype=torch.int32, device="cuda")
    args = lambda world, k, inter, ld, rank, local: (sc.data_ptr(), ld, ix.data_ptr(), ld, 2, world, k, inter, 8,
                                                     out.data_ptr(), rank, local, ws.data_ptr(), ws.numel(), s)
    assert lib.dsa_topk_merge(*args(2, 8, 1, 16, 0, None)) == 0
    assert lib.dsa_topk_merge(*args(0, 8, 1, 16, 0, None)) == -1      # world < 1
    assert lib.dsa_topk_merge(*args(2, 8, 0, 16, 0, None)) == -1      # interleave < 1
    assert lib.dsa_topk_merge(*args(2, 8, 1, 15, 0, None)) == -1      # leading dimension too short
    assert lib.dsa_topk_merge(*args(2, 8, 1, 16, 2, out.data_ptr())) == -1   # rank outside the world
    assert lib.dsa_decode_layout_dcp(None, 0, None, 0, 1, 2, 2, 1, out.data_ptr(), out.data_ptr(), s) == -1
