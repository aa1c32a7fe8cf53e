"""DCP on CPU ranks (gloo): every rank scores only its own keys (rank-local
bounds from decode_layout's DCP branch), keeps its local top-k, the ranks
exchange their candidates with all_gather, and the merge equals the top-k of
the whole row; each rank then finds its local slots.  Oracle arithmetic on
the host; the exchange runs through a real process group."""

import os
import socket
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD, INTER, K = 3, 16, 64


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    rng = np.random.default_rng(11)
    R = 5
    qlen = rng.integers(1, 4, R).astype(np.int32)
    seq = rng.integers(100, 3000, R).astype(np.int32)
    rows = int(qlen.sum()) + 1                         # one padding row
    scores = np.round(rng.standard_normal((rows, 3000)), 2).astype(np.float32)
    return seq, qlen, rows, scores


def _rank_main(rank, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    from oracle import dcp as D
    from oracle import indexer as O
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        seq, qlen, rows, full = _problem()
        _, ends = D.decode_layout_dcp(seq, qlen, rows, rank, WORLD, INTER)
        local = np.full((rows, int(ends.max(initial=0)) + 1), -np.inf, np.float32)
        for r in range(rows):
            local[r, :ends[r]] = full[r, D.local_to_global(np.arange(ends[r]), rank, WORLD, INTER)]
        top = O.topk(local, ends, K)
        sc = np.where(top >= 0, np.take_along_axis(local, np.maximum(top, 0), 1), -np.inf).astype(np.float32)
        gs = [torch.empty((rows, K), dtype=torch.float32) for _ in range(WORLD)]
        gi = [torch.empty((rows, K), dtype=torch.int32) for _ in range(WORLD)]
        dist.all_gather(gs, torch.from_numpy(sc))
        dist.all_gather(gi, torch.from_numpy(top))
        merged = D.topk_merge(torch.stack(gs, 1).numpy(), torch.stack(gi, 1).numpy(), WORLD, INTER, K)
        q.put((rank, merged, D.local_slots(merged, rank, WORLD, INTER)))
    finally:
        dist.destroy_process_group()


def test_dcp_merge_on_three_gloo_ranks():
    import torch.multiprocessing as mp
    sys.path.insert(0, ROOT)
    from oracle import dcp as D
    from oracle import indexer as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, merged, slots = q.get(timeout=180)
        got[rank] = (merged, slots)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    seq, qlen, rows, full = _problem()
    _, ends = O.decode_layout(seq, qlen, rows)
    want = O.topk(full, ends, K)
    for rank in range(WORLD):
        merged, slots = got[rank]
        assert np.array_equal(merged, want)
        mine = slots >= 0
        assert np.array_equal(D.local_to_global(slots[mine], rank, WORLD, INTER), want[mine])
    # every selected key is some rank's local slot
    assert np.array_equal(sum((got[r][1] >= 0).astype(int) for r in range(WORLD)), (want >= 0).astype(int))
