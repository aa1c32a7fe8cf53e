"""Glue between the seeded workloads, the CUDA path and the oracle for tests.

The GPU side and the oracle side each build their own cache from the same
raw inputs; nothing computed by one side is fed to the other.
"""

from __future__ import annotations

import numpy as np

from synth import Workload, bf16_bits_to_f32

TOL_REL, TOL_ABS = 1e-3, 1e-4


def bf16_tensor(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def gpu_run(wl: Workload, want_logits=True, device="cuda", page_stride=None):
    """Prefill + one decode step on the GPU.  Returns a dict of numpy arrays."""
    import torch
    from sparse_attention_indexer_score_gb300.step import DecodeIndexer

    dev = torch.device(device)
    ix = DecodeIndexer(wl.fmt, wl.num_pages, torch.from_numpy(wl.block_table), torch.from_numpy(wl.gamma),
                       torch.from_numpy(wl.beta), wl.eps, wl.num_rows, wl.topk, dev, page_stride=page_stride)
    for q in range(wl.R):
        kb, sl = wl.prefill(q)
        if kb.shape[0]:
            ix.insert(bf16_tensor(kb, dev), torch.from_numpy(sl).to(dev))
    out = ix.step(bf16_tensor(wl.q_bits, dev), bf16_tensor(wl.wv_bits, dev), bf16_tensor(wl.step_key_bits, dev),
                  torch.from_numpy(wl.step_slots).to(dev), torch.from_numpy(wl.seq_lens).to(dev),
                  torch.from_numpy(wl.query_lens).to(dev), int(wl.query_lens.max(initial=0)),
                  want_logits=want_logits)
    torch.cuda.synchronize()
    res = dict(
        q_rows=out.q_rows.cpu().numpy(), w=out.w.float().cpu().numpy(), starts=out.starts.cpu().numpy(),
        row_ends=out.row_ends.cpu().numpy(), topk=out.topk.cpu().numpy() if out.topk is not None else None,
        logits=out.logits.cpu().numpy() if out.logits is not None else None, status=ix.status_bits(),
        cache=ix.cache, page_stride=ix.page_stride)
    return res


def oracle_run(wl: Workload, rows=None, page_stride=None):
    """The oracle's step for the requests of `rows` (all rows when None)."""
    from oracle import indexer as O

    fmt = wl.fmt
    q = bf16_bits_to_f32(wl.q_bits)
    wv = bf16_bits_to_f32(wl.wv_bits)
    q_rows, w = O.quantize_query(fmt, q, wv)
    starts, row_ends = O.decode_layout(wl.seq_lens, wl.query_lens, wl.num_rows)
    rows = list(range(wl.num_rows)) if rows is None else list(rows)
    reqs = sorted({int(wl.row_request[r]) for r in rows if wl.row_request[r] >= 0})
    stride = int(page_stride or O.page_bytes(fmt))
    # compact cache holding only the pages of the requests involved
    remap = {}
    for qq in reqs:
        n = (int(wl.seq_lens[qq]) + 63) // 64
        for p in wl.block_table[qq, :n]:
            remap[int(p)] = len(remap)
    cache = np.zeros(max(1, len(remap)) * stride, np.uint8)
    bt = np.full_like(wl.block_table, -1)
    for qq in reqs:
        n = (int(wl.seq_lens[qq]) + 63) // 64
        bt[qq, :n] = [remap[int(p)] for p in wl.block_table[qq, :n]]
    for qq in reqs:
        kb, sl = wl.prefill(qq)
        pages = sl // 64
        sl2 = np.array([remap[int(p)] for p in pages], dtype=np.int64) * 64 + sl % 64 if len(sl) else sl
        O.insert_key(fmt, cache, stride, len(remap), bf16_bits_to_f32(kb), wl.gamma, wl.beta, wl.eps, sl2)
    step_rows = [r for r in range(wl.num_rows) if wl.row_request[r] in reqs and wl.step_slots[r] >= 0]
    if step_rows:
        ss = wl.step_slots[step_rows]
        sl2 = np.array([remap[int(s // 64)] * 64 + int(s % 64) for s in ss], dtype=np.int64)
        O.insert_key(fmt, cache, stride, len(remap), bf16_bits_to_f32(wl.step_key_bits[step_rows]), wl.gamma,
                     wl.beta, wl.eps, sl2)
    scores = O.score_paged(fmt, q_rows, w, cache, stride, bt, starts, row_ends, rows_subset=rows)
    top = O.topk(scores, row_ends, wl.topk)
    return dict(q_rows=q_rows, w=w, starts=starts, row_ends=row_ends, scores=scores, topk=top, rows=rows,
                remap=remap, cache=cache)


def _oracle_chunk(job):
    """Worker of ``oracle_rows``: the oracle's scores and top-k of some rows."""
    from synth import make_workload
    name, overrides, rows, page_stride = job
    o = oracle_run(make_workload(name, **overrides), rows=rows, page_stride=page_stride)
    rows = list(rows)
    return rows, o["scores"][rows], o["topk"][rows], o["row_ends"], o["starts"], o["q_rows"]


def oracle_rows(name, overrides, rows, page_stride=None, workers=None):
    """``oracle_run`` of a named workload over ``rows``, the requests split
    over spawned worker processes (each rebuilds the workload from its seed).
    Returns (scores {row: float64 [width]}, topk {row: int32 [k]}, row_ends,
    starts, q_rows)."""
    import multiprocessing as mp
    import os
    from synth import make_workload
    wl = make_workload(name, **overrides)
    by_req = {}
    for r in rows:
        by_req.setdefault(int(wl.row_request[r]), []).append(int(r))
    groups = list(by_req.values())
    workers = workers or max(1, min(len(groups), (os.cpu_count() or 2) - 1, 16))
    chunks = [[] for _ in range(workers)]
    for i, g in enumerate(sorted(groups, key=lambda g: -int(wl.seq_lens[wl.row_request[g[0]]]) if
                                 wl.row_request[g[0]] >= 0 else 0)):
        chunks[i % workers] += g
    jobs = [(name, overrides, sorted(c), page_stride) for c in chunks if c]
    ctx = mp.get_context("spawn")
    scores, top = {}, {}
    row_ends = starts = q_rows = None
    with ctx.Pool(len(jobs)) as pool:
        for rs, sc, tk, re_, st, qr in pool.imap_unordered(_oracle_chunk, jobs):
            for i, r in enumerate(rs):
                scores[r], top[r] = sc[i], tk[i]
            row_ends, starts, q_rows = re_, st, qr
    return scores, top, row_ends, starts, q_rows


def check_logits(got: np.ndarray, want: np.ndarray, row_ends, rows):
    """|got - want| <= max(1e-3 |want|, 1e-4) on every valid position; -inf past the bound."""
    for r in rows:
        n = int(row_ends[r])
        g = got[r, :n].astype(np.float64)
        o = want[r, :n]
        tol = np.maximum(TOL_REL * np.abs(o), TOL_ABS)
        bad = np.abs(g - o) > tol
        assert not bad.any(), (r, np.nonzero(bad)[0][:5], g[bad][:5], o[bad][:5])
        assert np.all(np.isneginf(got[r, n:])), r


def check_topk(got: np.ndarray, want_scores: np.ndarray, row_ends, k, rows):
    """Top-k sets identical except for positions whose oracle score lies within
    the logits tolerance of the k-th oracle score; every index valid and distinct."""
    for r in rows:
        n = int(row_ends[r])
        g = got[r]
        if n <= k:
            assert list(g[:n]) == list(range(n)) and np.all(g[n:] == -1), r
            continue
        assert np.all((g >= 0) & (g < n)), r
        assert len(set(g.tolist())) == k, r
        s = want_scores[r, :n]
        order = np.lexsort((np.arange(n), -s))
        want = set(order[:k].tolist())
        kth = s[order[k - 1]]
        tol = max(TOL_REL * abs(kth), TOL_ABS)
        for t in set(g.tolist()) ^ want:
            assert abs(s[t] - kth) <= tol, (r, t, s[t], kth)
