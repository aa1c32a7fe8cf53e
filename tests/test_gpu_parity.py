"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on GB300."""

import numpy as np
import pytest

from dsa_case import bf16_tensor, check_logits, check_topk, gpu_run, oracle_rows, oracle_run
from oracle import indexer as O
from synth import bf16_bits_to_f32, make_workload

pytestmark = pytest.mark.gpu
FMTS = ["fp8", "fp8_mx", "mxfp4", "mxfp4_rg"]


def _used(fmt):
    """Bytes of a quantised query row that carry data (row-group: 4 x 64 scale slots)."""
    return {"mxfp4": 2176, "mxfp4_rg": 2304}.get(fmt, 4096)


def _special_queries(rng, rows):
    q = rng.standard_normal((rows, 32, 128)).astype(np.float32)
    q[0, 0] = 0.0                                   # all-zero head: amax floor
    q[0, 1] = 1e-12                                 # below the FP8 amax floor
    q[0, 2] *= 1e30                                 # huge
    q[0, 3, ::7] *= 40.0                            # outliers
    q[0, 4] = -0.0
    q[0, 5, :32] = 0.0                              # one all-zero MXFP4 block
    q[0, 6] = np.float32(448.0) * np.sign(q[0, 6])  # on the FP8 saturation point
    q[0, 7, :] = np.float32(6.0)
    q[1] *= np.float32(2.0 ** -100)                 # tiny but normal
    u = q.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_query_bit_exact(cuda_lib, fmt):
    import torch
    rng = np.random.default_rng(1)
    rows = 37
    qb = _special_queries(rng, rows)
    wvb = ((rng.standard_normal((rows, 32)).astype(np.float32).view(np.uint32) >> 16)).astype(np.uint16)
    q_rows, w = cuda_lib.quantize_query(fmt, bf16_tensor(qb, "cuda"), bf16_tensor(wvb, "cuda"))
    want_rows, want_w = O.quantize_query(fmt, bf16_bits_to_f32(qb), bf16_bits_to_f32(wvb))
    used = _used(fmt)
    got = q_rows.cpu().numpy()
    assert np.array_equal(got[:, :used], want_rows[:, :used])
    assert not got[:, used:].any()
    assert np.array_equal(w.float().cpu().numpy(), want_w)


@pytest.mark.parametrize("heads", [16, 32, 64])
def test_quantize_queries_rg_bit_exact(cuda_lib, heads):
    """Page "amd.ops.fp4_indexer", quantize_queries: payload and row-group
    scales equal the oracle's byte for byte, in a strided input view."""
    import torch
    rng = np.random.default_rng(10 + heads)
    rows = 29
    x = rng.standard_normal((rows, heads, 128)).astype(np.float32)
    x[0, 0] = 0.0
    x[0, 1, :32] = 0.0
    x[0, 2] *= 1e30
    x[1] *= np.float32(2.0 ** -100)
    x[2, :, ::5] = -0.0
    u = x.view(np.uint32).astype(np.uint64)
    qb = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    big = torch.zeros((rows, heads, 160), dtype=torch.bfloat16, device="cuda")   # head stride 160
    big[:, :, :128] = bf16_tensor(qb, "cuda")
    payload, scales = cuda_lib.quantize_queries_rg(big[:, :, :128])
    want_p, want_s = O.quantize_queries(bf16_bits_to_f32(qb))
    assert np.array_equal(payload.cpu().numpy(), want_p)
    assert np.array_equal(scales.cpu().numpy(), want_s)


@pytest.mark.parametrize("fmt", FMTS)
def test_insert_key_bit_exact(cuda_lib, fmt):
    import torch
    rng = np.random.default_rng(2)
    n, num_pages = 300, 6
    x = (rng.standard_normal((n, 128)) * 2.0).astype(np.float32)
    x[0] = 3.25                                   # zero variance
    x[1, ::2] = 1e20                              # huge spread
    x[2] = 0.0
    x[3, :32] *= 1e-30
    kb = ((x.view(np.uint32).astype(np.uint64) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    gamma = bf16_bits_to_f32(((1 + 0.1 * rng.standard_normal(128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    beta = bf16_bits_to_f32(((0.1 * rng.standard_normal(128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    slots = rng.permutation(num_pages * 64)[:n].astype(np.int64)
    slots[5] = -1
    slots[6] = num_pages * 64 + 3                 # past the pool
    stride = O.page_bytes(fmt) + 64               # physical stride above the section size
    cache = torch.zeros(num_pages * stride, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.insert_key(fmt, bf16_tensor(kb, "cuda"), torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda(),
                        1e-6, torch.from_numpy(slots).cuda(), cache, stride, num_pages, status)
    want = np.zeros(num_pages * stride, np.uint8)
    bad = O.insert_key(fmt, want, stride, num_pages, bf16_bits_to_f32(kb), gamma, beta, 1e-6, slots)
    assert bad == 1
    got = cache.cpu().numpy()
    diff = np.nonzero(got != want)[0]
    assert diff.size == 0, (diff[:10], got[diff[:10]], want[diff[:10]])
    assert int(status.item()) & 1


def test_decode_layout_parity(cuda_lib):
    import json, os, torch
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "decode_layout.json")))
    cases = [(np.array(c["seq_lens"], np.int32), np.array(c["query_lens"], np.int32), c["num_rows"])
             for c in g["cases"]]
    rng = np.random.default_rng(4)
    for _ in range(40):
        R = int(rng.integers(0, 3000))
        qlen = rng.integers(0, 6, R).astype(np.int32)
        seq = rng.integers(0, 70000, R + int(rng.integers(0, 3))).astype(np.int32)
        cases.append((seq, qlen, int(qlen.sum()) + int(rng.integers(0, 5))))
    for seq, qlen, num_rows in cases:
        st, en = cuda_lib.decode_layout(torch.from_numpy(seq).cuda(), torch.from_numpy(qlen).cuda(), num_rows)
        ws, we = O.decode_layout(seq, qlen, num_rows)
        assert np.array_equal(st.cpu().numpy(), ws) and np.array_equal(en.cpu().numpy(), we)


@pytest.mark.parametrize("fmt", FMTS)
def test_prepare_step_bit_exact(cuda_lib, fmt):
    """The fused launch equals the oracle's quantize_query, insert_key and
    decode_layout, and the three separate calls, byte for byte."""
    import torch
    rng = np.random.default_rng(6)
    rows, n, num_pages = 41, 57, 5
    qb = _special_queries(rng, rows)
    wvb = ((rng.standard_normal((rows, 32)).astype(np.float32).view(np.uint32) >> 16)).astype(np.uint16)
    x = (rng.standard_normal((n, 128)) * 3.0).astype(np.float32)
    x[0] = -1.5                                   # zero variance
    kb = ((x.view(np.uint32).astype(np.uint64) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    gamma = (1 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    beta = (0.1 * rng.standard_normal(128)).astype(np.float32)
    slots = rng.permutation(num_pages * 64)[:n].astype(np.int64)
    slots[3] = -1                                 # padding
    slots[4] = num_pages * 64                     # past the pool
    R = 17
    qlen = rng.integers(0, 4, R).astype(np.int32)
    seq = rng.integers(0, 9000, R + 2).astype(np.int32)
    num_rows = int(qlen.sum()) + 3                # three padding rows
    stride = O.page_bytes(fmt) + 32
    dev = "cuda"

    def run(fused):
        cache = torch.zeros(num_pages * stride, dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        args = (bf16_tensor(qb, dev), bf16_tensor(wvb, dev))
        kargs = (bf16_tensor(kb, dev), torch.from_numpy(gamma).to(dev), torch.from_numpy(beta).to(dev), 1e-6,
                 torch.from_numpy(slots).to(dev))
        lens = (torch.from_numpy(seq).to(dev), torch.from_numpy(qlen).to(dev))
        if fused:
            q_rows, w, st, en = cuda_lib.prepare_step(fmt, *args, kargs[0], kargs[1], kargs[2], kargs[3], kargs[4],
                                                      cache, stride, num_pages, *lens, num_rows, status=status)
        else:
            q_rows, w = cuda_lib.quantize_query(fmt, *args)
            cuda_lib.insert_key(fmt, *kargs, cache, stride, num_pages, status)
            st, en = cuda_lib.decode_layout(*lens, num_rows)
        torch.cuda.synchronize()
        return [t.cpu().numpy() for t in (q_rows, w.float(), cache, st, en, status)]

    fused, separate = run(True), run(False)
    for a, b in zip(fused, separate):
        assert np.array_equal(a, b)
    want_rows, want_w = O.quantize_query(fmt, bf16_bits_to_f32(qb), bf16_bits_to_f32(wvb))
    used = _used(fmt)
    assert np.array_equal(fused[0][:, :used], want_rows[:, :used]) and not fused[0][:, used:].any()
    assert np.array_equal(fused[1], want_w)
    want_cache = np.zeros(num_pages * stride, np.uint8)
    bad = O.insert_key(fmt, want_cache, stride, num_pages, bf16_bits_to_f32(kb), gamma, beta, 1e-6, slots)
    assert bad == 1 and np.array_equal(fused[2], want_cache) and int(fused[5][0]) & 1
    ws, we = O.decode_layout(seq, qlen, num_rows)
    assert np.array_equal(fused[3], ws) and np.array_equal(fused[4], we)


SMALL = [
    dict(R=2, seq=(256, 256), qlen=(1, 1)),
    dict(R=5, seq=(100, 700), qlen=(1, 1)),
    dict(R=7, seq=(60, 400), qlen=(1, 6), pad_rows=3),      # segments of more than 4 rows
    dict(R=4, seq=(127, 130), qlen=(2, 4), pad_rows=1),     # ragged tails around one tile
    dict(R=3, seq=(1, 3), qlen=(1, 3)),                      # bounds of 0..3 keys
    dict(R=9, seq=(2000, 5000), qlen=(1, 4), pad_rows=2),
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_score_topk_parity_small(cuda_lib, fmt, case):
    spec = dict(SMALL[case])
    wl = make_workload("tiny_fp8", fmt=fmt, seed=100 + case, topk=[16, 64, 100, 5, 2, 512][case], **spec)
    g = gpu_run(wl)
    o = oracle_run(wl)
    assert g["status"] == 0
    assert np.array_equal(g["starts"], o["starts"]) and np.array_equal(g["row_ends"], o["row_ends"])
    used = _used(fmt)
    assert np.array_equal(g["q_rows"][:, :used], o["q_rows"][:, :used])
    rows = range(wl.num_rows)
    check_logits(g["logits"], o["scores"], o["row_ends"], rows)
    check_topk(g["topk"], o["scores"], o["row_ends"], wl.topk, rows)


@pytest.mark.parametrize("fmt", FMTS)
def test_score_cache_bytes_match_oracle(cuda_lib, fmt):
    """The GPU cache after prefill + step equals the oracle's, page by page."""
    wl = make_workload("tiny_fp8", fmt=fmt, seed=7, R=3, seq=(100, 300), qlen=(1, 2), topk=8)
    g = gpu_run(wl)
    o = oracle_run(wl)
    cache = g["cache"].cpu().numpy()
    stride = g["page_stride"]
    for p_gpu, p_or in o["remap"].items():
        assert np.array_equal(cache[p_gpu * stride:p_gpu * stride + O.page_bytes(fmt)],
                              o["cache"][p_or * stride:p_or * stride + O.page_bytes(fmt)]), p_gpu


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("case", [1, 2, 3, 5])
def test_score_page_stride(cuda_lib, fmt, case):
    """Every format in a pool whose physical page stride is 48 bytes above the
    page section (8496 for FP8, 4400 for MXFP4: merged caches, page
    "amd.ops.fp4_indexer", cache_views), not a multiple of 32."""
    spec = dict(SMALL[case])
    wl = make_workload("tiny_fp8", fmt=fmt, seed=300 + case, topk=[16, 64, 100, 5, 2, 512][case], **spec)
    section = O.page_bytes(fmt)
    stride = section + 48
    g = gpu_run(wl, page_stride=stride)
    o = oracle_run(wl, page_stride=stride)
    assert g["status"] == 0
    cache = g["cache"].cpu().numpy()
    for p_gpu, p_or in o["remap"].items():
        assert np.array_equal(cache[p_gpu * stride:p_gpu * stride + section],
                              o["cache"][p_or * stride:p_or * stride + section])
    rows = range(wl.num_rows)
    check_logits(g["logits"], o["scores"], o["row_ends"], rows)
    check_topk(g["topk"], o["scores"], o["row_ends"], wl.topk, rows)


def _fp8_code_bytes(rng, shape):
    """E4M3 codes of magnitude 2^-2 .. 3.75: random sign, exponent field 5..8,
    random mantissa (no NaN code)."""
    sign = rng.integers(0, 2, shape, dtype=np.uint8) << 7
    exp = rng.integers(5, 9, shape, dtype=np.uint8) << 3
    man = rng.integers(0, 8, shape, dtype=np.uint8)
    return (sign | exp | man).astype(np.uint8)


@pytest.mark.parametrize("page_stride", [8448, 8448 + 64])
def test_fp8_mx_unequal_block_scales(cuda_lib, page_stride):
    """FP8-MX keys whose four UE8M0 bytes differ: byte b scales columns
    32b..32b+31 (page "cutedsl.dsa.index", module docstring: the MX scales of
    the logits kernels).  Cache, query rows and weights are seeded bytes
    written on the host, not by the library's writer; the oracle decodes the
    same bytes per 32-column block."""
    import torch
    rng = np.random.default_rng(77 + page_stride)
    qlen = np.array([1, 3, 4, 2, 1, 4], np.int32)
    seq = np.array([1, 700, 129, 64, 1000, 300], np.int32)
    R = len(qlen)
    npg = (seq + 63) // 64
    num_pages = int(npg.sum()) + 3
    max_pages = int(npg.max())
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((R, max_pages), -1, np.int32)
    off = 0
    for q in range(R):
        bt[q, :npg[q]] = perm[off:off + npg[q]]
        off += npg[q]
    cache = np.zeros(num_pages * page_stride, np.uint8)
    for p in range(num_pages):
        base = p * page_stride
        cache[base:base + 8192] = _fp8_code_bytes(rng, 8192)
        cache[base + 8192:base + 8448] = rng.integers(124, 131, 256).astype(np.uint8)   # 2^-3 .. 2^3, unequal
    rows = int(qlen.sum()) + 2                                                         # two padding rows
    q_rows = _fp8_code_bytes(rng, (rows, 4096))
    # positive head weights: the weighted head sum does not cancel, so FP32
    # accumulation stays far inside the tolerance whatever the block scales
    w = ((np.abs(rng.standard_normal((rows, 32))).astype(np.float32).view(np.uint32) >> 16) << 16).view(np.float32)
    starts, row_ends = O.decode_layout(seq, qlen, rows)
    k = 96
    dev = "cuda"
    wt = torch.from_numpy(w).to(torch.bfloat16).to(dev)
    logits, top = cuda_lib.score_paged("fp8_mx", torch.from_numpy(q_rows).to(dev), wt,
                                       torch.from_numpy(cache).to(dev), page_stride, num_pages,
                                       torch.from_numpy(bt).to(dev), torch.from_numpy(starts).to(dev),
                                       torch.from_numpy(row_ends).to(dev), int(qlen.max()), k=k, want_logits=True)
    torch.cuda.synchronize()
    want = O.score_paged("fp8_mx", q_rows, w, cache, page_stride, bt, starts, row_ends)
    check_logits(logits.cpu().numpy(), want, row_ends, range(rows))
    check_topk(top.cpu().numpy(), want, row_ends, k, range(rows))
    # the writer's form: the four scale bytes of each key equal (byte 0 copied to bytes 1-3)
    eq = cache.copy()
    for p in range(num_pages):
        base = p * page_stride + 8192
        sb = eq[base:base + 256].reshape(64, 4)
        sb[:, 1:] = sb[:, :1]
    want_eq = O.score_paged("fp8_mx", q_rows, w, eq, page_stride, bt, starts, row_ends)
    logits_eq, _ = cuda_lib.score_paged("fp8_mx", torch.from_numpy(q_rows).to(dev), wt,
                                        torch.from_numpy(eq).to(dev), page_stride, num_pages,
                                        torch.from_numpy(bt).to(dev), torch.from_numpy(starts).to(dev),
                                        torch.from_numpy(row_ends).to(dev), int(qlen.max()), want_logits=True)
    torch.cuda.synchronize()
    check_logits(logits_eq.cpu().numpy(), want_eq, row_ends, range(rows))


def test_topk_standalone_exact(cuda_lib):
    import torch
    rng = np.random.default_rng(5)
    rows, width = 23, 20000
    logits = np.round(rng.standard_normal((rows, width)), 2).astype(np.float32)   # heavy ties
    logits[3] = 1.0                                                               # all equal
    logits[4, :5000] = -np.inf
    logits[5] = -2.5                                                              # all equal, short row
    ends = rng.integers(0, width + 1, rows).astype(np.int32)
    ends[0], ends[1], ends[2], ends[3], ends[5], ends[6] = width, 0, 10, width, 6000, 8192
    for k in (1, 7, 64, 2048, 19999):
        got = cuda_lib.topk(torch.from_numpy(logits).cuda(), torch.from_numpy(ends).cuda(), k).cpu().numpy()
        want = O.topk(logits, ends, k)
        for r in range(rows):
            n = int(ends[r])
            if n <= k:
                assert list(got[r, :n]) == list(range(n)) and np.all(got[r, n:] == -1), (k, r)
                continue
            assert len(set(got[r].tolist())) == k and np.all((got[r] >= 0) & (got[r] < n))
            kth = logits[r, want[r, k - 1]]
            g_vals = logits[r, got[r]]
            assert np.all(g_vals >= kth), (k, r)
            # the multiset of selected values is unique
            assert np.array_equal(np.sort(g_vals), np.sort(logits[r, want[r]])), (k, r)


def test_topk_split_rows_with_overflowing_candidates_exact(cuda_lib):
    """Rows split over several CTAs whose scores all fall in one level-1 bin
    (1 + 7i ulp, shuffled: distinct, below 1.25): every span's candidate
    buffer overflows, so the row's last span builds the level-2 histogram by
    re-reading the row.  The selection is unique and must equal the oracle's
    exactly, as sets."""
    import torch
    rng = np.random.default_rng(9)
    rows, width = 5, 20000
    base = np.uint32(0x3F800000) + (np.arange(width, dtype=np.uint32) * np.uint32(7))
    logits = np.stack([rng.permutation(base) for _ in range(rows)]).view(np.float32)
    assert float(logits.max()) < 1.25
    ends = np.array([width, width, 15000, 9000, 4097], np.int32)
    for k in (64, 2048, 3000):
        got = cuda_lib.topk(torch.from_numpy(logits).cuda(), torch.from_numpy(ends).cuda(), k).cpu().numpy()
        want = O.topk(logits, ends, k)
        for r in range(rows):
            assert sorted(got[r].tolist()) == sorted(want[r].tolist()), (k, r)


def test_workspace_reuse_and_status(cuda_lib):
    """A second call on the same workspace gives the same answer (the workspace
    is left zero-filled), and a bad block-table entry sets the status bit."""
    import torch
    from dsa_case import bf16_tensor
    wl = make_workload("tiny_fp8", fmt="fp8", seed=11, R=4, seq=(3000, 6000), qlen=(1, 3), topk=256)
    g1 = gpu_run(wl)
    g2 = gpu_run(wl)
    for r in range(wl.num_rows):
        assert set(g1["topk"][r].tolist()) == set(g2["topk"][r].tolist())
    q_rows = torch.from_numpy(g1["q_rows"]).cuda()
    w = torch.from_numpy(g1["w"]).to(torch.bfloat16).cuda()
    bt = torch.from_numpy(wl.block_table).cuda()
    bt[0, 0] = wl.num_pages + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = torch.zeros(wl.num_pages * 8448, dtype=torch.uint8, device="cuda")
    cuda_lib.score_paged("fp8", q_rows, w, cache, 8448, wl.num_pages, bt, torch.from_numpy(g1["starts"]).cuda(),
                         torch.from_numpy(g1["row_ends"]).cuda(), 3, k=16, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2


def test_empty_and_degenerate(cuda_lib):
    import torch
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    st, en = cuda_lib.decode_layout(e, e, 4)
    assert st.cpu().tolist() == [0] and en.cpu().tolist() == [0, 0, 0, 0]
    q = torch.zeros((0, 32, 128), dtype=torch.bfloat16, device="cuda")
    wv = torch.zeros((0, 32), dtype=torch.bfloat16, device="cuda")
    r, w = cuda_lib.quantize_query("fp8", q, wv)
    assert r.shape == (0, 4096)
    # rows outside every request score nothing: logits -inf, top-k -1
    wl = make_workload("tiny_fp8", fmt="fp8", seed=3, R=1, seq=(300, 300), qlen=(1, 1), pad_rows=2, topk=8)
    g = gpu_run(wl)
    assert np.all(np.isneginf(g["logits"][1:])) and np.all(g["topk"][1:] == -1)


@pytest.mark.parametrize("name", ["tiny_fp8", "fp8_decode", "mxfp4_decode", "spec_verify", "long_mxfp4",
                                  "long_mxfp4/mxfp4_rg", "fp8_decode@8512"])
def test_full_size_all_rows(cuda_lib, name):
    """The named decode-step workloads at full size, in the launch configuration
    the bench times (``name/format`` overrides the cache format, ``name@stride``
    the physical page stride), every row against the oracle: logits element by
    element, top-k sets, row bounds and quantised query rows."""
    name, _, stride = name.partition("@")
    name, _, fmt = name.partition("/")
    overrides = {"fmt": fmt} if fmt else {}
    page_stride = int(stride) if stride else None
    wl = make_workload(name, **overrides)
    g = gpu_run(wl, want_logits=True, page_stride=page_stride)
    assert g["status"] == 0
    rows = list(range(wl.num_rows))
    scores, top, row_ends, starts, q_rows = oracle_rows(name, overrides, rows, page_stride=page_stride)
    assert np.array_equal(g["row_ends"], row_ends) and np.array_equal(g["starts"], starts)
    used = _used(wl.fmt)
    assert np.array_equal(g["q_rows"][:, :used], q_rows[:, :used])
    for r in rows:
        check_logits(g["logits"][r:r + 1], scores[r][None], row_ends[r:r + 1], [0])
        check_topk(g["topk"][r:r + 1], scores[r][None], row_ends[r:r + 1], wl.topk, [0])


def test_graphed_step_matches_eager(cuda_lib):
    """The graph-captured step (one staging copy in, step, top-k copy back)
    gives the eager step's top-k sets, replay after replay, and reads what the
    caller writes into its staging views."""
    import torch
    from sparse_attention_indexer_score_gb300.step import DecodeIndexer, GraphedStep
    wl = make_workload("tiny_fp8", fmt="mxfp4", seed=21, R=5, seq=(300, 900), qlen=(1, 3), pad_rows=1, topk=64)
    want = gpu_run(wl)["topk"]
    dev = torch.device("cuda")
    ix = DecodeIndexer(wl.fmt, wl.num_pages, torch.from_numpy(wl.block_table), torch.from_numpy(wl.gamma),
                       torch.from_numpy(wl.beta), wl.eps, wl.num_rows, wl.topk, dev)
    for q in range(wl.R):
        kb, sl = wl.prefill(q)
        if kb.shape[0]:
            ix.insert(bf16_tensor(kb, dev), torch.from_numpy(sl).to(dev))
    like = dict(q=bf16_tensor(wl.q_bits, "cpu"), wv=bf16_tensor(wl.wv_bits, "cpu"),
                keys=bf16_tensor(wl.step_key_bits, "cpu"), slots=torch.from_numpy(wl.step_slots),
                seq_lens=torch.from_numpy(wl.seq_lens), query_lens=torch.from_numpy(wl.query_lens))
    g = GraphedStep(ix, like, int(wl.query_lens.max()))
    assert all(g.inputs[k].is_pinned() for k in GraphedStep.NAMES) and g.host_topk.is_pinned()
    for _ in range(3):
        g.host_topk.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        got = g.host_topk.numpy()
        for r in range(wl.num_rows):
            assert sorted(got[r].tolist()) == sorted(want[r].tolist()), r
    # rows whose request length the caller sets to 1 now select only position 0
    g.inputs["seq_lens"].fill_(1)
    g.inputs["query_lens"].fill_(1)
    g.replay()
    torch.cuda.synchronize()
    got = g.host_topk.numpy()
    assert ix.status_bits() == 0
    for r in range(min(wl.R, wl.num_rows)):
        assert got[r, 0] == 0 and np.all(got[r, 1:] == -1), r


def test_bounded_wait_runs_out_and_the_context_stays_usable(cuda_lib):
    """Failure detection: a pipeline wait on a barrier nothing completes gives
    up after its limit, the host reads the timeout bit, and the next calls run."""
    import time
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    cuda_lib.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    assert 0.5 < time.time() - t0 < 30.0
    assert int(status.item()) == 8
    wl = make_workload("tiny_fp8", fmt="fp8", seed=4, R=2, seq=(200, 300), qlen=(1, 2), topk=16)
    g = gpu_run(wl)
    o = oracle_run(wl)
    assert g["status"] == 0
    check_topk(g["topk"], o["scores"], o["row_ends"], wl.topk, range(wl.num_rows))


def test_more_rows_and_segments_than_the_plan_keeps_on_chip(cuda_lib):
    """4200 one-row requests: more row bounds and segments than the plan keeps
    in shared memory (4096 of each), so its global-memory paths run; sampled
    rows against the oracle, all rows' bounds exactly."""
    wl = make_workload("tiny_fp8", fmt="fp8", seed=33, R=4200, seq=(1, 300), qlen=(1, 1), pad_rows=5, topk=32)
    assert wl.num_rows > 4096
    g = gpu_run(wl)
    assert g["status"] == 0
    rng = np.random.default_rng(1)
    rows = sorted(set(rng.choice(wl.num_rows - 5, 40, replace=False).tolist() + [0, 4095, 4096, 4199, wl.num_rows - 1]))
    o = oracle_run(wl, rows=rows)
    assert np.array_equal(g["row_ends"], o["row_ends"]) and np.array_equal(g["starts"], o["starts"])
    check_logits(g["logits"], o["scores"], o["row_ends"], rows)
    check_topk(g["topk"], o["scores"], o["row_ends"], wl.topk, rows)


def test_step_pipeline_matches_eager(cuda_lib):
    """Steps with their copies overlapped on separate streams give the eager
    step's top-k sets in both staging sets, step after step."""
    import torch
    from sparse_attention_indexer_score_gb300.step import DecodeIndexer, StepPipeline
    wl = make_workload("tiny_fp8", fmt="fp8", seed=22, R=6, seq=(300, 2000), qlen=(1, 4), pad_rows=2, topk=100)
    want = gpu_run(wl)["topk"]
    dev = torch.device("cuda")
    ix = DecodeIndexer(wl.fmt, wl.num_pages, torch.from_numpy(wl.block_table), torch.from_numpy(wl.gamma),
                       torch.from_numpy(wl.beta), wl.eps, wl.num_rows, wl.topk, dev)
    for q in range(wl.R):
        kb, sl = wl.prefill(q)
        if kb.shape[0]:
            ix.insert(bf16_tensor(kb, dev), torch.from_numpy(sl).to(dev))
    like = dict(q=bf16_tensor(wl.q_bits, "cpu"), wv=bf16_tensor(wl.wv_bits, "cpu"),
                keys=bf16_tensor(wl.step_key_bits, "cpu"), slots=torch.from_numpy(wl.step_slots),
                seq_lens=torch.from_numpy(wl.seq_lens), query_lens=torch.from_numpy(wl.query_lens))
    pipe = StepPipeline(ix, like, int(wl.query_lens.max()), caches=[ix.cache, ix.cache.clone()])
    for rnd in range(3):
        for i in range(2):
            pipe.host_topk(i).fill_(-7)
        pipe.run(6)
        torch.cuda.synchronize()
        for i in range(2):
            got = pipe.host_topk(i).numpy()
            for r in range(wl.num_rows):
                assert sorted(got[r].tolist()) == sorted(want[r].tolist()), (rnd, i, r)
    assert ix.status_bits() == 0


@pytest.mark.parametrize("heads", [16, 32, 64])
@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp4_rg"])
@pytest.mark.parametrize("case", [2, 3, 5])
def test_score_heads_parity(cuda_lib, fmt, heads, case):
    """Page "amd.ops.fp4_indexer", score_paged: queries of 16, 32 or 64 heads,
    quantised by quantize_queries on each side, scored against the MXFP4 cache
    in either placement; logits and top-k against the oracle."""
    import torch
    spec = dict(SMALL[case])
    wl = make_workload("tiny_fp8", fmt=fmt, seed=500 + case + heads, topk=[16, 64, 100, 5, 2, 512][case], **spec)
    rng = np.random.default_rng(900 + heads + case)
    x = rng.standard_normal((wl.num_rows, heads, 128)).astype(np.float32)
    qb = ((x.view(np.uint32).astype(np.uint64) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    wf = rng.standard_normal((wl.num_rows, heads)).astype(np.float32)
    wb = ((wf.view(np.uint32).astype(np.uint64) + 0x7FFF + ((wf.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    g = gpu_run(wl)                                     # the GPU cache (prefill + step keys) and row bounds
    o = oracle_run(wl)                                  # the oracle's own cache of the same keys
    payload, scales = cuda_lib.quantize_queries_rg(bf16_tensor(qb, "cuda"))
    w = bf16_tensor(wb, "cuda")
    dev = "cuda"
    logits, top = cuda_lib.score_paged_heads(fmt, payload, scales, w, g["cache"], g["page_stride"], wl.num_pages,
                                             torch.from_numpy(wl.block_table).to(dev),
                                             torch.from_numpy(g["starts"]).to(dev),
                                             torch.from_numpy(g["row_ends"]).to(dev),
                                             int(wl.query_lens.max(initial=0)), k=wl.topk, want_logits=True)
    torch.cuda.synchronize()
    want_p, want_s = O.quantize_queries(bf16_bits_to_f32(qb))
    bt = np.full_like(wl.block_table, -1)
    for qq in range(wl.R):
        n = (int(wl.seq_lens[qq]) + 63) // 64
        bt[qq, :n] = [o["remap"][int(pg)] for pg in wl.block_table[qq, :n]]
    want = O.score_paged_heads(fmt, want_p, want_s, bf16_bits_to_f32(wb), o["cache"], O.page_bytes(fmt), bt,
                               o["starts"], o["row_ends"])
    rows = range(wl.num_rows)
    check_logits(logits.cpu().numpy(), want, o["row_ends"], rows)
    check_topk(top.cpu().numpy(), want, o["row_ends"], wl.topk, rows)


@pytest.mark.parametrize("seq", [(5000, 7000), (20000, 30000)])
def test_topk_all_equal_logits(cuda_lib, seq):
    """Zero queries make every logit +0: one histogram bin holds a whole row, so
    the level-3 candidates exceed what a selecting team keeps on chip and, for
    rows over 8192 keys, the level-1 candidate list overflows and the row is
    re-read.  Any k distinct positions below the row's bound are correct."""
    wl = make_workload("tiny_fp8", fmt="fp8", seed=41, R=3, seq=seq, qlen=(1, 2), pad_rows=1, topk=2048)
    wl.q_bits[:] = 0
    g = gpu_run(wl)
    assert g["status"] == 0
    k = wl.topk
    for r in range(wl.num_rows):
        n = int(g["row_ends"][r])
        assert np.all(g["logits"][r, :n] == 0.0) and np.all(np.isneginf(g["logits"][r, n:]))
        t = g["topk"][r]
        if n <= k:
            assert np.array_equal(t[:n], np.arange(n)) and np.all(t[n:] == -1)
        else:
            assert len(set(t.tolist())) == k and t.min() >= 0 and t.max() < n, r


@pytest.mark.parametrize("topk", [64, 700])
def test_topk_few_distinct_logits(cuda_lib, topk):
    """One non-zero query element against MXFP4 keys: each logit is w * ReLU(q * k_d)
    with k_d on the E2M1 grid times a power of two, about ten distinct values a
    row, so 66..454 keys tie in the level-2 boundary bin and the level-3
    histogram decides; the selected multiset of values is unique."""
    wl = make_workload("tiny_fp8", fmt="mxfp4", seed=43, R=2, seq=(5000, 7000), qlen=(1, 2), pad_rows=0, topk=topk)
    q = np.zeros_like(wl.q_bits)
    q[:, 0, 0] = 0x3F80   # BF16 1.0
    wl.q_bits[:] = q
    g = gpu_run(wl)
    o = oracle_run(wl)
    assert g["status"] == 0
    rows = range(wl.num_rows)
    check_logits(g["logits"], o["scores"], o["row_ends"], rows)
    check_topk(g["topk"], o["scores"], o["row_ends"], wl.topk, rows)


def test_logits_buffer_with_odd_row_stride(cuda_lib):
    """A caller logits buffer whose rows are not 16-byte aligned (row stride
    width + 1): the top-k reads it with scalar loads.  Logits equal those of a
    packed buffer, columns past the buffer's width stay untouched, and the top-k
    sets agree with the logits."""
    import torch
    wl = make_workload("tiny_fp8", fmt="fp8_mx", seed=45, R=3, seq=(3000, 9000), qlen=(1, 3), pad_rows=1, topk=256)
    g = gpu_run(wl)
    dev = torch.device("cuda")
    bt = torch.from_numpy(wl.block_table).to(dev)
    width = bt.shape[1] * 64
    big = torch.full((wl.num_rows, width + 1), 7.0, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _, top = cuda_lib.score_paged(wl.fmt, torch.from_numpy(g["q_rows"]).to(dev),
                                  torch.from_numpy(g["w"]).to(torch.bfloat16).to(dev), g["cache"], g["page_stride"],
                                  wl.num_pages, bt, torch.from_numpy(g["starts"]).to(dev),
                                  torch.from_numpy(g["row_ends"]).to(dev), int(wl.query_lens.max()), k=wl.topk,
                                  status=status, logits=big[:, :width])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = big.cpu().numpy()
    assert np.array_equal(got[:, :width], g["logits"]) and np.all(got[:, width] == 7.0)
    check_topk(top.cpu().numpy(), g["logits"].astype(np.float64), g["row_ends"], wl.topk, range(wl.num_rows))


@pytest.mark.parametrize("kind", ["fp8", "mxf4"])
def test_mma_probe_rate_is_plausible(cuda_lib, kind):
    """The tensor-core rate probe behind roofline.tensor: its final wait ends
    (status 0), a longer run takes longer, and the rate lies between a floor and
    the nominal dense peak (FP8 4.5, FP4 13.5 PFLOP/s per GPU)."""
    import torch
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    times = {}
    for iters in (1 << 14, 1 << 16):
        cuda_lib.probe_mma(kind, iters, status)   # warm-up
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        cuda_lib.probe_mma(kind, iters, status)
        b.record()
        torch.cuda.synchronize()
        times[iters] = a.elapsed_time(b)
    assert int(status.item()) == 0
    assert times[1 << 16] > times[1 << 14]
    flops = 2 * 128 * 128 * cuda_lib.MMA_K[kind] * (1 << 16) * sms
    pflops = flops / (times[1 << 16] / 1e3) / 1e15
    nominal = {"fp8": 4.5, "mxf4": 13.5}[kind]
    assert 0.1 * nominal < pflops < 1.05 * nominal, pflops
    with pytest.raises(RuntimeError):
        cuda_lib.probe_mma(kind, 0, status)


@pytest.mark.parametrize("name", ["fp8_decode", "mxfp4_decode", "long_mxfp4", "spec_verify"])
def test_full_size_topk_as_benched(cuda_lib, name):
    """The decode step exactly as the bench times it (logits kept in the
    workspace, no -inf fill), at full size, twice on one workspace: top-k sets
    against the oracle (every row; spec_verify 40 sampled rows and the first and
    last real rows), all row bounds exactly, the status word clean."""
    import torch
    from dsa_case import bf16_tensor
    from sparse_attention_indexer_score_gb300.step import DecodeIndexer
    wl = make_workload(name)
    dev = torch.device("cuda")
    ix = DecodeIndexer(wl.fmt, wl.num_pages, torch.from_numpy(wl.block_table), torch.from_numpy(wl.gamma),
                       torch.from_numpy(wl.beta), wl.eps, wl.num_rows, wl.topk, dev)
    for q in range(wl.R):
        kb, sl = wl.prefill(q)
        if kb.shape[0]:
            ix.insert(bf16_tensor(kb, dev), torch.from_numpy(sl).to(dev))
    args = (bf16_tensor(wl.q_bits, dev), bf16_tensor(wl.wv_bits, dev), bf16_tensor(wl.step_key_bits, dev),
            torch.from_numpy(wl.step_slots).to(dev), torch.from_numpy(wl.seq_lens).to(dev),
            torch.from_numpy(wl.query_lens).to(dev), int(wl.query_lens.max(initial=0)))
    tops = []
    for _ in range(2):   # the second call reuses the workspace the first left zero-filled
        out = ix.step(*args, want_logits=False)
        torch.cuda.synchronize()
        assert out.logits is None
        tops.append(out.topk.cpu().numpy())
    assert ix.status_bits() == 0
    real = [r for r in range(wl.num_rows) if wl.row_request[r] >= 0]
    if name == "spec_verify":
        rng = np.random.default_rng(5)
        rows = sorted(set(rng.choice(real, 40, replace=False).tolist() + [real[0], real[-1]]))
    else:
        rows = real
    scores, top, row_ends, starts, q_rows = oracle_rows(name, {}, rows)
    assert np.array_equal(out.row_ends.cpu().numpy(), row_ends)
    for r in rows:
        for t in tops:
            check_topk(t[r:r + 1], scores[r][None], row_ends[r:r + 1], wl.topk, [0])
    pad = [r for r in range(wl.num_rows) if wl.row_request[r] < 0]
    for t in tops:
        assert np.all(t[pad] == -1)


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_step_equals_prepare_then_score(cuda_lib, fmt):
    """dsa_decode_step gives the bytes of dsa_prepare_step followed by
    dsa_score_paged: query rows, weights, cache,
    row bounds, logits and top-k; with no rows it only inserts the keys."""
    import torch
    wl = make_workload("tiny_fp8", fmt=fmt, seed=31, R=9, seq=(60, 3000), qlen=(1, 5), pad_rows=2, topk=64)
    dev = torch.device("cuda")
    stride = O.page_bytes(fmt)
    bt = torch.from_numpy(wl.block_table).to(dev)
    gamma, beta = torch.from_numpy(wl.gamma).to(dev), torch.from_numpy(wl.beta).to(dev)
    base = torch.zeros(wl.num_pages * stride, dtype=torch.uint8, device=dev)
    for q in range(wl.R):
        kb, sl = wl.prefill(q)
        if kb.shape[0]:
            cuda_lib.insert_key(fmt, bf16_tensor(kb, dev), gamma, beta, wl.eps, torch.from_numpy(sl).to(dev), base,
                                stride, wl.num_pages)
    args = (bf16_tensor(wl.q_bits, dev), bf16_tensor(wl.wv_bits, dev), bf16_tensor(wl.step_key_bits, dev), gamma,
            beta, wl.eps, torch.from_numpy(wl.step_slots).to(dev))
    lens = (torch.from_numpy(wl.seq_lens).to(dev), torch.from_numpy(wl.query_lens).to(dev))
    mq = int(wl.query_lens.max())

    def run(fused, num_rows):
        cache = base.clone()
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if fused:
            q_rows, w, st, en, lg, top = cuda_lib.decode_step(fmt, args[0][:num_rows], args[1][:num_rows], *args[2:],
                                                              cache, stride, wl.num_pages, *lens, bt, mq,
                                                              top_k=wl.topk if num_rows else 0,
                                                              want_logits=num_rows > 0, status=status)
        else:
            q_rows, w, st, en = cuda_lib.prepare_step(fmt, args[0][:num_rows], args[1][:num_rows], *args[2:], cache,
                                                      stride, wl.num_pages, *lens, num_rows, status=status)
            lg = top = None
            if num_rows:
                lg, top = cuda_lib.score_paged(fmt, q_rows, w, cache, stride, wl.num_pages, bt, st, en, mq,
                                               k=wl.topk, want_logits=True, status=status)
        torch.cuda.synchronize()
        return q_rows.cpu(), w.float().cpu(), cache.cpu(), st.cpu(), en.cpu(), lg, top, int(status.item())

    a, b = run(True, wl.num_rows), run(False, wl.num_rows)
    for x, y in zip(a[:5], b[:5]):
        assert torch.equal(x, y)
    assert a[7] == b[7] == 0
    ends = b[4].numpy()
    la, lb = a[5].cpu().numpy(), b[5].cpu().numpy()
    for r in range(wl.num_rows):
        assert np.array_equal(la[r, :ends[r]], lb[r, :ends[r]]), r
    check_topk(a[6].cpu().numpy(), lb.astype(np.float64), ends, wl.topk, range(wl.num_rows))
    a0, b0 = run(True, 0), run(False, 0)
    assert torch.equal(a0[2], b0[2]) and not torch.equal(a0[2], base.cpu())
    assert a0[3].numel() == b0[3].numel() and torch.equal(a0[3], b0[3]) and a0[7] == b0[7] == 0
