"""The C ABI library loads and exports every symbol include/dsa.h declares, and
its host-side argument checks return the documented codes (CPU only: no call
here reaches the GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_score_gb300 import build
    try:
        path = build.build()
    except RuntimeError as e:   # no nvcc on this machine
        pytest.skip(str(e))
    from sparse_attention_indexer_score_gb300 import dsa
    dsa._lib = None
    return dsa.lib()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes_are_host_only(lib):
    a = lib.dsa_workspace_size(0, 64, 64, 128, 2048)
    b = lib.dsa_workspace_size(0, 128, 64, 128, 2048)
    assert a > 64 * 128 * 64 * 4 and b > a
    assert lib.dsa_topk_workspace_size(10, 64) >= 10 * 2048 * 4


def test_host_argument_checks(lib):
    # format, counts and strides are checked before anything touches the GPU
    assert lib.dsa_quantize_query(7, None, 4096, None, 32, 1, None, None, None) == -2
    assert lib.dsa_quantize_query(0, None, 4096, None, 32, -1, None, None, None) == -1
    assert lib.dsa_quantize_query(0, None, 4096, None, 32, 0, None, None, None) == 0
    assert lib.dsa_quantize_query(0, 16, 4000, 16, 32, 2, 16, 16, None) == -1
    assert lib.dsa_insert_key(0, 16, 128, 16, 16, 1e-6, 16, 1, 16, 4352, 1, None, None) == -1   # FP8 stride < 8448
    assert lib.dsa_insert_key(2, 16, 128, 16, 16, 1e-6, 16, 0, 16, 4352, 1, None, None) == 0
    assert lib.dsa_decode_layout(None, 0, None, 0, -1, None, None, None) == -1
    assert lib.dsa_decode_layout(16, 1, 16, 2, 2, 16, 16, None) == -1        # fewer seq_lens than requests
    assert lib.dsa_score_paged(4, *([0] * 21)) == -2
    assert lib.dsa_selftest_wait_timeout(None, None) == -1
    assert lib.dsa_quantize_queries_rg(16, 4096, 128, 48, 1, 16, 16, None) == -2      # 48 heads
    assert lib.dsa_quantize_queries_rg(None, 0, 128, 64, 0, None, None, None) == 0    # no rows
    assert lib.dsa_quantize_queries_rg(16, 4096, 100, 32, 1, 16, 16, None) == -1     # head stride < 128
    assert lib.dsa_insert_key(4, 16, 128, 16, 16, 1e-6, 16, 0, 16, 4352, 1, None, None) == -2
    assert lib.dsa_insert_key(3, 16, 128, 16, 16, 1e-6, 16, 0, 16, 4352, 1, None, None) == 0   # row-group MXFP4
    assert lib.dsa_insert_key(3, 16, 128, 16, 16, 1e-6, 16, 1, 16, 4352 - 16, 1, None, None) == -1
    assert lib.dsa_score_paged(3, 32, 32, 32, 4352 + 8, 1, 16, 1, 1, 16, 16, 1, 1, 1, None, 0, 4, None, 256,
                               10**9, None, None) == -1                         # row-group stride not a multiple of 16
    assert lib.dsa_score_paged(0, 16, 16, 16, 8448, 1, 16, 1, 1, 16, 16, 1, 0, 1, None, 0, 4, None, 256, 10**9,
                               None, None) == 0                                 # zero rows
    assert lib.dsa_score_paged(2, 32, 32, 32, 4352 + 8, 1, 16, 1, 1, 16, 16, 1, 1, 1, None, 0, 4, None, 256,
                               10**9, None, None) == -1                         # MXFP4 stride not a multiple of 16
    assert lib.dsa_topk(None, 10, None, 1, 20, 4, None, None, 0, None) == -1  # ld < width


def test_more_host_argument_checks(lib):
    """The documented error codes of the remaining calls, all decided on the host."""
    A = 1 << 20   # a 256-byte-aligned stand-in address (never dereferenced: every call below fails its checks)
    # dsa_decode_layout_dcp: rank outside the world, interleave < 1, world < 1
    assert lib.dsa_decode_layout_dcp(A, 1, A, 1, 1, 2, 2, 64, A, A, None) == -1
    assert lib.dsa_decode_layout_dcp(A, 1, A, 1, 1, 0, 2, 0, A, A, None) == -1
    assert lib.dsa_decode_layout_dcp(A, 1, A, 1, 1, 0, 0, 64, A, A, None) == -1
    # dsa_topk_merge: short leading dimension, bad rank with out_local, unaligned workspace, world < 1
    assert lib.dsa_topk_merge(A, 63, A, 64, 2, 2, 32, 16, 32, A, 0, None, A, 10**9, None) == -1
    assert lib.dsa_topk_merge(A, 64, A, 64, 2, 2, 32, 16, 32, A, 2, A, A, 10**9, None) == -1
    assert lib.dsa_topk_merge(A, 64, A, 64, 2, 2, 32, 16, 32, A, 0, None, A + 16, 10**9, None) == -1
    assert lib.dsa_topk_merge(A, 64, A, 64, 2, 0, 32, 16, 32, A, 0, None, A, 10**9, None) == -1
    assert lib.dsa_topk_merge(A, 64, A, 64, 2, 2, 32, 16, 32, A, 0, None, A, 16, None) == -1   # workspace too small
    # dsa_query_norm: unknown variant, short or odd row stride, unaligned rows
    assert lib.dsa_query_norm(A, 1536, A, 1e-6, 4, A, 1536, 2, None) == -1
    assert lib.dsa_query_norm(A, 1500, A, 1e-6, 4, A, 1536, 0, None) == -1
    assert lib.dsa_query_norm(A, 1540, A, 1e-6, 4, A, 1536, 0, None) == -1
    assert lib.dsa_query_norm(A + 2, 1536, A, 1e-6, 4, A, 1536, 0, None) == -1
    assert lib.dsa_query_norm(None, 1536, None, 1e-6, 0, None, 1536, 0, None) == 0    # empty batch
    # dsa_score_paged: unaligned query rows or workspace, short block-table stride, short logits
    # leading dimension, a workspace too small, missing cache with pages
    base = [0, A, A, A, 8448, 1, A, 4, 4, A, A, 1, 1, 1, None, 0, 16, A, A, 10**9, None, None]   # never called as is
    for i, v in ((1, A + 8), (18, A + 128), (7, 3), (19, 64)):
        bad = list(base)
        bad[i] = v
        assert lib.dsa_score_paged(*bad) == -1, i
    bad = list(base)
    bad[14], bad[15] = A, 100                             # logits with ld < max_pages * 64
    assert lib.dsa_score_paged(*bad) == -1
    bad = list(base)
    bad[3] = None                                         # pages but no cache
    assert lib.dsa_score_paged(*bad) == -1


def test_prepare_step_returns_each_part_s_error(lib):
    """The fused preparation reports the argument error of whichever part
    (quantize, insert, layout) is wrong, before any launch."""
    A = 1 << 20
    ok_q = [0, A, 4096, A, 32, 1, A, A]                       # fmt, q, stride, wv, stride, rows, q_out, w_out
    ok_k = [A, 128, A, A, 1e-6, A, 1, A, 8448, 1]             # k, stride, gamma, beta, eps, slots, n, cache, stride, pages
    ok_l = [A, 1, A, 1, 1, A, A]                              # seq, num_seq, qlen, R, num_rows, starts, row_ends
    tail = [None, None]                                       # status, stream

    def call(q, k, l):
        return lib.dsa_prepare_step(*q, *k, *l, *tail)

    bad_q = list(ok_q)
    bad_q[0] = 9                                              # unknown format
    assert call(bad_q, ok_k, ok_l) == -2
    bad_q = list(ok_q)
    bad_q[2] = 4000                                           # query row stride < 4096
    assert call(bad_q, ok_k, ok_l) == -1
    bad_k = list(ok_k)
    bad_k[8] = 4352                                           # FP8 page stride < 8448
    assert call(ok_q, bad_k, ok_l) == -1
    bad_l = list(ok_l)
    bad_l[1] = 0                                              # fewer seq_lens than requests
    assert call(ok_q, ok_k, bad_l) == -1


def test_the_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No fallback: a missing libdsa.so raises instead of computing anything."""
    from sparse_attention_indexer_score_gb300 import dsa
    monkeypatch.setattr(dsa, "_lib", None)
    monkeypatch.setattr(dsa, "LIB_PATH", str(tmp_path / "libdsa.so"))
    with pytest.raises(RuntimeError, match="missing"):
        dsa.lib()


def test_decode_step_returns_argument_errors_before_any_launch(lib):
    """dsa_decode_step reports the argument error of the preparation or of the
    scoring (no launch, so this runs without a GPU)."""
    A = 1 << 20
    prep_q = [0, A, 4096, A, 32]                              # fmt, q, stride, wv, stride
    prep_k = [A, 128, A, A, 1e-6, A, 1, A, 8448, 1]           # k, stride, gamma, beta, eps, slots, n, cache, stride, pages
    layout = [A, 1, A, 1, 1]                                  # seq_lens, num_seq, query_lens, R, num_rows
    score = [A, 1, 1, 1, A, A, A, A, None, 0, 4, A, A, 1 << 30, None, None]
    # block table, bt_stride, max_pages, max_query_len, q_out, w_out, starts, row_ends,
    # logits, logits_ld, top_k, topk, workspace, workspace_bytes, status, stream

    def call(q=prep_q, k=prep_k, l=layout, sc=score):
        return lib.dsa_decode_step(*q, *k, *l, *sc)

    bad = list(prep_q)
    bad[0] = 9                                                # unknown format
    assert call(q=bad) == -2
    bad = list(prep_q)
    bad[2] = 4000                                             # query row stride < 4096
    assert call(q=bad) == -1
    bad = list(prep_k)
    bad[8] = 4352                                             # FP8 page stride < 8448
    assert call(k=bad) == -1
    bad = list(layout)
    bad[1] = 0                                                # fewer seq_lens than requests
    assert call(l=bad) == -1
    bad = list(score)
    bad[1] = 0                                                # block-table row stride < max_pages
    assert call(sc=bad) == -1
    bad = list(score)
    bad[13] = 16                                              # workspace too small
    assert call(sc=bad) == -1
