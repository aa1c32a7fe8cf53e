"""Pins of the row-group MXFP4 page ("mxfp4_rg", page *amd.ops.fp4_indexer*,
``cache_views``): the page's own strided views of a section must show the
same codes and scales as the token-major MXFP4 page holds for the same keys,
and the decoded keys and scores must agree."""

import numpy as np
from numpy.lib.stride_tricks import as_strided

from oracle import indexer as O


def _pages(rng, n, num_pages, stride):
    x = (rng.standard_normal((n, 128)) * 2.0).astype(np.float32)
    x[0, :32] = 0.0                                   # an all-zero block
    gamma = (1 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    beta = (0.1 * rng.standard_normal(128)).astype(np.float32)
    slots = rng.permutation(num_pages * 64)[:n].astype(np.int64)
    out = {}
    for fmt in ("mxfp4", "mxfp4_rg"):
        cache = np.zeros(num_pages * stride, np.uint8)
        assert O.insert_key(fmt, cache, stride, num_pages, x, gamma, beta, 1e-6, slots) == 0
        out[fmt] = cache
    return out, slots


def test_page_views_show_the_token_major_codes():
    rng = np.random.default_rng(0)
    num_pages, stride = 5, 4352 + 96                  # a merged cache: stride above the section
    c, _ = _pages(rng, 200, num_pages, stride)
    rg, tm = c["mxfp4_rg"], c["mxfp4"]
    # the page's views: payload (pages, 1, 4, 64, 16) strides (stride, 4096, 1024, 16, 1),
    # scales (pages, 1, 4, 64) strides (stride, 256, 64, 1) from byte 4096
    payload = as_strided(rg, (num_pages, 1, 4, 64, 16), (stride, 4096, 1024, 16, 1))
    scales = as_strided(rg[4096:], (num_pages, 1, 4, 64), (stride, 256, 64, 1))
    for p in range(num_pages):
        sec = tm[p * stride: p * stride + 4352]
        codes = sec[:4096].reshape(64, 64)             # token t: 64 bytes, column group g at bytes 16g..
        sb = sec[4096:].reshape(64, 4)                 # token t: the 4 group bytes
        for g in range(4):
            assert np.array_equal(payload[p, 0, g], codes[:, 16 * g:16 * g + 16])
            assert np.array_equal(scales[p, 0, g], sb[:, g])
        assert not rg[p * stride + 4352:(p + 1) * stride].any()     # the rest of the stride untouched


def test_decoded_keys_and_scores_agree():
    rng = np.random.default_rng(1)
    num_pages, stride = 6, 4352
    c, slots = _pages(rng, 6 * 64, num_pages, stride)
    table = rng.permutation(num_pages).astype(np.int32)
    n = 6 * 64 - 17
    a = O.decode_keys("mxfp4", c["mxfp4"], stride, table, n)
    b = O.decode_keys("mxfp4_rg", c["mxfp4_rg"], stride, table, n)
    assert np.array_equal(a, b)
    q = rng.standard_normal((3, 32, 128)).astype(np.float32)
    wv = rng.standard_normal((3, 32)).astype(np.float32)
    qa, wa = O.quantize_query("mxfp4", q, wv)
    qb, wb = O.quantize_query("mxfp4_rg", q, wv)
    assert np.array_equal(qa, qb) and np.array_equal(wa, wb)
    for r in range(3):
        assert np.array_equal(O.score_row("mxfp4", qa[r], wa[r], a), O.score_row("mxfp4_rg", qb[r], wb[r], b))
