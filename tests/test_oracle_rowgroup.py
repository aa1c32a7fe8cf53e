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
    assert np.array_equal(qa[:, :2048], qb[:, :2048]) and np.array_equal(wa, wb)
    for r in range(3):
        assert np.array_equal(O.decode_query("mxfp4", qa[r]), O.decode_query("mxfp4_rg", qb[r]))
    for r in range(3):
        assert np.array_equal(O.score_row("mxfp4", qa[r], wa[r], a), O.score_row("mxfp4_rg", qb[r], wb[r], b))


# E2M1 (OCP MX) magnitudes and their 3-bit codes; bit 3 is the sign.
_E2M1 = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def _grid_queries(rng, rows, heads):
    """Queries whose every 32-column block has max |x| = 6 * 2^k exactly and
    values on the E2M1 grid times 2^k: the MX scale byte is k + 127 and every
    code is exact, so both follow from the format's definition alone."""
    mags = np.array(sorted(_E2M1))
    k = rng.integers(-20, 20, (rows, heads, 4))
    v = rng.choice(mags, (rows, heads, 4, 32)) * rng.choice([-1.0, 1.0], (rows, heads, 4, 32))
    v[..., 0] = 6.0 * rng.choice([-1.0, 1.0], (rows, heads, 4))        # the block maximum
    x = (v * np.ldexp(1.0, k)[..., None]).astype(np.float32)
    codes = np.vectorize(lambda t: _E2M1[abs(t)] | (8 if np.signbit(t) else 0))(v).astype(np.uint8)   # -0 keeps its sign
    pairs = (codes[..., 0::2] | (codes[..., 1::2] << 4)).reshape(rows, heads, 64)
    return x.reshape(rows, heads, 128), pairs, (k + 127).astype(np.uint8)


def test_quantize_queries_closed_form():
    """Page *amd.ops.fp4_indexer*, ``quantize_queries``: payload [rows, heads, 64]
    and scales [rows, 1, 4, 16, 4] for 16, 32 and 64 heads; the scale of block
    g of head h at flat g * 64 + h (the group-major reading), unused head slots zero."""
    rng = np.random.default_rng(7)
    for heads in (16, 32, 64):
        x, pairs, sbytes = _grid_queries(rng, 5, heads)
        payload, scales = O.quantize_queries(x)
        assert payload.shape == (5, heads, 64) and scales.shape == (5, 1, 4, 16, 4)
        assert np.array_equal(payload, pairs)
        flat = scales.reshape(5, 256)
        for h in range(64):
            for g in range(4):
                want = sbytes[:, h, g] if h < heads else np.zeros(5, np.uint8)
                assert np.array_equal(flat[:, g * 64 + h], want), (heads, h, g)


def test_quantize_queries_rejects_other_head_counts():
    import pytest
    for heads in (8, 24, 128):
        with pytest.raises(ValueError):
            O.quantize_queries(np.zeros((2, heads, 128), np.float32))
    with pytest.raises(ValueError):
        O.quantize_queries(np.zeros((2, 32, 64), np.float32))


def test_rowgroup_query_rows_carry_the_same_codes_and_scales():
    """A "mxfp4_rg" query row is the page's 32-head payload followed by its
    row-group scales, and it decodes to the token-major row's values."""
    rng = np.random.default_rng(8)
    x, pairs, sbytes = _grid_queries(rng, 4, 32)
    wv = rng.standard_normal((4, 32)).astype(np.float32)
    rg, w_rg = O.quantize_query("mxfp4_rg", x, wv)
    tm, w_tm = O.quantize_query("mxfp4", x, wv)
    payload, scales = O.quantize_queries(x)
    assert np.array_equal(rg[:, :2048], payload.reshape(4, 2048))
    assert np.array_equal(rg[:, 2048:2304], scales.reshape(4, 256))
    assert not rg[:, 2304:].any() and np.array_equal(w_rg, w_tm)
    assert np.array_equal(tm[:, 2048:2176].reshape(4, 32, 4), sbytes)
    for r in range(4):
        assert np.array_equal(O.decode_query("mxfp4_rg", rg[r]), O.decode_query("mxfp4", tm[r]))
        assert np.array_equal(O.decode_query("mxfp4_rg", rg[r]), x[r].astype(np.float64))
