"""Pins of the oracle's scoring of 16-, 32- and 64-head MXFP4 queries (page
*amd.ops.fp4_indexer*, ``score_paged`` with queries from ``quantize_queries``).

The closed form builds the cache bytes by hand from the MXFP4 definition (an
E2M1 code table of its own and UE8M0 bytes), in either page placement, and
queries whose codes and scales are exact on the E2M1 grid, so every logit is
sum_h w_h * max(0, x_h . k_t) of known values, computed here directly.
"""

import numpy as np
import pytest

from oracle import indexer as O

_E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _code_value(code):
    v = _E2M1_VALUES[code & 7]
    return np.where(code & 8, -v, v)


def _grid_queries(rng, rows, heads):
    """Queries whose every 32-column block has max |x| = 6 * 2^k (k in -3..3)
    and values on the E2M1 grid times 2^k: quantize_queries keeps them exactly."""
    k = rng.integers(-3, 4, (rows, heads, 4))
    v = rng.choice(_E2M1_VALUES, (rows, heads, 4, 32)) * rng.choice([-1.0, 1.0], (rows, heads, 4, 32))
    v[..., 0] = 6.0 * rng.choice([-1.0, 1.0], (rows, heads, 4))
    return (v * np.ldexp(1.0, k)[..., None]).reshape(rows, heads, 128).astype(np.float32)


def _hand_cache(rng, fmt, num_pages, stride):
    """Random codes and scale bytes written at the placement's byte positions;
    returns (cache, values [num_pages, 64, 128])."""
    codes = rng.integers(0, 16, (num_pages, 64, 128)).astype(np.uint8)
    sbytes = rng.integers(123, 132, (num_pages, 64, 4)).astype(np.uint8)          # 2^-4 .. 2^4
    vals = _code_value(codes) * np.ldexp(1.0, sbytes.astype(np.int64) - 127).repeat(32, axis=2)
    pairs = codes[..., 0::2] | (codes[..., 1::2] << 4)                             # [pages, 64, 64]
    cache = np.zeros(num_pages * stride, np.uint8)
    for p in range(num_pages):
        base = p * stride
        for t in range(64):
            if fmt == "mxfp4":
                cache[base + t * 64: base + t * 64 + 64] = pairs[p, t]
                cache[base + 4096 + t * 4: base + 4096 + t * 4 + 4] = sbytes[p, t]
            else:
                for g in range(4):
                    cache[base + g * 1024 + t * 16: base + g * 1024 + t * 16 + 16] = pairs[p, t, 16 * g:16 * g + 16]
                    cache[base + 4096 + g * 64 + t] = sbytes[p, t, g]
    return cache, vals


@pytest.mark.parametrize("heads", [16, 32, 64])
@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp4_rg"])
def test_score_heads_closed_form(heads, fmt):
    rng = np.random.default_rng(heads + (0 if fmt == "mxfp4" else 1000))
    num_pages, stride = 7, 4352 + 32
    cache, vals = _hand_cache(rng, fmt, num_pages, stride)
    qlen = np.array([2, 1, 3], np.int32)
    seq = np.array([150, 1, 260], np.int32)
    rows = int(qlen.sum()) + 1                                                     # one padding row
    x = _grid_queries(rng, rows, heads)
    payload, scales = O.quantize_queries(x)
    w = rng.standard_normal((rows, heads))
    starts, row_ends = O.decode_layout(seq, qlen, rows)
    bt = np.full((3, 5), -1, np.int32)
    perm = rng.permutation(num_pages)
    bt[0, :3], bt[1, :1], bt[2, :5] = perm[:3], perm[3:4], np.r_[perm[4:7], perm[0:2]]
    got = O.score_paged_heads(fmt, payload, scales, w, cache, stride, bt, starts, row_ends)
    assert got.shape == (rows, 5 * 64)
    xv = x.astype(np.float64)
    for q in range(3):
        for r in range(starts[q], starts[q + 1]):
            n = int(row_ends[r])
            for t in range(n):
                k = vals[bt[q, t // 64], t % 64]
                # every product is a multiple of 2^-9 below 2^13: the dot products are exact,
                # only the weighted head sum rounds (in a different order here)
                relu = [max(0.0, float(np.dot(xv[r, h], k))) for h in range(heads)]
                want = sum(w[r, h] * relu[h] for h in range(heads))
                mag = sum(abs(w[r, h]) * relu[h] for h in range(heads))
                assert abs(got[r, t] - want) <= 1e-13 * mag, (q, r, t, got[r, t], want)
            assert np.all(np.isneginf(got[r, n:]))
    assert np.all(np.isneginf(got[rows - 1]))                                      # the padding row


def test_score_heads_32_equals_the_query_row_path():
    """With 32 heads, quantize_queries' payload and scales score exactly as the
    "mxfp4_rg" query rows of quantize_query that carry the same bytes."""
    rng = np.random.default_rng(3)
    num_pages, stride = 5, 4352
    cache, _ = _hand_cache(rng, "mxfp4_rg", num_pages, stride)
    q = rng.standard_normal((4, 32, 128)).astype(np.float32)
    wv = rng.standard_normal((4, 32)).astype(np.float32)
    q_rows, w = O.quantize_query("mxfp4_rg", q, wv)
    payload, scales = O.quantize_queries(q)
    starts, row_ends = O.decode_layout(np.array([300, 250], np.int32), np.array([3, 1], np.int32), 4)
    bt = rng.permutation(num_pages)[:5].reshape(1, 5).repeat(2, axis=0).astype(np.int32)
    a = O.score_paged("mxfp4_rg", q_rows, w, cache, stride, bt, starts, row_ends)
    b = O.score_paged_heads("mxfp4_rg", payload, scales, w, cache, stride, bt, starts, row_ends)
    assert np.array_equal(a, b)


def test_score_heads_rejects_bad_shapes():
    z = np.zeros((2, 24, 64), np.uint8)
    with pytest.raises(ValueError):
        O.score_paged_heads("mxfp4", z, np.zeros((2, 256), np.uint8), np.zeros((2, 24)), np.zeros(4352, np.uint8),
                            4352, np.zeros((1, 1), np.int32), np.array([0, 2]), np.array([1, 1]))
    with pytest.raises(ValueError):
        O.score_paged_heads("fp8", np.zeros((2, 32, 64), np.uint8), np.zeros((2, 256), np.uint8),
                            np.zeros((2, 32)), np.zeros(8448, np.uint8), 8448, np.zeros((1, 1), np.int32),
                            np.array([0, 2]), np.array([1, 1]))
