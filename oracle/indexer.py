"""Plain CPU oracle of the DSA lightning-indexer decode step.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA path.

It follows three pages: *cutedsl.dsa.index* (query quantisation, key
LayerNorm + quantise + insert, cache and query-row layouts), *cutedsl.dsa.overlap*
(the order "wq_b -> DsaIndex -> scoring and top-k") and *amd.ops.fp4_indexer*
(``decode_layout``, ``score_paged``, ``store_keys``).  Where the pages leave
a step open, the docstring states the reading taken ("a reading").

Precision: FP32 where the pages compute in FP32 (LayerNorm, the scale and
weight folds), exact arithmetic for the scale exponents, FP64 for the scores.
Dot products of decoded E4M3/E2M1 values times powers of two are exact in
FP64 at these sizes, so the only rounding in a score is the FP64 weighted sum
over heads.
"""

from __future__ import annotations

import numpy as np

from .codecs import (
    bf16_round,
    e2m1_decode,
    e2m1_encode,
    e4m3_decode,
    e4m3_encode,
    pack_e2m1,
    pow2_exponent,
    unpack_e2m1,
)

HEADS, DIM, PAGE = 32, 128, 64
Q_ROW_BYTES = HEADS * DIM            # one FP8 query row: 32 heads x 128 E4M3
FP4_SCALES = HEADS * DIM // 2        # not printed; a reading: scale bytes follow the 32 x 64 B of E2M1
FP4_QUERY_ROW = FP4_SCALES + HEADS * 4
FP8_KEY_BYTES, FP8_PAGE_BYTES = PAGE * DIM, PAGE * (DIM + 4)          # 8192, 8448
FP4_KEY_BYTES, FP4_PAGE_BYTES = PAGE * DIM // 2, PAGE * (DIM // 2 + 4)  # 4096, 4352
WEIGHT_SCALE = (HEADS * DIM) ** -0.5   # 1/64, page *cutedsl.dsa.index*, ``DsaIndex.fp8_query``
# "the indexer weight scale" is not printed; a reading: the FP8 fold's 1/64
FP4_WEIGHT = WEIGHT_SCALE
FP8_AMAX_FLOOR = np.float32(1e-10)     # ``DsaIndex.fp8_query``: amax starts at 1e-10
MX_AMAX_FLOOR = 6.0 * 2.0 ** -126      # ``mxfp4_scale``: max(amax, 6 * 2^-126)

FORMATS = ("fp8", "fp8_mx", "mxfp4", "mxfp4_rg")
# "mxfp4_rg" (page *amd.ops.fp4_indexer*, ``cache_views``): the MXFP4 codes and
# scales of "mxfp4" placed group-major ("row-group") within the 4352-byte page
# section: payload byte j of column group g of token t at g * 1024 + t * 16 + j,
# the group's UE8M0 byte at 4096 + g * 64 + t (a reading: the page prints
# the views' strides, not their writer).
RG_GROUP_BYTES, RG_SCALE_GROUP = 1024, 64
# Row-group query scales (page *amd.ops.fp4_indexer*, ``quantize_queries``: a
# [rows, 1, 4, 16, 4] uint8 tensor, 256 bytes a row): the scale of block g of
# head h at g * 64 + h, group-major like the cache's scale views (a reading:
# the page fixes the shape, not the order).
RG_QUERY_HEAD_SLOTS = 64
RG_QUERY_HEADS = (16, 32, 64)


def _fp4(fmt: str) -> bool:
    return fmt in ("mxfp4", "mxfp4_rg")


def page_bytes(fmt: str) -> int:
    return FP4_PAGE_BYTES if _fp4(fmt) else FP8_PAGE_BYTES


# --------------------------------------------------------------------------
# scales
# --------------------------------------------------------------------------

def fp8_scale_exponent(amax) -> np.ndarray:
    """Exponent e of the FP8 power-of-two scale: the smallest e with
    ``448 * 2**e >= amax`` (a reading: ``pow2_ceil(amax / 448)`` in exact arithmetic;
    page *cutedsl.dsa.index*, ``DsaIndex.fp8_query``)."""
    return pow2_exponent(np.asarray(amax, dtype=np.float64), 448.0)


def mx_scale_exponent(amax) -> np.ndarray:
    """Exponent of an MXFP4 block scale (page *cutedsl.dsa.index*, ``mxfp4_scale``):
    ``clamp(ceil(log2(max(amax, 6 * 2^-126) / 6)), -127, 127)``, taken as an exact
    mathematical definition (a reading: the page's compiled ``log2`` sequence is not
    reproduced)."""
    a = np.maximum(np.asarray(amax, dtype=np.float64), MX_AMAX_FLOOR)
    return np.clip(pow2_exponent(a, 6.0), -127, 127)


# --------------------------------------------------------------------------
# query quantisation
# --------------------------------------------------------------------------

def quantize_query(fmt: str, q, wv):
    """Quantise indexer query rows (page *cutedsl.dsa.index*, ``DsaIndex.kernel``,
    ``DsaIndex.fp8_query``, ``quantize_fp4_query``, ``fp4_query_views``).

    q: float32 [rows, 32, 128] (BF16 values); wv: float32 [rows, 32] (BF16 values).
    Returns (q_rows uint8 [rows, 4096], w float32 [rows, 32] holding BF16 values).
    FP8 rows hold head h's 128 E4M3 codes at ``h * 128``.  MXFP4 rows hold
    head h's E2M1 pairs at ``h * 64`` and its four UE8M0 bytes (block b at
    byte b, a reading) at ``2048 + h * 4``; bytes from 2176 on are left zero.
    Row-group MXFP4 ("mxfp4_rg") rows hold the same pairs and the scale of
    block b of head h at ``2048 + b * 64 + h`` (group-major, a reading); the slots of heads 32..63
    and bytes from 2304 on are left zero."""
    q = np.asarray(q, dtype=np.float32)
    wv = np.asarray(wv, dtype=np.float32)
    rows = q.shape[0]
    out = np.zeros((rows, Q_ROW_BYTES), dtype=np.uint8)
    if fmt in ("fp8", "fp8_mx"):
        amax = np.maximum(np.abs(q).max(axis=2), FP8_AMAX_FLOOR)           # [rows, 32]
        e = fp8_scale_exponent(amax)
        codes = e4m3_encode(q.astype(np.float64) * np.ldexp(1.0, -e)[..., None])
        out[:, :] = codes.reshape(rows, Q_ROW_BYTES)
        scale = np.ldexp(np.float32(1.0), e).astype(np.float32)
        fold = (wv * scale).astype(np.float32) * np.float32(WEIGHT_SCALE)
        w = bf16_round(fold.astype(np.float32))
    elif _fp4(fmt):
        blocks = q.reshape(rows, HEADS, 4, 32).astype(np.float64)
        e = mx_scale_exponent(np.abs(blocks).max(axis=3))                   # [rows, 32, 4]
        codes = e2m1_encode(blocks * np.ldexp(1.0, -e)[..., None]).reshape(rows, HEADS, DIM)
        out[:, :FP4_SCALES] = pack_e2m1(codes).reshape(rows, FP4_SCALES)
        if fmt == "mxfp4_rg":
            sc = np.zeros((rows, 4, RG_QUERY_HEAD_SLOTS), np.uint8)
            sc[:, :, :HEADS] = (e + 127).astype(np.uint8).transpose(0, 2, 1)
            out[:, FP4_SCALES:FP4_SCALES + sc.shape[1] * sc.shape[2]] = sc.reshape(rows, -1)
        else:
            out[:, FP4_SCALES:FP4_QUERY_ROW] = (e + 127).astype(np.uint8).reshape(rows, HEADS * 4)
        w = bf16_round((wv * np.float32(FP4_WEIGHT)).astype(np.float32))
    else:
        raise ValueError(f"unknown format {fmt!r}")
    return out, w


def quantize_queries(q):
    """Page *amd.ops.fp4_indexer*, ``quantize_queries``: MXFP4 of q float32
    [rows, heads, 128] (BF16 values), heads in {16, 32, 64}, with no scale
    folded into head weights.  Returns (payload uint8 [rows, heads, 64]: head
    h's E2M1 pairs, column 2j in the low nibble of byte j; scales uint8
    [rows, 1, 4, 16, 4]: the UE8M0 byte of block g of head h at flat position
    g * 64 + h of the row's 256 bytes, group-major (a reading); slots of
    heads >= ``heads`` zero).  The codec is the one of ``quantize_query``'s
    MXFP4 rows."""
    q = np.asarray(q, dtype=np.float32)
    if q.ndim != 3 or q.shape[2] != DIM:
        raise ValueError("queries must be [rows, heads, 128]")
    rows, heads = q.shape[0], q.shape[1]
    if heads not in RG_QUERY_HEADS:
        raise ValueError("row-group queries support 16, 32 or 64 heads")
    blocks = q.reshape(rows, heads, 4, 32).astype(np.float64)
    e = mx_scale_exponent(np.abs(blocks).max(axis=3))                       # [rows, heads, 4]
    codes = e2m1_encode(blocks * np.ldexp(1.0, -e)[..., None]).reshape(rows, heads, DIM)
    payload = pack_e2m1(codes).reshape(rows, heads, DIM // 2)
    flat = np.zeros((rows, 4, RG_QUERY_HEAD_SLOTS), np.uint8)
    flat[:, :, :heads] = (e + 127).astype(np.uint8).transpose(0, 2, 1)
    return payload, flat.reshape(rows, 1, 4, 16, 4)


# --------------------------------------------------------------------------
# key LayerNorm + quantise + insert
# --------------------------------------------------------------------------

def _half_warp_sum(lane_values: np.ndarray) -> np.ndarray:
    """Sum over 16 lanes by an xor butterfly with distances 8, 4, 2, 1 (a reading: the
    order is not printed);
    every lane ends with the same FP32 value."""
    s = lane_values.astype(np.float32)
    lane = np.arange(16)
    for d in (8, 4, 2, 1):
        s = (s + s[:, lane ^ d]).astype(np.float32)
    return s[:, 0]


def layer_norm_bf16(x, gamma, beta, eps):
    """LayerNorm (FP32) of 128-column keys rounded to BF16 (page *cutedsl.dsa.index*,
    ``insert_key``).  Lane j of a half-warp holds columns 8j..8j+7; its 8 values
    are summed in order, the 16 lane sums are combined by ``_half_warp_sum``;
    mean = sum / 128; the variance repeats the scheme on (x - mean)^2;
    rstd = 1 / sqrt(var + eps) with a correctly rounded square root and
    division; y = ((x - mean) * rstd) * gamma + beta, every operation rounded
    on its own (no fused multiply-add), then BF16 (a reading: the order and
    rounding are not printed)."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    X = x.reshape(n, 16, 8)
    total = np.zeros((n, 16), dtype=np.float32)
    for i in range(8):
        total = (total + X[:, :, i]).astype(np.float32)
    mean = (_half_warp_sum(total) / np.float32(DIM)).astype(np.float32)
    D = (X - mean[:, None, None]).astype(np.float32)
    square = np.zeros((n, 16), dtype=np.float32)
    for i in range(8):
        square = (square + (D[:, :, i] * D[:, :, i]).astype(np.float32)).astype(np.float32)
    variance = (_half_warp_sum(square) / np.float32(DIM)).astype(np.float32)
    rstd = (np.float32(1.0) / np.sqrt((variance + np.float32(eps)).astype(np.float32))).astype(np.float32)
    g = np.asarray(gamma, dtype=np.float32).reshape(16, 8)
    b = np.asarray(beta, dtype=np.float32).reshape(16, 8)
    y = ((D * rstd[:, None, None]).astype(np.float32) * g).astype(np.float32)
    y = (y + b).astype(np.float32)
    return bf16_round(y).reshape(n, DIM)


def quantize_key(fmt: str, normed):
    """Codes and scale bytes of BF16-valued normalised keys [n, 128].

    FP8 (a reading: ``insert_fp8_key`` is not printed): amax over the 128
    values, floored at 1e-10; scale ``2**e`` with e from
    ``fp8_scale_exponent``; 128 E4M3 codes and 4 scale bytes: FP32 ``2**e``
    little-endian ("fp8"), or the byte ``e + 127`` four times ("fp8_mx", page
    *cutedsl.dsa.index*, module docstring).
    MXFP4 (``insert_fp4_key``): per 32-column block b a UE8M0 exponent as in
    ``mx_scale_exponent``; 64 bytes of E2M1 pairs and 4 scale bytes (block b at
    byte b)."""
    normed = np.asarray(normed, dtype=np.float32)
    n = normed.shape[0]
    if fmt in ("fp8", "fp8_mx"):
        amax = np.maximum(np.abs(normed).max(axis=1), FP8_AMAX_FLOOR)
        e = fp8_scale_exponent(amax)
        codes = e4m3_encode(normed.astype(np.float64) * np.ldexp(1.0, -e)[:, None])
        if fmt == "fp8":
            scale = np.ldexp(np.float32(1.0), e).astype("<f4")
            scale_bytes = scale.view(np.uint8).reshape(n, 4)
        else:
            scale_bytes = np.repeat((e + 127).astype(np.uint8)[:, None], 4, axis=1)
        return codes.astype(np.uint8), scale_bytes
    if _fp4(fmt):
        blocks = normed.reshape(n, 4, 32).astype(np.float64)
        e = mx_scale_exponent(np.abs(blocks).max(axis=2))
        codes = e2m1_encode(blocks * np.ldexp(1.0, -e)[..., None]).reshape(n, DIM)
        return pack_e2m1(codes), (e + 127).astype(np.uint8)
    raise ValueError(f"unknown format {fmt!r}")


def insert_key(fmt: str, cache: np.ndarray, page_stride: int, num_pages: int,
               x, gamma, beta, eps, slots) -> int:
    """LayerNorm + quantise + insert keys into a paged cache, in place.

    cache: uint8 array of at least ``num_pages * page_stride`` bytes.  A slot is
    ``page * 64 + offset`` (page *cutedsl.dsa.index*, ``insert_fp4_key``).  A page
    holds the 64 tokens' codes, then their 4-byte scales: FP8 codes at
    ``offset * 128``, scales at ``8192 + offset * 4`` (a reading); MXFP4 codes at
    ``offset * 64``, scales at ``64 * 64 + offset * 4``.  Slots < 0 are padding
    and write nothing (``insert_key``; *amd.ops.fp4_indexer*, ``store_keys``).
    Slots at or past ``num_pages * 64`` are skipped too; the return value
    counts them."""
    slots = np.asarray(slots, dtype=np.int64)
    if slots.size == 0:
        return 0
    normed = layer_norm_bf16(x, gamma, beta, eps)
    codes, scale_bytes = quantize_key(fmt, normed)
    flat = cache.reshape(-1)
    inside = slots < num_pages * PAGE
    bad = int(np.count_nonzero((slots >= 0) & ~inside))
    # keys written in order: where a slot repeats, the last key's bytes stay
    order = np.arange(slots.size)[(slots >= 0) & inside]
    _, last = np.unique(slots[order][::-1], return_index=True)
    keep = order[::-1][last]
    page, off = np.divmod(slots[keep], PAGE)
    base = page * page_stride
    if fmt == "mxfp4_rg":
        for g in range(4):
            flat[(base + g * RG_GROUP_BYTES + off * 16)[:, None] + np.arange(16)] = codes[keep, g * 16:(g + 1) * 16]
            flat[base + FP4_KEY_BYTES + g * RG_SCALE_GROUP + off] = scale_bytes[keep, g]
        return bad
    code_bytes = DIM if not _fp4(fmt) else DIM // 2
    scale_base = PAGE * code_bytes
    flat[(base + off * code_bytes)[:, None] + np.arange(code_bytes)] = codes[keep]
    flat[(base + scale_base + off * 4)[:, None] + np.arange(4)] = scale_bytes[keep]
    return bad


# --------------------------------------------------------------------------
# row bounds of grouped verify rows
# --------------------------------------------------------------------------

def decode_layout(seq_lens, query_lens, num_rows: int):
    """Row grouping and causal key bounds (page *amd.ops.fp4_indexer*,
    ``decode_layout``, without the DCP branch).

    starts = [0, cumsum(query_lens)] (int32).  Row r belongs to the request
    found by ``searchsorted(starts[1:], r, right=True)`` capped at R - 1;
    its bound is ``max(0, seq_len - query_len + (r - start) + 1)``.  Rows at
    or past ``starts[-1]`` are padding with bound 0 (as printed)."""
    if num_rows < 0:
        raise ValueError("Invalid DCP geometry or query row count")
    seq_lens = np.asarray(seq_lens)
    query_lens = np.asarray(query_lens)
    if seq_lens.ndim != 1 or query_lens.ndim != 1:
        raise ValueError("Sequence and query lengths must be one-dimensional")
    if seq_lens.size < query_lens.size:
        raise ValueError("Each decode request requires a global sequence length")
    starts = np.concatenate([[0], np.cumsum(query_lens.astype(np.int64))]).astype(np.int32)
    rows = np.arange(num_rows, dtype=np.int64)
    R = query_lens.size
    if R == 0:
        return starts, np.zeros(num_rows, dtype=np.int32)
    req = np.minimum(np.searchsorted(starts[1:], rows, side="right"), R - 1)
    ends = seq_lens[req].astype(np.int64) - query_lens[req] + rows - starts[req] + 1
    ends = np.maximum(ends, 0)
    return starts, np.where(rows < starts[-1], ends, 0).astype(np.int32)


# --------------------------------------------------------------------------
# paged MQA logits
# --------------------------------------------------------------------------

def decode_query(fmt: str, q_row) -> np.ndarray:
    """float64 [32, 128] values of one quantised query row.  FP8 rows carry
    plain E4M3 codes (their scale is folded into the head weights); MXFP4 rows
    carry E2M1 codes times their block scales."""
    q_row = np.asarray(q_row, dtype=np.uint8)
    if fmt in ("fp8", "fp8_mx"):
        return e4m3_decode(q_row[:Q_ROW_BYTES]).reshape(HEADS, DIM)
    codes = unpack_e2m1(q_row[:FP4_SCALES].reshape(HEADS, DIM // 2))
    if fmt == "mxfp4_rg":
        sc = q_row[FP4_SCALES:FP4_SCALES + 4 * RG_QUERY_HEAD_SLOTS].reshape(4, RG_QUERY_HEAD_SLOTS)
        e = sc[:, :HEADS].T.astype(np.int64) - 127
    else:
        e = q_row[FP4_SCALES:FP4_QUERY_ROW].reshape(HEADS, 4).astype(np.int64) - 127
    return (e2m1_decode(codes).reshape(HEADS, 4, 32) * np.ldexp(1.0, e)[..., None]).reshape(HEADS, DIM)


def decode_keys(fmt: str, cache: np.ndarray, page_stride: int, pages, n: int) -> np.ndarray:
    """float64 [n, 128] values of positions 0..n-1 of a request whose block-table
    row is ``pages``.  FP8: codes times the token scale (FP32 for "fp8"; for
    "fp8_mx" byte b scales columns 32b..32b+31 as an MX block, which with the
    four equal bytes the writer stores is the token's one scale).  MXFP4:
    E2M1 codes times each block's UE8M0 scale."""
    flat = cache.reshape(-1)
    t = np.arange(n, dtype=np.int64)
    page = np.asarray(pages, dtype=np.int64)[t // PAGE]
    off = t % PAGE
    base = page * page_stride
    if fmt in ("fp8", "fp8_mx"):
        code_idx = (base + off * DIM)[:, None] + np.arange(DIM)
        vals = e4m3_decode(flat[code_idx])
        sidx = (base + FP8_KEY_BYTES + off * 4)[:, None] + np.arange(4)
        sb = flat[sidx]
        if fmt == "fp8":
            scale = sb.copy().view("<f4").reshape(n).astype(np.float64)
            return vals * scale[:, None]
        e = sb.astype(np.int64) - 127
        return (vals.reshape(n, 4, 32) * np.ldexp(1.0, e)[..., None]).reshape(n, DIM)
    if fmt == "mxfp4_rg":
        j = np.arange(DIM // 2)
        code_idx = base[:, None] + (j // 16) * RG_GROUP_BYTES + off[:, None] * 16 + j % 16
        sidx = base[:, None] + FP4_KEY_BYTES + np.arange(4) * RG_SCALE_GROUP + off[:, None]
    else:
        code_idx = (base + off * (DIM // 2))[:, None] + np.arange(DIM // 2)
        sidx = (base + FP4_KEY_BYTES + off * 4)[:, None] + np.arange(4)
    codes = unpack_e2m1(flat[code_idx])
    e = flat[sidx].astype(np.int64) - 127
    return (e2m1_decode(codes).reshape(n, 4, 32) * np.ldexp(1.0, e)[..., None]).reshape(n, DIM)


def decode_queries(payload_row, scales_row) -> np.ndarray:
    """float64 [heads, 128] values of one row of ``quantize_queries``' output:
    payload [heads, 64] (E2M1 pairs) and the row's 256 scale bytes, block g of
    head h at g * 64 + h (page *amd.ops.fp4_indexer*, ``quantize_queries``; the
    group-major order is a reading)."""
    payload_row = np.asarray(payload_row, dtype=np.uint8)
    heads = payload_row.shape[0]
    codes = unpack_e2m1(payload_row)                                        # [heads, 128]
    sc = np.asarray(scales_row, dtype=np.uint8).reshape(4, RG_QUERY_HEAD_SLOTS)
    e = sc[:, :heads].T.astype(np.int64) - 127                              # [heads, 4]
    return (e2m1_decode(codes).reshape(heads, 4, 32) * np.ldexp(1.0, e)[..., None]).reshape(heads, DIM)


def relu_weighted(Q: np.ndarray, w_row, keys: np.ndarray) -> np.ndarray:
    """score[t] = sum_h w_h * ReLU(q_h . k_t) in float64 for decoded queries Q
    [heads, 128] and keys [n, 128] (page *cutedsl.dsa.index*, module docstring;
    *amd.ops.fp4_indexer*, ``score_paged``)."""
    dots = keys @ Q.T                                   # [n, heads], exact
    return np.maximum(dots, 0.0) @ np.asarray(w_row, dtype=np.float64)


def score_row(fmt: str, q_row, w_row, keys: np.ndarray) -> np.ndarray:
    """score[t] = sum_h w_h * ReLU(q_h . k_t) in float64 for one 32-head query
    row of ``quantize_query``."""
    return relu_weighted(decode_query(fmt, q_row), w_row, keys)


def score_paged(fmt: str, q_rows, w, cache, page_stride: int, block_table,
                starts, row_ends, rows_subset=None):
    """Logits float64 [rows, max_pages * 64] of every query row against the
    keys of its request's block-table row; positions at or past the row's
    bound are -inf (a reading: the page leaves them unset).  ``rows_subset``
    restricts the work to some rows (the others stay -inf)."""
    block_table = np.asarray(block_table)
    starts = np.asarray(starts, dtype=np.int64)
    row_ends = np.asarray(row_ends, dtype=np.int64)
    rows = row_ends.shape[0]
    width = block_table.shape[1] * PAGE
    out = np.full((rows, width), -np.inf, dtype=np.float64)
    R = starts.shape[0] - 1
    wanted = None if rows_subset is None else set(int(r) for r in rows_subset)
    for q in range(R):
        rs = [r for r in range(int(starts[q]), int(starts[q + 1]))
              if r < rows and (wanted is None or r in wanted)]
        rs = [r for r in rs if row_ends[r] > 0]
        if not rs:
            continue
        n = int(max(row_ends[r] for r in rs))
        keys = decode_keys(fmt, cache, page_stride, block_table[q], n)
        for r in rs:
            e = int(row_ends[r])
            out[r, :e] = score_row(fmt, q_rows[r], w[r], keys[:e])
    return out


def score_paged_heads(fmt: str, payload, scales, w, cache, page_stride: int, block_table,
                      starts, row_ends, rows_subset=None):
    """Logits of MXFP4 queries with 16, 32 or 64 heads against an MXFP4 cache in
    either placement (page *amd.ops.fp4_indexer*, ``score_paged``: queries
    quantised by ``quantize_queries``, weights [rows, heads] carrying the head
    factors but no group scales).  payload uint8 [rows, heads, 64]; scales
    uint8 [rows, 1, 4, 16, 4] (or [rows, 256]); w [rows, heads].  Rows,
    bounds and -inf fill as ``score_paged``."""
    if not _fp4(fmt):
        raise ValueError("queries of quantize_queries score against MXFP4 caches")
    payload = np.asarray(payload, dtype=np.uint8)
    if payload.ndim != 3 or payload.shape[1] not in RG_QUERY_HEADS or payload.shape[2] != DIM // 2:
        raise ValueError("payload must be [rows, heads, 64] with heads 16, 32 or 64")
    scales = np.asarray(scales, dtype=np.uint8).reshape(payload.shape[0], 4 * RG_QUERY_HEAD_SLOTS)
    w = np.asarray(w, dtype=np.float64)
    block_table = np.asarray(block_table)
    starts = np.asarray(starts, dtype=np.int64)
    row_ends = np.asarray(row_ends, dtype=np.int64)
    rows = row_ends.shape[0]
    width = block_table.shape[1] * PAGE
    out = np.full((rows, width), -np.inf, dtype=np.float64)
    wanted = None if rows_subset is None else set(int(r) for r in rows_subset)
    for q in range(starts.shape[0] - 1):
        rs = [r for r in range(int(starts[q]), int(starts[q + 1]))
              if r < rows and (wanted is None or r in wanted) and row_ends[r] > 0]
        if not rs:
            continue
        n = int(max(row_ends[r] for r in rs))
        keys = decode_keys(fmt, cache, page_stride, block_table[q], n)
        for r in rs:
            e = int(row_ends[r])
            out[r, :e] = relu_weighted(decode_queries(payload[r], scales[r]), w[r], keys[:e])
    return out


# --------------------------------------------------------------------------
# top-k
# --------------------------------------------------------------------------

def topk(scores, row_ends, k: int) -> np.ndarray:
    """Per row, the positions t < row_end of the k largest scores, ordered by
    (score descending, t ascending); rows with fewer than k candidates are
    filled with -1 (a reading: the pages do not say).  Indices are logical
    positions in the request."""
    scores = np.asarray(scores)
    rows = scores.shape[0]
    out = np.full((rows, k), -1, dtype=np.int32)
    for r in range(rows):
        n = int(row_ends[r])
        if n <= 0 or k <= 0:
            continue
        s = scores[r, :n]
        order = np.lexsort((np.arange(n), -s))
        m = min(k, n)
        out[r, :m] = order[:m]
    return out
