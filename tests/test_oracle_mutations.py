"""The oracle's pins catch plausible mistakes: each case below plants one
mistake in the oracle (on the CPU, for the duration of the case) and checks
that at least one of the pins named with it fails.  A dropped term, a wrong
sign, order or index, or a transposed operand in any step must show up."""

import numpy as np
import pytest

from oracle import codecs as C
from oracle import dcp as D
from oracle import indexer as O
from oracle import query_norm as QN

import test_oracle_codecs as TC
import test_oracle_dcp as TD
import test_oracle_indexer as TI
import test_oracle_query_norm as TQ
import test_oracle_rowgroup as TR

_orig = {name: getattr(O, name) for name in (
    "score_row", "decode_query", "decode_keys", "decode_layout", "topk", "fp8_scale_exponent",
    "mx_scale_exponent", "layer_norm_bf16", "_half_warp_sum", "quantize_queries", "score_paged")}
_orig_rank_local_ends = D.rank_local_ends
_orig_quantize_query = O.quantize_query
_orig_quantize_key = O.quantize_key


# ---------------------------------------------------------------- planted mistakes

def score_without_relu(fmt, q_row, w_row, keys):
    return (keys @ O.decode_query(fmt, q_row).T) @ np.asarray(w_row, np.float64)


def score_weights_reversed(fmt, q_row, w_row, keys):
    dots = keys @ O.decode_query(fmt, q_row).T
    return np.maximum(dots, 0.0) @ np.asarray(w_row, np.float64)[::-1]


def score_relu_after_weighting(fmt, q_row, w_row, keys):
    dots = keys @ O.decode_query(fmt, q_row).T
    return np.maximum(dots * np.asarray(w_row, np.float64), 0.0).sum(axis=1)


def query_heads_transposed(fmt, q_row):
    if fmt in ("fp8", "fp8_mx"):
        return C.e4m3_decode(np.asarray(q_row, np.uint8)[:O.Q_ROW_BYTES]).reshape(O.DIM, O.HEADS).T
    return _orig["decode_query"](fmt, q_row)


def _keys_fp8_unscaled(cache, page_stride, pages, n):
    flat = cache.reshape(-1)
    t = np.arange(n, dtype=np.int64)
    base = np.asarray(pages, np.int64)[t // O.PAGE] * page_stride
    return C.e4m3_decode(flat[(base + (t % O.PAGE) * O.DIM)[:, None] + np.arange(O.DIM)])


def keys_without_scale(fmt, cache, page_stride, pages, n):
    if fmt in ("fp8", "fp8_mx"):
        return _keys_fp8_unscaled(cache, page_stride, pages, n)
    return _orig["decode_keys"](fmt, cache, page_stride, pages, n)


def keys_block_scales_reversed(fmt, cache, page_stride, pages, n):
    if fmt != "mxfp4":
        return _orig["decode_keys"](fmt, cache, page_stride, pages, n)
    flat = cache.reshape(-1)
    t = np.arange(n, dtype=np.int64)
    base = np.asarray(pages, np.int64)[t // O.PAGE] * page_stride
    off = t % O.PAGE
    codes = C.unpack_e2m1(flat[(base + off * (O.DIM // 2))[:, None] + np.arange(O.DIM // 2)])
    e = flat[(base + O.FP4_KEY_BYTES + off * 4)[:, None] + np.arange(4)[::-1]].astype(np.int64) - 127
    return (C.e2m1_decode(codes).reshape(n, 4, 32) * np.ldexp(1.0, e)[..., None]).reshape(n, O.DIM)


def layout_bound_one_short(seq_lens, query_lens, num_rows):
    starts, ends = _orig["decode_layout"](seq_lens, query_lens, num_rows)
    return starts, np.maximum(ends - 1, 0).astype(np.int32)


def layout_request_off_by_one(seq_lens, query_lens, num_rows):
    starts, ends = _orig["decode_layout"](seq_lens, query_lens, num_rows)
    return starts, np.roll(ends, 1).astype(np.int32)


def _topk_by(order_fn):
    def f(scores, row_ends, k):
        scores = np.asarray(scores)
        out = np.full((scores.shape[0], k), -1, np.int32)
        for r in range(scores.shape[0]):
            n = int(row_ends[r])
            if n <= 0 or k <= 0:
                continue
            order = order_fn(scores[r, :n], n)
            out[r, :min(k, n)] = order[:min(k, n)]
        return out
    return f


topk_ascending = _topk_by(lambda s, n: np.lexsort((np.arange(n), s)))
topk_ties_last_position_first = _topk_by(lambda s, n: np.lexsort((-np.arange(n), -s)))


def fp8_exponent_one_high(amax):
    return _orig["fp8_scale_exponent"](amax) + 1


def mx_exponent_floor(amax):
    a = np.maximum(np.asarray(amax, np.float64), O.MX_AMAX_FLOOR)
    return np.clip(np.floor(np.log2(a / 6.0)), -127, 127).astype(np.int64)


def layer_norm_without_beta(x, gamma, beta, eps):
    return _orig["layer_norm_bf16"](x, gamma, np.zeros_like(np.asarray(beta, np.float32)), eps)


def _layer_norm_variant(eps_outside=False, fused=False):
    """The oracle's LayerNorm with the square root's eps or the output's
    rounding changed (the rest as in the oracle)."""
    def ln(x, gamma, beta, eps):
        x = np.asarray(x, np.float32)
        n = x.shape[0]
        X = x.reshape(n, 16, 8)
        total = np.zeros((n, 16), np.float32)
        for i in range(8):
            total = (total + X[:, :, i]).astype(np.float32)
        mean = (O._half_warp_sum(total) / np.float32(O.DIM)).astype(np.float32)
        Dv = (X - mean[:, None, None]).astype(np.float32)
        square = np.zeros((n, 16), np.float32)
        for i in range(8):
            square = (square + (Dv[:, :, i] * Dv[:, :, i]).astype(np.float32)).astype(np.float32)
        var = (O._half_warp_sum(square) / np.float32(O.DIM)).astype(np.float32)
        if eps_outside:
            rstd = (np.float32(1.0) / (np.sqrt(var) + np.float32(eps))).astype(np.float32)
        else:
            rstd = (np.float32(1.0) / np.sqrt((var + np.float32(eps)).astype(np.float32))).astype(np.float32)
        g = np.asarray(gamma, np.float32).reshape(16, 8)
        b = np.asarray(beta, np.float32).reshape(16, 8)
        p = (Dv * rstd[:, None, None]).astype(np.float32)
        if fused:
            y = (p.astype(np.float64) * g + b).astype(np.float32)
        else:
            y = ((p * g).astype(np.float32) + b).astype(np.float32)
        return C.bf16_round(y).reshape(n, O.DIM)
    return ln


def lanes_left_to_right(lane_values):
    s = np.zeros(lane_values.shape[0], np.float32)
    for j in range(lane_values.shape[1]):
        s = (s + lane_values[:, j].astype(np.float32)).astype(np.float32)
    return s


def e4m3_truncating(x):
    """E4M3 codes rounding toward zero instead of to nearest even."""
    x = np.asarray(x, np.float64)
    codes = np.arange(0x7F)                                  # non-negative finite codes
    vals = np.array([C.E4M3_TABLE[c] for c in codes], np.float64)
    order = np.argsort(vals, kind="stable")
    vals, codes = vals[order], codes[order]
    idx = np.searchsorted(vals, np.minimum(np.abs(x), 448.0), side="right") - 1
    return (codes[np.maximum(idx, 0)] | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def query_nibbles_swapped(fmt, q, wv):
    rows, w = _orig_quantize_query(fmt, q, wv)
    if fmt in ("mxfp4", "mxfp4_rg"):
        b = rows[:, :O.FP4_SCALES].copy()
        rows[:, :O.FP4_SCALES] = ((b & 0xF) << 4) | (b >> 4)
    return rows, w


def fp8_query_heads_reversed(fmt, q, wv):
    rows, w = _orig_quantize_query(fmt, q, wv)
    if fmt in ("fp8", "fp8_mx"):
        rows[:, :O.Q_ROW_BYTES] = rows[:, :O.Q_ROW_BYTES].reshape(-1, O.HEADS, O.DIM)[:, ::-1].reshape(-1, O.Q_ROW_BYTES)
    return rows, w


def mxfp4_query_scales_block_major(fmt, q, wv):
    rows, w = _orig_quantize_query(fmt, q, wv)
    if fmt == "mxfp4":
        sc = rows[:, O.FP4_SCALES:O.FP4_QUERY_ROW]
        rows[:, O.FP4_SCALES:O.FP4_QUERY_ROW] = sc.reshape(-1, O.HEADS, 4).transpose(0, 2, 1).reshape(-1, O.HEADS * 4)
    return rows, w


def fp8_key_scale_big_endian(fmt, normed):
    codes, sc = _orig_quantize_key(fmt, normed)
    return (codes, sc[:, ::-1].copy()) if fmt == "fp8" else (codes, sc)


def mxfp4_key_scale_blocks_reversed(fmt, normed):
    codes, sc = _orig_quantize_key(fmt, normed)
    return (codes, sc[:, ::-1].copy()) if fmt == "mxfp4" else (codes, sc)


def fp8_key_codes_unscaled(fmt, normed):
    codes, sc = _orig_quantize_key(fmt, normed)
    if fmt in ("fp8", "fp8_mx"):
        codes = C.e4m3_encode(np.asarray(normed, np.float64)).reshape(codes.shape).astype(np.uint8)
    return codes, sc


def rows_scored_to_the_request_bound(fmt, q_rows, w, cache, page_stride, block_table, starts, row_ends,
                                     rows_subset=None):
    bounds = np.asarray(row_ends).copy()
    st = np.asarray(starts)
    for q in range(len(st) - 1):
        a, b = int(st[q]), int(st[q + 1])
        if b > a:
            bounds[a:b] = bounds[a:b].max()
    return _orig["score_paged"](fmt, q_rows, w, cache, page_stride, block_table, starts, bounds, rows_subset)


def every_request_reads_request_zero(fmt, q_rows, w, cache, page_stride, block_table, starts, row_ends,
                                     rows_subset=None):
    bt = np.asarray(block_table).copy()
    bt[:] = bt[0]
    return _orig["score_paged"](fmt, q_rows, w, cache, page_stride, bt, starts, row_ends, rows_subset)


def positions_paged_column_major(fmt, cache, page_stride, pages, n):
    """Position t read from page t mod P, offset t div P (P pages) instead of
    page t div 64, offset t mod 64."""
    if n == 0:
        return _orig["decode_keys"](fmt, cache, page_stride, pages, 0)
    npg = (n + 63) // 64
    full = _orig["decode_keys"](fmt, cache, page_stride, pages, npg * 64)
    t = np.arange(n)
    return full[(t % npg) * 64 + t // npg]


def queries_head_major_scales(q):
    payload, scales = _orig["quantize_queries"](q)
    rows, heads = payload.shape[0], payload.shape[1]
    by_group = scales.reshape(rows, 4, 64)
    flat = np.zeros((rows, 256), np.uint8)
    for h in range(heads):
        for g in range(4):
            flat[:, h * 4 + g] = by_group[:, g, h]
    return payload, flat.reshape(rows, 1, 4, 16, 4)


def keys_rowgroup_scales_token_major(fmt, cache, page_stride, pages, n):
    if fmt != "mxfp4_rg":
        return _orig["decode_keys"](fmt, cache, page_stride, pages, n)
    flat = cache.reshape(-1)
    t = np.arange(n, dtype=np.int64)
    base = np.asarray(pages, np.int64)[t // O.PAGE] * page_stride
    off = t % O.PAGE
    j = np.arange(O.DIM // 2)
    codes = C.unpack_e2m1(flat[base[:, None] + (j // 16) * O.RG_GROUP_BYTES + off[:, None] * 16 + j % 16])
    e = flat[(base + O.FP4_KEY_BYTES + off * 4)[:, None] + np.arange(4)].astype(np.int64) - 127
    return (C.e2m1_decode(codes).reshape(n, 4, 32) * np.ldexp(1.0, e)[..., None]).reshape(n, O.DIM)


def rsqrt_without_eps(total, eps):
    mean = (total.astype(np.float32) / np.float32(QN.COLS)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        return (np.float32(1.0) / np.sqrt(mean)).astype(np.float32)


def rsqrt_mean_over_one_column_less(total, eps):
    mean = (total.astype(np.float32) / np.float32(QN.COLS - 1)).astype(np.float32)
    return (np.float32(1.0) / np.sqrt((mean + np.float32(eps)).astype(np.float32))).astype(np.float32)


def warp_sum_left_to_right(lanes):
    s = np.zeros(lanes.shape[:-1], np.float32)
    for j in range(lanes.shape[-1]):
        s = (s + lanes[..., j].astype(np.float32)).astype(np.float32)
    return s


def scale_weight_first(x, rr, w):
    y = (x * w[None, :]).astype(np.float32)
    return C.bf16_round((y * rr[:, None]).astype(np.float32))


def owner_ignoring_interleave(t, world, interleave):
    return np.asarray(t, np.int64) % world


def rank_local_ends_partial_short(ends, rank, world, interleave):
    e = np.asarray(ends, np.int64)
    full = e // (world * interleave) * interleave
    return (full + np.clip(e - full * world - rank * interleave, 0, max(interleave - 1, 0))).astype(np.int32)


def local_to_global_without_rank(l, rank, world, interleave):
    l = np.asarray(l, np.int64)
    return (l // interleave) * (world * interleave) + l % interleave


def merge_ties_toward_later_position(scores, idx, world, interleave, k_out):
    scores = np.asarray(scores, np.float64)
    idx = np.asarray(idx, np.int64)
    out = np.full((scores.shape[0], k_out), -1, np.int32)
    ranks = np.broadcast_to(np.arange(world)[None, :, None], idx.shape)
    for r in range(scores.shape[0]):
        keep = idx[r] >= 0
        g = (idx[r][keep] // interleave) * (world * interleave) + idx[r][keep] % interleave + ranks[r][keep] * interleave
        order = np.lexsort((-g, -scores[r][keep]))
        m = min(k_out, order.size)
        out[r, :m] = g[order[:m]]
    return out


# ---------------------------------------------------------------- cases

CASES = [
    ("ReLU dropped", O, "score_row", score_without_relu, [TI.test_score_hand_cases_fp8]),
    ("head weights reversed", O, "score_row", score_weights_reversed, [TI.test_score_hand_cases_fp8]),
    ("ReLU applied after the head weight", O, "score_row", score_relu_after_weighting,
     [TI.test_score_matches_dequantised_float_reference]),
    ("query heads read transposed", O, "decode_query", query_heads_transposed, [TI.test_score_hand_cases_fp8]),
    ("FP8 key scale dropped", O, "decode_keys", keys_without_scale, [TI.test_score_hand_cases_fp8]),
    ("MXFP4 key block scales in reverse byte order", O, "decode_keys", keys_block_scales_reversed,
     [TI.test_score_matches_dequantised_float_reference]),
    ("row bound one short", O, "decode_layout", layout_bound_one_short, [TI.test_decode_layout_golden]),
    ("verify rows scored to their request's largest bound", O, "score_paged", rows_scored_to_the_request_bound,
     [TI.test_rows_of_a_request_stop_at_their_own_bounds]),
    ("every request reads the first request's pages", O, "score_paged", every_request_reads_request_zero,
     [TI.test_score_matches_dequantised_float_reference]),
    ("positions paged column-major", O, "decode_keys", positions_paged_column_major,
     [TI.test_score_matches_dequantised_float_reference]),
    ("row bounds shifted by one row", O, "decode_layout", layout_request_off_by_one,
     [TI.test_decode_layout_golden, TI.test_decode_layout_bruteforce_random]),
    ("top-k ascending", O, "topk", topk_ascending, [TI.test_topk_short_rows_return_all_positions]),
    ("top-k ties broken toward the later position", O, "topk", topk_ties_last_position_first,
     [TI.test_topk_bruteforce]),
    ("FP8 scale exponent one too high", O, "fp8_scale_exponent", fp8_exponent_one_high,
     [TC.test_scale_invariants, TC.test_scales_golden]),
    ("MXFP4 exponent rounded down", O, "mx_scale_exponent", mx_exponent_floor,
     [TC.test_scale_invariants, TC.test_scales_golden]),
    ("LayerNorm without beta", O, "layer_norm_bf16", layer_norm_without_beta, [TI.test_layer_norm_special_cases]),
    ("LayerNorm lanes summed left to right", O, "_half_warp_sum", lanes_left_to_right,
     [TI.test_layer_norm_lane_order_is_the_stated_one]),
    ("LayerNorm eps outside the square root", O, "layer_norm_bf16", _layer_norm_variant(eps_outside=True),
     [TI.test_layer_norm_eps_inside_the_root]),
    ("LayerNorm output with a fused multiply-add", O, "layer_norm_bf16", _layer_norm_variant(fused=True),
     [TI.test_layer_norm_output_has_no_fused_multiply_add]),
    ("E4M3 rounding toward zero", C, "e4m3_encode", e4m3_truncating, [lambda: TC.test_e4m3_exhaustive_bf16(1.0)]),
    ("FP8 weight fold without the 1/64", O, "WEIGHT_SCALE", 1.0, [TC.test_scales_golden]),
    ("MXFP4 weight without the 1/64", O, "FP4_WEIGHT", 1.0, [TI.test_mxfp4_weights_share_the_fp8_fold]),
    ("MXFP4 query nibbles swapped", O, "quantize_query", query_nibbles_swapped,
     [TR.test_rowgroup_query_rows_carry_the_same_codes_and_scales]),
    ("FP8 query heads in reverse order", O, "quantize_query", fp8_query_heads_reversed, [TC.test_scales_golden]),
    ("MXFP4 query scale bytes block-major", O, "quantize_query", mxfp4_query_scales_block_major,
     [TR.test_decoded_keys_and_scores_agree]),
    ("FP8 key scale big-endian", O, "quantize_key", fp8_key_scale_big_endian,
     [lambda: TI.test_insert_layout_golden("fp8")]),
    ("MXFP4 key scale blocks reversed", O, "quantize_key", mxfp4_key_scale_blocks_reversed,
     [TR.test_page_views_show_the_token_major_codes]),
    ("FP8 key codes without the scale divided out", O, "quantize_key", fp8_key_codes_unscaled,
     [lambda: TI.test_insert_layout_golden("fp8")]),
    ("row-group query scales head-major", O, "quantize_queries", queries_head_major_scales,
     [TR.test_quantize_queries_closed_form]),
    ("row-group key scales read token-major", O, "decode_keys", keys_rowgroup_scales_token_major,
     [TR.test_decoded_keys_and_scores_agree]),
    ("QueryNorm eps dropped", QN, "_rsqrt", rsqrt_without_eps,
     [lambda: TQ.test_zero_row_with_eps_is_zero(QN.query_norm_cta)]),
    ("QueryNorm mean over 1535 columns", QN, "_rsqrt", rsqrt_mean_over_one_column_less,
     [TQ.test_orders_agree_when_sums_are_exact]),
    ("QueryNorm warp sum left to right", QN, "_warp_sum", warp_sum_left_to_right,
     [TQ.test_warp_sum_is_the_stated_butterfly]),
    ("QueryNorm weight applied before rr", QN, "_scale", scale_weight_first,
     [lambda: TQ.test_output_products_in_the_printed_order(QN.query_norm_cta),
      lambda: TQ.test_output_products_in_the_printed_order(QN.query_norm_tiled)]),
    ("DCP owner ignoring the interleave", D, "owner", owner_ignoring_interleave,
     [TD.test_rank_local_ends_count_the_owned_keys]),
    ("DCP partial round one key short", D, "rank_local_ends", rank_local_ends_partial_short,
     [TD.test_rank_local_ends_count_the_owned_keys, TD.test_hand_case]),
    ("DCP local to global without the rank's offset", D, "local_to_global", local_to_global_without_rank,
     [TD.test_hand_case]),
    ("DCP merge ties toward the later position", D, "topk_merge", merge_ties_toward_later_position,
     [TD.test_merge_of_local_topks_is_the_global_topk]),
]


@pytest.mark.filterwarnings("ignore::RuntimeWarning")   # a planted mistake may divide by zero
@pytest.mark.parametrize("name,module,attr,mutant,pins", CASES, ids=[c[0] for c in CASES])
def test_pins_catch_the_planted_mistake(monkeypatch, name, module, attr, mutant, pins):
    for pin in pins:   # every pin passes on the oracle as it stands
        pin()
    monkeypatch.setattr(module, attr, mutant)
    caught = []
    for pin in pins:
        try:
            pin()
        except AssertionError:   # a pin's own check failed (a mutant that crashed would not count)
            caught.append(getattr(pin, "__name__", "pin"))
    assert caught, f"no pin caught: {name}"



def test_the_layer_norm_variant_without_changes_is_the_oracle():
    """The LayerNorm mutants differ from the oracle only in what they plant."""
    rng = np.random.default_rng(4)
    x = C.bf16_round((rng.standard_normal((64, 128)) * 3).astype(np.float32))
    gamma = C.bf16_round((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    beta = C.bf16_round((0.1 * rng.standard_normal(128)).astype(np.float32))
    assert np.array_equal(_layer_norm_variant()(x, gamma, beta, 1e-6), O.layer_norm_bf16(x, gamma, beta, 1e-6))
