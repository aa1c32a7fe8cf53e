"""The oracle's pins catch plausible mistakes: each case below plants one
mistake in the oracle (on the CPU, for the duration of the case) and checks
that at least one of the pins named with it fails.  A dropped term, a wrong
sign, order or index, or a transposed operand in any step must show up."""

import numpy as np
import pytest

from oracle import codecs as C
from oracle import indexer as O

import test_oracle_codecs as TC
import test_oracle_indexer as TI

_orig = {name: getattr(O, name) for name in (
    "score_row", "decode_query", "decode_keys", "decode_layout", "topk", "fp8_scale_exponent",
    "mx_scale_exponent", "layer_norm_bf16", "_half_warp_sum")}


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
    ("E4M3 rounding toward zero", C, "e4m3_encode", e4m3_truncating, [lambda: TC.test_e4m3_exhaustive_bf16(1.0)]),
]


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

