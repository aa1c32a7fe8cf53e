"""Pins of the oracle's indexer steps (CPU only): LayerNorm against FP64 and
torch, the cache byte layout, decode_layout hand cases and brute force,
hand-computed scores, score invariants and brute-force top-k."""

import json
import os

import numpy as np
import pytest

from oracle import codecs as C
from oracle import indexer as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- LayerNorm

def _bf16_values(rng, shape, scale=1.0):
    return C.bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))


def test_layer_norm_close_to_fp64_and_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = _bf16_values(rng, (4000, 128), 3.0)
    gamma = C.bf16_round((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    beta = C.bf16_round((0.1 * rng.standard_normal(128)).astype(np.float32))
    got = O.layer_norm_bf16(x, gamma, beta, 1e-6)
    xd = x.astype(np.float64)
    mean = xd.mean(axis=1, keepdims=True)
    var = ((xd - mean) ** 2).mean(axis=1, keepdims=True)
    exact = (xd - mean) / np.sqrt(var + 1e-6) * gamma + beta
    # BF16 output within one BF16 ulp of the exact value (plus FP32 noise)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    assert np.all(np.abs(got - exact) <= ulp * 0.5 + 1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (128,), torch.from_numpy(gamma),
                                         torch.from_numpy(beta), 1e-6).to(torch.bfloat16).float().numpy()
    assert np.mean(got == ref) >= 0.999


def test_layer_norm_special_cases():
    rng = np.random.default_rng(1)
    beta = _bf16_values(rng, (128,), 0.3)
    gamma = _bf16_values(rng, (128,))
    const = np.full((3, 128), 1.5, np.float32)
    assert np.array_equal(O.layer_norm_bf16(const, gamma, beta, 1e-6), np.broadcast_to(beta, (3, 128)))
    alt = np.tile(np.float32([2.0, -2.0]), 64)[None, :]
    out = O.layer_norm_bf16(alt, np.ones(128, np.float32), np.zeros(128, np.float32), 1e-6)
    assert np.array_equal(out[0], np.tile(np.float32([1.0, -1.0]), 64))


def test_layer_norm_lane_order_is_the_stated_one():
    # Lane 0 holds 2^24, lane 8 holds -2^24, lane 1 holds 1.  The xor butterfly
    # adds lanes 0 and 8 first, so the sum is exactly 1 and mean = 2^-7; a
    # left-to-right sum would lose the 1 against 2^24 and give mean 0.
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = 2.0 ** 24
    x[0, 64] = -(2.0 ** 24)
    x[0, 8] = 1.0
    normed = O.layer_norm_bf16(x, np.ones(128, np.float32), np.zeros(128, np.float32), 1e-6)
    # var = (2 * 2^48) / 128 = 2^42 (the small squares are lost), rstd = 2^-21,
    # so a zero column gives (0 - 2^-7) * 2^-21 = -2^-28.
    assert normed[0, 16] == np.float32(-(2.0 ** -28))
    assert normed[0, 0] == np.float32(8.0) and normed[0, 64] == np.float32(-8.0)


def test_layer_norm_eps_inside_the_root():
    """A row of +-2^-10 has variance 2^-20, the size of eps = 1e-6: the closed
    form 2^-10 / sqrt(2^-20 + 1e-6) = 0.69867... rounds to the BF16 0.69921875
    (eps added outside the root would give 0.99898... and 1.0)."""
    d = 2.0 ** -10
    x = np.tile(np.float32([d, -d]), 64)[None, :]
    out = O.layer_norm_bf16(x, np.ones(128, np.float32), np.zeros(128, np.float32), 1e-6)[0]
    closed = d / np.sqrt(d * d + 1e-6)
    assert out[0] == C.bf16_round(np.float32(closed)) == np.float32(0.69921875)
    assert out[1] == -out[0]


def test_layer_norm_output_has_no_fused_multiply_add():
    """Row of +-1.234375 (mean 0, variance 1.523681640625 exactly): in FP32
    var + eps = 1.5236825942993164, rstd = 0.8101263642311096 and
    (x - mean) * rstd = 0.9999997019767761 on column 0.  With gamma -0.2109375
    and beta -0.80078125: the product rounds to -0.21093744039535522 and the
    sum to -1.01171875 exactly, a BF16 tie that rounds to the even -1.015625.
    A fused multiply-add would round the exact -1.01171863... once, to
    -1.0117186307907104, and give -1.0078125."""
    x = np.tile(np.float32([1.234375, -1.234375]), 64)[None, :]
    gamma, beta = np.ones(128, np.float32), np.zeros(128, np.float32)
    gamma[0], beta[0] = -0.2109375, -0.80078125
    assert O.layer_norm_bf16(x, gamma, beta, 1e-6)[0, 0] == np.float32(-1.015625)


# ---------------------------------------------------------------- cache layout

@pytest.mark.parametrize("fmt", ["fp8", "fp8_mx", "mxfp4"])
def test_insert_layout_golden(fmt):
    g = json.load(open(os.path.join(GOLDEN, "cache_layout.json")))
    stride = O.page_bytes(fmt) + 32          # a physical page stride larger than the section
    num_pages = 4
    cache = np.full(num_pages * stride, 0xAA, np.uint8)
    key = np.tile(np.float32([1.0, -1.0]), 64)[None, :]
    bad = O.insert_key(fmt, cache, stride, num_pages, key, np.ones(128, np.float32),
                       np.zeros(128, np.float32), 1e-6, np.array([g["slot"]]))
    assert bad == 0
    page, off = g["page"], g["offset"]
    base = page * stride
    written = np.zeros_like(cache, dtype=bool)
    if fmt == "mxfp4":
        codes = cache[base + off * 64: base + off * 64 + 64]
        assert np.all(codes == g["mxfp4"]["pair_byte"])
        sc = cache[base + 4096 + off * 4: base + 4096 + off * 4 + 4]
        assert np.all(sc == g["mxfp4"]["scale_byte"])
        written[base + off * 64: base + off * 64 + 64] = True
        written[base + 4096 + off * 4: base + 4096 + off * 4 + 4] = True
    else:
        codes = cache[base + off * 128: base + off * 128 + 128]
        assert np.all(codes[0::2] == g["fp8"]["code_even"]) and np.all(codes[1::2] == g["fp8"]["code_odd"])
        sc = cache[base + 8192 + off * 4: base + 8192 + off * 4 + 4]
        want = g["fp8"]["scale_f32_bytes"] if fmt == "fp8" else [g["fp8"]["mx_byte"]] * 4
        assert list(sc) == want
        written[base + off * 128: base + off * 128 + 128] = True
        written[base + 8192 + off * 4: base + 8192 + off * 4 + 4] = True
    assert np.all(cache[~written] == 0xAA)


def test_insert_padding_and_out_of_range_slots():
    cache = np.zeros(2 * O.FP8_PAGE_BYTES, np.uint8)
    x = np.random.default_rng(0).standard_normal((3, 128)).astype(np.float32)
    bad = O.insert_key("fp8", cache, O.FP8_PAGE_BYTES, 2, x, np.ones(128, np.float32),
                       np.zeros(128, np.float32), 1e-6, np.array([-1, 128, 1000]))
    assert bad == 2 and not cache.any()


@pytest.mark.parametrize("fmt", ["fp8", "fp8_mx", "mxfp4", "mxfp4_rg"])
def test_insert_repeated_slot_keeps_the_last_key(fmt):
    """Keys are written in order: a slot named twice holds the later key's
    bytes, as if that key alone had been inserted there."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((5, 128)).astype(np.float32)
    g, b = np.ones(128, np.float32), np.zeros(128, np.float32)
    stride = O.page_bytes(fmt)
    both = np.zeros(2 * stride, np.uint8)
    O.insert_key(fmt, both, stride, 2, x, g, b, 1e-6, np.array([70, 3, 70, 9, 3], np.int64))
    alone = np.zeros(2 * stride, np.uint8)
    O.insert_key(fmt, alone, stride, 2, x[2:], g, b, 1e-6, np.array([70, 9, 3], np.int64))
    assert np.array_equal(both, alone)


def test_key_scale_power_of_two_equivariance():
    rng = np.random.default_rng(5)
    normed = _bf16_values(rng, (64, 128))
    for fmt in ("fp8", "fp8_mx", "mxfp4"):
        c0, s0 = O.quantize_key(fmt, normed)
        for j in (-3, 4):
            c1, s1 = O.quantize_key(fmt, (normed * np.float32(2.0 ** j)).astype(np.float32))
            assert np.array_equal(c0, c1)
            if fmt == "fp8":
                assert np.array_equal(s1.copy().view("<f4"), s0.copy().view("<f4") * np.float32(2.0 ** j))
            else:
                assert np.array_equal(s1.astype(int), s0.astype(int) + j)


# ---------------------------------------------------------------- decode_layout

def _layout_bruteforce(seq, qlen, num_rows):
    starts = [0]
    for n in qlen:
        starts.append(starts[-1] + int(n))
    ends = []
    for r in range(num_rows):
        end = 0
        for q in range(len(qlen)):
            if starts[q] <= r < starts[q + 1]:
                end = max(0, int(seq[q]) - int(qlen[q]) + (r - starts[q]) + 1)
        ends.append(end)
    return starts, ends


def test_decode_layout_golden():
    g = json.load(open(os.path.join(GOLDEN, "decode_layout.json")))
    for case in g["cases"]:
        starts, ends = O.decode_layout(np.array(case["seq_lens"], np.int32),
                                       np.array(case["query_lens"], np.int32), case["num_rows"])
        assert list(starts) == case["starts"] and list(ends) == case["row_ends"], case


def test_decode_layout_bruteforce_random():
    rng = np.random.default_rng(9)
    for _ in range(300):
        R = int(rng.integers(0, 8))
        qlen = rng.integers(0, 5, R).astype(np.int32)
        seq = rng.integers(0, 40, R + int(rng.integers(0, 3))).astype(np.int32)
        num_rows = int(qlen.sum()) + int(rng.integers(0, 4))
        starts, ends = O.decode_layout(seq, qlen, num_rows)
        bs, be = _layout_bruteforce(seq, qlen, num_rows)
        assert list(starts) == bs and list(ends) == be


def test_decode_layout_errors():
    with pytest.raises(ValueError):
        O.decode_layout(np.array([1]), np.array([1]), -1)
    with pytest.raises(ValueError):
        O.decode_layout(np.array([1]), np.array([1, 1]), 2)
    with pytest.raises(ValueError):
        O.decode_layout(np.array([[1]]), np.array([1]), 1)


# ---------------------------------------------------------------- scores

def _fp8_cache_one_page(codes_rows, scale_words, mx=False):
    """A one-page FP8 cache with the given per-token code rows and scales."""
    cache = np.zeros(O.FP8_PAGE_BYTES, np.uint8)
    for t, (codes, sc) in enumerate(zip(codes_rows, scale_words)):
        cache[t * 128:(t + 1) * 128] = codes
        cache[8192 + t * 4: 8192 + t * 4 + 4] = sc
    return cache


def test_score_hand_cases_fp8():
    q_row = np.zeros(4096, np.uint8)
    q_row[:128] = 0x38                                          # head 0: 128 x 1.0
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 0.5
    two = list(np.float32(2.0).tobytes())
    cache = _fp8_cache_one_page([np.full(128, 0x38), np.full(128, 0xB8)], [two, two])
    s = O.score_paged("fp8", q_row[None], w, cache, O.FP8_PAGE_BYTES, np.array([[0]]),
                      np.array([0, 1]), np.array([2]))
    assert s[0, 0] == 128.0          # 0.5 * ReLU(128 * 1 * 1 * 2)
    assert s[0, 1] == 0.0            # ReLU of a negative dot
    assert np.all(np.isneginf(s[0, 2:]))


def test_score_hand_case_fp8_mx_blocks():
    q_row = np.zeros(4096, np.uint8)
    q_row[:128] = 0x38
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 1.0
    cache = _fp8_cache_one_page([np.full(128, 0x38)], [[127, 128, 129, 130]])
    s = O.score_paged("fp8_mx", q_row[None], w, cache, O.FP8_PAGE_BYTES, np.array([[0]]),
                      np.array([0, 1]), np.array([1]))
    assert s[0, 0] == 32.0 * (1 + 2 + 4 + 8)


def test_score_hand_case_mxfp4():
    q_row = np.zeros(4096, np.uint8)
    q_row[:64] = 0x22                                           # head 0: 128 x 1.0 (code 2)
    q_row[2048:2052] = 127
    q_row[2052:2048 + 128] = 127
    w = np.zeros((1, 32), np.float32)
    w[0, 1] = -1.0
    w[0, 0] = 0.25
    cache = np.zeros(O.FP4_PAGE_BYTES, np.uint8)
    cache[:64] = 0x22
    cache[4096:4100] = [126, 127, 128, 129]
    s = O.score_paged("mxfp4", q_row[None], w, cache, O.FP4_PAGE_BYTES, np.array([[0]]),
                      np.array([0, 1]), np.array([1]))
    assert s[0, 0] == 0.25 * 32.0 * (0.5 + 1 + 2 + 4)


def _step(fmt, seed=0, R=3, seq=(70, 200), qlen=(1, 3)):
    from synth import bf16_bits_to_f32, make_workload
    wl = make_workload("tiny_fp8", fmt=fmt, R=R, seq=seq, qlen=qlen, seed=seed, pad_rows=1, topk=16)
    q, wv = bf16_bits_to_f32(wl.q_bits), bf16_bits_to_f32(wl.wv_bits)
    qr, w = O.quantize_query(fmt, q, wv)
    stride = O.page_bytes(fmt)
    cache = np.zeros(wl.num_pages * stride, np.uint8)
    kb, sl = wl.prefill_all()
    O.insert_key(fmt, cache, stride, wl.num_pages, bf16_bits_to_f32(kb), wl.gamma, wl.beta, wl.eps, sl)
    O.insert_key(fmt, cache, stride, wl.num_pages, bf16_bits_to_f32(wl.step_key_bits), wl.gamma,
                 wl.beta, wl.eps, wl.step_slots)
    starts, ends = O.decode_layout(wl.seq_lens, wl.query_lens, wl.num_rows)
    s = O.score_paged(fmt, qr, w, cache, stride, wl.block_table, starts, ends)
    return wl, qr, w, cache, starts, ends, s


def test_fp8_scale_forms_give_identical_logits():
    a = _step("fp8", seed=4)
    b = _step("fp8_mx", seed=4)
    assert np.array_equal(a[6], b[6])


def test_nonnegative_weights_give_nonnegative_scores():
    wl, qr, w, cache, starts, ends, s = _step("fp8", seed=2)
    neg = qr.copy()
    neg[:, :4096] ^= 0x80                                        # flip every E4M3 sign
    s_pos = O.score_paged("fp8", qr, np.abs(w), cache, O.FP8_PAGE_BYTES, wl.block_table, starts, ends)
    s_neg = O.score_paged("fp8", neg, np.abs(w), cache, O.FP8_PAGE_BYTES, wl.block_table, starts, ends)
    # sum_h |w_h| (ReLU(d) + ReLU(-d)) = sum_h |w_h| |d|; both parts are non-negative
    fin = np.isfinite(s_pos)
    assert np.all(s_pos[fin] >= 0) and np.all(s_neg[fin] >= 0)
    assert np.any(s_pos[fin] > 0)


def test_rows_of_a_request_stop_at_their_own_bounds():
    """Verify rows of one request share its keys but each is scored only below
    its own causal bound: row i of a request of length L with Q rows ends at
    L - Q + i + 1; the logits there and past it are -inf."""
    wl, qr, w, cache, starts, ends, s = _step("fp8", seed=8, R=2, seq=(100, 130), qlen=(3, 3))
    for q in range(wl.R):
        L, Q = int(wl.seq_lens[q]), int(wl.query_lens[q])
        for i, r in enumerate(range(int(starts[q]), int(starts[q + 1]))):
            assert ends[r] == L - Q + i + 1
            assert np.all(np.isfinite(s[r, :ends[r]])) and np.all(np.isneginf(s[r, ends[r]:]))


def test_score_matches_dequantised_float_reference():
    """The oracle's logits against an independent dequantisation: each cache
    byte decoded through the brute-force codebook tables and the layout
    offsets of the golden file, summed with Python's exact fractions."""
    from fractions import Fraction
    wl, qr, w, cache, starts, ends, s = _step("mxfp4", seed=6, R=2, seq=(65, 70), qlen=(1, 1))
    r = 1
    qv = {}
    for h in range(32):
        for c in range(128):
            byte = int(qr[r, h * 64 + c // 2])
            code = byte & 0xF if c % 2 == 0 else byte >> 4
            ex = int(qr[r, 2048 + h * 4 + c // 32]) - 127
            qv[h, c] = Fraction(C.E2M1_TABLE[code]) * Fraction(2) ** ex
    for t in (0, 63, 64, int(ends[r]) - 1):
        page = int(wl.block_table[1, t // 64])
        base = page * O.FP4_PAGE_BYTES
        off = t % 64
        total = Fraction(0)
        for h in range(32):
            dot = Fraction(0)
            for c in range(128):
                byte = int(cache[base + off * 64 + c // 2])
                code = byte & 0xF if c % 2 == 0 else byte >> 4
                ex = int(cache[base + 4096 + off * 4 + c // 32]) - 127
                dot += qv[h, c] * Fraction(C.E2M1_TABLE[code]) * Fraction(2) ** ex
            total += Fraction(float(w[r, h])) * max(dot, Fraction(0))
        assert abs(float(total) - s[r, t]) <= 1e-12 * max(1.0, abs(float(total)))


def test_mxfp4_weights_share_the_fp8_fold():
    """The MXFP4 head weight carries the same 1/64 as the FP8 fold (pinned by
    the scale fixtures) but no query scale: for one query, w_fp8 = w_mxfp4 *
    2^e with e each head's FP8 exponent, exactly (powers of two, no underflow
    at these sizes)."""
    rng = np.random.default_rng(12)
    q = _bf16_values(rng, (6, 32, 128), 2.0)
    wv = _bf16_values(rng, (6, 32))
    _, w8 = O.quantize_query("fp8", q, wv)
    _, w4 = O.quantize_query("mxfp4", q, wv)
    e = O.fp8_scale_exponent(np.maximum(np.abs(q).max(axis=2), O.FP8_AMAX_FLOOR))
    assert np.array_equal(np.asarray(w8, np.float64), np.asarray(w4, np.float64) * np.ldexp(1.0, e))
    assert np.any(w4 != wv)


# ---------------------------------------------------------------- top-k

def test_topk_bruteforce():
    rng = np.random.default_rng(2)
    for _ in range(50):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 50))
        scores = np.round(rng.standard_normal((1, 45)), 1)   # many ties
        scores[0, n:] = -np.inf
        got = O.topk(scores, np.array([n]), k)[0]
        s = list(scores[0, :n])
        want = []
        avail = list(range(n))
        for _ in range(min(k, n)):
            best = max(avail, key=lambda t: (s[t], -t))
            want.append(best)
            avail.remove(best)
        want += [-1] * (k - len(want))
        assert list(got) == want


def test_topk_short_rows_return_all_positions():
    scores = np.array([[3.0, 1.0, 2.0, -np.inf]])
    assert list(O.topk(scores, np.array([3]), 5)[0]) == [0, 2, 1, -1, -1]
    assert list(O.topk(scores, np.array([0]), 2)[0]) == [-1, -1]
