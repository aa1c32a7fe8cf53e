"""Pins of the QueryNorm oracle (page *cutedsl.dsa.overlap*, ``QueryNorm``)
against facts other than itself: exact rational arithmetic for its FMA, closed
forms, rows whose sums are exact in any order, and an FP64 / library RMSNorm
within the BF16 rounding."""

from fractions import Fraction

import numpy as np
import pytest

from oracle.codecs import bf16_round
from oracle.query_norm import COLS, _fma32, query_norm_cta, query_norm_tiled

VARIANTS = [query_norm_cta, query_norm_tiled]


def _bf16(rng, shape, scale=1.0):
    return bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))


def _round_f32(q: Fraction) -> np.float32:
    """Correct rounding of an exact rational to FP32 (ties to even), by search
    between the two neighbouring FP32 values."""
    f = np.float32(float(q))                 # within one ulp of the answer
    cands = {f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))}
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - q),
                                     int(np.array(c, np.float32).view(np.uint32)) & 1))
    return np.float32(best)


def test_fma_matches_exact_rounding():
    rng = np.random.default_rng(0)
    a = np.concatenate([_bf16(rng, 4000), _bf16(rng, 500, 1e10), _bf16(rng, 500, 1e-10)])
    c = np.concatenate([(rng.standard_normal(4000) * 1e3).astype(np.float32),
                        (rng.standard_normal(500) * 1e-8).astype(np.float32),
                        (rng.standard_normal(500) * 1e12).astype(np.float32)])
    c = np.abs(c)
    got = _fma32(a, a, c)
    for x, y, g in zip(a, c, got):
        want = _round_f32(Fraction(float(x)) * Fraction(float(x)) + Fraction(float(y)))
        assert g == want, (x, y, g, want)


@pytest.mark.parametrize("norm", VARIANTS)
def test_constant_power_of_two_rows_give_the_weights(norm):
    """x = +-2^k everywhere, eps = 0: mean square 4^k, rr = 2^-k exactly, so
    q_c = BF16(+-w) exactly."""
    rng = np.random.default_rng(1)
    w = _bf16(rng, COLS)
    x = np.stack([np.full(COLS, s * 2.0 ** k, np.float32) for s, k in ((1, 0), (-1, 3), (1, -20), (-1, 50))])
    got = norm(x, w, 0.0)
    want = bf16_round(np.sign(x) * w[None, :])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("norm", VARIANTS)
def test_zero_row_with_eps_is_zero(norm):
    w = _bf16(np.random.default_rng(2), COLS)
    got = norm(np.zeros((2, COLS), np.float32), w, 1e-6)
    assert not np.any(got)


def test_orders_agree_when_sums_are_exact():
    """Small integers: every partial sum of squares is an exact FP32 integer,
    so the two kernels' orders give the same bits, and both equal the formula
    evaluated with an exact total."""
    rng = np.random.default_rng(3)
    x = rng.integers(-3, 4, (6, COLS)).astype(np.float32)
    w = _bf16(rng, COLS)
    a, b = query_norm_cta(x, w, 1e-5), query_norm_tiled(x, w, 1e-5)
    assert np.array_equal(a, b)
    total = (x.astype(np.float64) ** 2).sum(axis=1).astype(np.float32)
    rr = (np.float32(1) / np.sqrt((total / np.float32(COLS) + np.float32(1e-5)).astype(np.float32))).astype(np.float32)
    want = bf16_round(((x * rr[:, None]).astype(np.float32) * w).astype(np.float32))
    assert np.array_equal(a, want)


def test_warp_sum_is_the_stated_butterfly():
    """Lane 0 holds 2^26 (FP32 spacing 8 there), lanes 1..31 hold 4.  The xor
    butterfly (16, 8, 4, 2, 1) loses lane 16's 4 in its first step (2^26 + 4
    is a tie, rounded to even) and then adds 8, 16, 32 and 64 exactly: 2^26 +
    120.  A left-to-right sum would lose every 4 and give 2^26; the exact sum
    is 2^26 + 124."""
    from oracle.query_norm import _warp_sum
    lanes = np.full((1, 32), 4.0, np.float32)
    lanes[0, 0] = 2.0 ** 26
    assert _warp_sum(lanes)[0] == np.float32(2.0 ** 26 + 120)


@pytest.mark.parametrize("norm", VARIANTS)
def test_output_products_in_the_printed_order(norm):
    """Both kernels print q_c = BF16((x * rr) * w).  Row [1.4140625, 1.40625,
    0, ...] with eps 0: the sum of squares 3.97711181640625 is exact in any
    order; in FP32 the mean is 0.0025892655830830336 and rr 19.652223587036133.
    Column 0 with w = 0.81640625: x * rr = 27.789472579956055, times w =
    22.6875 exactly, a BF16 tie that rounds to the even 22.75.  The other
    order, x * w = 1.154449462890625 (exact) times rr = 22.687498..., would
    give 22.625."""
    x = np.zeros((1, COLS), np.float32)
    x[0, 0], x[0, 1] = 1.4140625, 1.40625
    w = np.ones(COLS, np.float32)
    w[0] = 0.81640625
    assert norm(x, w, 0.0)[0, 0] == np.float32(22.75)


@pytest.mark.parametrize("norm", VARIANTS)
def test_close_to_fp64_rmsnorm(norm):
    """Within one BF16 unit of the FP64 RMSNorm rounded to BF16; equal to it
    for nearly every element."""
    rng = np.random.default_rng(4)
    x = np.concatenate([_bf16(rng, (20, COLS)), _bf16(rng, (4, COLS), 1e3), _bf16(rng, (4, COLS), 1e-3)])
    w = _bf16(rng, COLS)
    eps = 1e-6
    xd = x.astype(np.float64)
    ref = xd / np.sqrt((xd ** 2).mean(axis=1, keepdims=True) + eps) * w
    got = norm(x, w, eps).astype(np.float64)
    ulp = np.abs(bf16_round(ref.astype(np.float32)).astype(np.float64)) * 2.0 ** -7
    assert np.all(np.abs(got - ref) <= ulp + 1e-30)
    assert np.mean(got == bf16_round(ref.astype(np.float32))) > 0.99


def test_matches_torch_rms_norm_within_a_bf16_unit():
    torch = pytest.importorskip("torch")
    if not hasattr(torch.nn.functional, "rms_norm"):
        pytest.skip("torch without rms_norm")
    rng = np.random.default_rng(5)
    x = _bf16(rng, (16, COLS))
    w = _bf16(rng, COLS)
    t = torch.nn.functional.rms_norm(torch.from_numpy(x), (COLS,), torch.from_numpy(w), eps=1e-6).numpy()
    for norm in VARIANTS:
        got = norm(x, w, 1e-6)
        tb = bf16_round(t)
        assert np.all(np.abs(got - tb) <= np.abs(tb) * 2.0 ** -7 + 1e-30)


def test_scaling_the_row_by_a_power_of_two_changes_nothing():
    rng = np.random.default_rng(6)
    x = _bf16(rng, (5, COLS))
    w = _bf16(rng, COLS)
    for norm in VARIANTS:
        assert np.array_equal(norm(x, w, 0.0), norm(x * np.float32(8.0), w, 0.0))
