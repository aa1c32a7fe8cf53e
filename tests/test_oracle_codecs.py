"""Pins of the oracle's number formats against brute force, a library cast and
hand-worked values (CPU only)."""

import json
import os

import numpy as np
import pytest

from oracle import codecs as C
from oracle import indexer as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _all_bf16_finite():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)]


def _bruteforce(x, values, maximum):
    """Nearest code by exhaustive search over a codebook (same sign as x,
    ties to the even code), with saturation; a different method from the
    encoder's grid rounding."""
    codes = np.arange(values.shape[0])
    finite = np.isfinite(values)
    out = np.empty(x.shape[0], dtype=np.int64)
    for start in range(0, x.shape[0], 4096):
        xs = x[start:start + 4096].astype(np.float64)
        neg = np.signbit(xs)
        a = np.minimum(np.abs(xs), maximum)
        sign_ok = np.signbit(values)[None, :] == neg[:, None]
        ok = sign_ok & finite[None, :]
        dist = np.where(ok, np.abs(np.abs(values)[None, :] - a[:, None]), np.inf)
        best = dist.min(axis=1, keepdims=True)
        tie = (dist == best)
        # prefer the even code among the nearest
        pref = np.where(tie, (codes[None, :] & 1) * 2 + (codes[None, :] >= 0), 99)
        out[start:start + 4096] = np.argmin(pref * 1000 + (~tie) * 10**6 + codes[None, :] * 0, axis=1)
    return out


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -7, 2.0 ** 5, 2.0 ** -20])
def test_e4m3_exhaustive_bf16(scale):
    x = _all_bf16_finite().astype(np.float64) * scale
    got = C.e4m3_encode(x).astype(np.int64)
    want = _bruteforce(x, C.E4M3_TABLE, 448.0)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -3, 2.0 ** 2])
def test_e2m1_exhaustive_bf16(scale):
    x = _all_bf16_finite().astype(np.float64) * scale
    got = C.e2m1_encode(x).astype(np.int64)
    want = _bruteforce(x, C.E2M1_TABLE, 6.0)
    assert np.array_equal(got, want)


def test_e4m3_matches_torch_cast():
    torch = pytest.importorskip("torch")
    x = _all_bf16_finite()
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(C.e4m3_encode(x), ref)


def test_e4m3_decode_roundtrip_and_codebook():
    vals = C.E4M3_TABLE
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    finite = np.isfinite(vals)
    codes = np.arange(256)[finite]
    assert np.array_equal(C.e4m3_encode(vals[finite]), codes.astype(np.uint8))


def test_e2m1_codebook():
    assert list(C.E2M1_TABLE[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(C.E2M1_TABLE[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    assert np.array_equal(C.e2m1_encode(C.E2M1_TABLE), np.arange(16, dtype=np.uint8))


def test_pack_e2m1_low_nibble_first():
    codes = np.array([1, 2, 3, 4, 15, 0], dtype=np.uint8)
    packed = C.pack_e2m1(codes)
    assert list(packed) == [0x21, 0x43, 0x0F]
    assert np.array_equal(C.unpack_e2m1(packed), codes)


def test_bf16_round_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32),
        (rng.standard_normal(10000) * 1e-39).astype(np.float32),   # FP32 subnormals
        (rng.standard_normal(10000) * 1e30).astype(np.float32),
    ])
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).float().numpy()
    assert np.array_equal(C.bf16_round(x), ref)


def test_scale_invariants():
    rng = np.random.default_rng(3)
    amax = np.exp(rng.uniform(np.log(1e-10), np.log(1e30), 200000)).astype(np.float32)
    amax = np.concatenate([amax, np.float32([1e-10, 448.0, 3.5, 2.0 ** -20])])
    e = O.fp8_scale_exponent(amax)
    ratio = amax.astype(np.float64) / np.ldexp(1.0, e)
    assert np.all(ratio <= 448.0) and np.all(ratio > 224.0)
    a = np.concatenate([amax, np.float32([0.0, 6.0, 2.0 ** -126, 1e-38])])
    em = O.mx_scale_exponent(a)
    byte = em + 127
    assert np.all((byte >= 1) & (byte <= 254))
    above = a.astype(np.float64) > 6.0 * 2.0 ** -126
    r = a[above].astype(np.float64) / np.ldexp(1.0, em[above])
    assert np.all(r <= 6.0) and np.all(r > 3.0)
    assert np.all(em[~above] == -126)


def test_scales_golden():
    g = json.load(open(os.path.join(GOLDEN, "scales.json")))
    for case in g["fp8"]:
        amax = np.float32(case["amax"])
        e = int(O.fp8_scale_exponent(np.maximum(amax, O.FP8_AMAX_FLOOR)))
        assert e == case["exponent"], case
        v = np.float64(np.float32(case["value"])) * 2.0 ** -e
        assert int(C.e4m3_encode(v)) == case["code"], case
        word = (e + 127) * 0x01010101
        assert word == int(case["mx_word"], 16)
        q = np.zeros((1, 32, 128), np.float32)
        q[0, 0, 0] = amax if case["amax"] >= 1e-10 else np.float32(case["value"])
        q[0, 0, 1] = np.float32(case["value"])
        wv = np.zeros((1, 32), np.float32)
        wv[0, 0] = case["wv"]
        rows, w = O.quantize_query("fp8", q, wv)
        assert rows[0, 1] == case["code"] and w[0, 0] == np.float32(case["w"]), case
    for case in g["mxfp4"]:
        e = int(O.mx_scale_exponent(np.float32(case["amax"])))
        assert e == case["exponent"] and e + 127 == case["byte"], case
        v = np.float64(np.float32(case["value"])) * 2.0 ** -e
        assert int(C.e2m1_encode(v)) == case["code"], case
