"""Number formats of the DSA indexer, written from their definitions.

TEST INFRASTRUCTURE ONLY: nothing on the product path imports this module.

Formats (page *cutedsl.dsa.index*, module docstring and ``e2m1x2``):

* E4M3 (FP8, the "FN" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
  largest finite value 448, subnormals down to 2**-9, codes 0x7F/0xFF are NaN.
* E2M1 (FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}, bit 3 is the sign.
* UE8M0: an unsigned byte ``e + 127`` standing for the power of two ``2**e``.
* BF16: the top 16 bits of an FP32.

Every encoder rounds to nearest with ties to even and saturates to the
largest finite value ("round to nearest even, satfinite").  The sign of the
input is kept, so negative inputs that round to zero give negative zero.
All arithmetic is exact: an input is scaled by a power of two onto the grid of
its binade, ``np.rint`` (ties to even) picks the grid point, and the result is
scaled back.  On every grid used here an even grid count is an even mantissa.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _round_to_grid(a: np.ndarray, mant_bits: int, min_exp: int) -> np.ndarray:
    """Round non-negative float64 values to the nearest point of a binary
    floating-point grid with ``mant_bits`` stored mantissa bits whose smallest
    normal binade is ``2**min_exp`` (subnormals share that binade's spacing);
    ties go to the even grid count.  No upper bound is applied."""
    _, E = np.frexp(a)                       # a = m * 2**E with 0.5 <= m < 1
    e = np.maximum(E - 1, min_exp)           # binade of a, floored at the subnormal range
    quantum = np.ldexp(1.0, e - mant_bits)   # spacing of the grid in that binade
    return np.rint(a / quantum) * quantum    # exact: division by a power of two


def bf16_round(x) -> np.ndarray:
    """Round float32 values to BF16 (8 significant bits, FP32 exponent range),
    returned as float32."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    v = _round_to_grid(np.abs(x), 7, -126)
    return np.copysign(v, x).astype(np.float32)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of finite values: RNE, saturating to +-448."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    v = np.minimum(_round_to_grid(np.abs(x), 3, -6), E4M3_MAX)
    _, Ev = np.frexp(v)
    ev = Ev - 1
    normal = (v > 0) & (ev >= -6)
    field = np.where(normal, ev + 7, 0)
    mant = np.where(normal, (v / np.ldexp(1.0, np.where(normal, ev, 0)) - 1.0) * 8.0,
                    v / 2.0 ** -9)
    code = (neg.astype(np.int64) << 7) | (field.astype(np.int64) << 3) | mant.astype(np.int64)
    return code.astype(np.uint8)


def _e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    field, mant = (code >> 3) & 0xF, code & 0x7
    if field == 0xF and mant == 0x7:
        return float("nan")
    if field == 0:
        return s * mant * 2.0 ** -9
    return s * (1.0 + mant / 8.0) * 2.0 ** (field - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e2m1_encode(x) -> np.ndarray:
    """E2M1 codes (uint8 values 0..15) of finite values: RNE, saturating to +-6."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    v = np.minimum(_round_to_grid(np.abs(x), 1, 0), E2M1_MAX)
    _, Ev = np.frexp(v)
    ev = Ev - 1
    normal = (v > 0) & (ev >= 0)
    field = np.where(normal, ev + 1, 0)
    mant = np.where(normal, (v / np.ldexp(1.0, np.where(normal, ev, 0)) - 1.0) * 2.0, v / 0.5)
    code = (neg.astype(np.int64) << 3) | (field.astype(np.int64) << 1) | mant.astype(np.int64)
    return code.astype(np.uint8)


def _e2m1_value(code: int) -> float:
    s = -1.0 if code & 0x8 else 1.0
    field, mant = (code >> 1) & 0x3, code & 0x1
    if field == 0:
        return s * mant * 0.5
    return s * (1.0 + mant / 2.0) * 2.0 ** (field - 1)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def pack_e2m1(codes) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis: element 2j in the low
    nibble of byte j, element 2j+1 in the high nibble (page *cutedsl.dsa.index*,
    ``e2m1x2``: "low in the low nibble")."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def pow2_exponent(amax, maximum: float) -> np.ndarray:
    """The smallest integer e with ``maximum * 2**e >= amax`` (amax > 0), exactly.

    This is ``ceil(log2(amax / maximum))`` in exact arithmetic: an estimate
    from ``log2`` is corrected by exact comparisons (``ldexp`` of 448 or 6 is
    exact in float64)."""
    a = np.asarray(amax, dtype=np.float64)
    e = np.ceil(np.log2(a / maximum)).astype(np.int64)
    e = e + (np.ldexp(maximum, e) < a)
    e = e - (np.ldexp(maximum, e - 1) >= a)
    return e
