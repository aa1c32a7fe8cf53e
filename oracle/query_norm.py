"""Plain CPU oracle of ``QueryNorm``: the q_a RMSNorm of the packed projection.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA path.

Page *cutedsl.dsa.overlap*, class ``QueryNorm``: each of ``batch`` rows holds
1536 BF16 columns (the q_a part of the packed projection); the row is scaled
by the reciprocal root of its mean square and by the BF16 weights, and
stored as BF16 q_c.  The page prints two kernels that must give identical
results to the model's query kernel, and so fixes their FP32 operation order:

* ``kernel`` (one row per CTA of 256 threads): thread t < 192 holds columns
  8t..8t+7 and sums their squares with sequential fused multiply-adds from
  0; each warp sums its lanes; the 8 warp sums (warps 6 and 7 hold nothing)
  are added in warp order.
* ``tiled`` (one row per warp): lane l holds the 48 columns 256i + 8l + j
  (i < 6, j < 8) as values e = 8i + j; squares go to four FMA chains, value e
  to chain e mod 4 in increasing e (two packed pairs); the lane total is
  (c0 + c1) + (c2 + c3), then the warp sum.

Readings where the page is silent:
- ``warp_sum`` is an xor butterfly over 32 lanes with distances 16, 8, 4,
2, 1 (addition is commutative, so every lane ends with the same value).
- ``query_norm_rsqrt(total, eps)`` = 1 / sqrt(total / 1536 + eps), each
operation correctly rounded in FP32.
- the output is BF16_rne((x * rr) * w) with two FP32 products, as both
kernels print them (left to right); the packed products round each lane.
- ``tiled_from`` is not printed: the caller picks the variant.

Every FP32 operation below is rounded on its own.  A fused multiply-add
``fma(x, x, c)`` is evaluated as FP64 ``x * x + c`` rounded to FP32: x is a
BF16 value, so x * x is exact in FP64 and needs at most 16 significant bits;
the FP64 sum is then exact unless the two terms are more than 29 binary
orders apart, and in that case the smaller one lies far below half an FP32
unit of the larger, so no FP32 tie can arise.  The result is therefore the
single rounding of the exact value (checked against exact rational
arithmetic in the tests).
"""

from __future__ import annotations

import numpy as np

from .codecs import bf16_round

COLS = 1536


def _fma32(a, b, c):
    """FP32 fused multiply-add of BF16-valued a, b and FP32 c (single rounding)."""
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(np.float32)


def _warp_sum(lanes: np.ndarray) -> np.ndarray:
    """Reading: xor butterfly over the last axis (32 lanes), distances 16..1."""
    s = lanes.astype(np.float32)
    lane = np.arange(32)
    for d in (16, 8, 4, 2, 1):
        s = (s + s[..., lane ^ d]).astype(np.float32)
    return s[..., 0]


def _rsqrt(total: np.ndarray, eps: float) -> np.ndarray:
    """Reading: 1 / sqrt(total / 1536 + eps), each operation rounded to FP32."""
    mean = (total.astype(np.float32) / np.float32(COLS)).astype(np.float32)
    return (np.float32(1.0) / np.sqrt((mean + np.float32(eps)).astype(np.float32))).astype(np.float32)


def _scale(x: np.ndarray, rr: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Reading: BF16((x * rr) * w), two FP32 products."""
    y = (x * rr[:, None]).astype(np.float32)
    return bf16_round((y * w[None, :]).astype(np.float32))


def query_norm_cta(x, w, eps: float) -> np.ndarray:
    """``QueryNorm.kernel``: x FP32 [B, 1536] (BF16 values), w [1536] (BF16
    values) -> q_c as FP32 holding BF16 values."""
    x = np.asarray(x, np.float32)
    w = np.asarray(w, np.float32)
    B = x.shape[0]
    T = x.reshape(B, 192, 8)                       # thread t: columns 8t .. 8t + 7
    thread = np.zeros((B, 256), np.float32)
    acc = np.zeros((B, 192), np.float32)
    for i in range(8):
        acc = _fma32(T[:, :, i], T[:, :, i], acc)
    thread[:, :192] = acc
    warp = _warp_sum(thread.reshape(B, 8, 32))     # [B, 8]
    total = np.zeros(B, np.float32)
    for k in range(8):
        total = (total + warp[:, k]).astype(np.float32)
    return _scale(x, _rsqrt(total, eps), w)


def query_norm_tiled(x, w, eps: float) -> np.ndarray:
    """``QueryNorm.tiled``: as ``query_norm_cta`` with the tiled kernel's order."""
    x = np.asarray(x, np.float32)
    w = np.asarray(w, np.float32)
    B = x.shape[0]
    # lane l, value e = 8i + j  <->  column 256i + 8l + j
    V = x.reshape(B, 6, 32, 8).transpose(0, 2, 1, 3).reshape(B, 32, 48)
    chains = np.zeros((B, 32, 4), np.float32)
    for e in range(48):
        chains[:, :, e % 4] = _fma32(V[:, :, e], V[:, :, e], chains[:, :, e % 4])
    lane_total = ((chains[:, :, 0] + chains[:, :, 1]).astype(np.float32) +
                  (chains[:, :, 2] + chains[:, :, 3]).astype(np.float32)).astype(np.float32)
    return _scale(x, _rsqrt(_warp_sum(lane_total), eps), w)


def query_norm(x, w, eps: float, variant: str) -> np.ndarray:
    if variant == "cta":
        return query_norm_cta(x, w, eps)
    if variant == "tiled":
        return query_norm_tiled(x, w, eps)
    raise ValueError(f"unknown variant {variant!r}")
