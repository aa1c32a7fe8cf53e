"""Seeded workloads of the DSA lightning-indexer decode step.

Every array here is a raw input of the step: BF16 bit patterns of the indexer
query rows and of the wk key projections, the head-weight logits wv, the
LayerNorm affine parameters, the request geometry (sequence and query
lengths, padding rows), a paged block table drawn as a random permutation of
the page pool, and the cache slots the keys go to.  Nothing is quantised,
normalised or scored here.

The five named workloads follow the decode-step shapes of the indexer pages
(32 heads x 128 columns, 64-token cache pages, FP8 or MXFP4 caches):

* ``tiny_fp8``      2 requests x 1 row, 256 keys each, FP8 keys with FP32
                    scales, top-64.
* ``fp8_decode``    64 requests x 1 row, 4096..8192 keys, FP8/FP32 scales,
                    top-2048.
* ``mxfp4_decode``  64 requests x 1 row, 16384..32768 keys, MXFP4 cache,
                    1 % of query elements scaled by 20, top-2048.
* ``spec_verify``   128 requests x 1..4 verify rows, 4096..65536 keys, FP8
                    keys with UE8M0 (MX) scales, 4 padding rows, top-2048.
* ``long_mxfp4``    8 requests x 1 row, 131072 keys, MXFP4 cache, the last
                    request's new key has slot -1 (padding), top-2048.

Placement of the step's tokens (the workload's own definition, not the
method): the rows of request ``q`` are its last ``query_lens[q]`` positions,
so row ``i`` of the request sits at position ``seq_len - query_len + i``.
Positions ``0 .. seq_len - query_len - 1`` are prefilled before the step.
A position ``t`` of request ``q`` lives in slot
``block_table[q, t // 64] * 64 + t % 64``.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HEADS = 32
DIM = 128
PAGE = 64

# Format names shared by both sides; each side maps them to its own enum.
FORMATS = ("fp8", "fp8_mx", "mxfp4", "mxfp4_rg")

CONFIGS = {
    "tiny_fp8": dict(fmt="fp8", R=2, qlen=(1, 1), seq=(256, 256), pad_rows=0,
                     topk=64, seed=0, outliers=0.0, no_slot_rows=()),
    "fp8_decode": dict(fmt="fp8", R=64, qlen=(1, 1), seq=(4096, 8192), pad_rows=0,
                       topk=2048, seed=2, outliers=0.0, no_slot_rows=()),
    "mxfp4_decode": dict(fmt="mxfp4", R=64, qlen=(1, 1), seq=(16384, 32768), pad_rows=0,
                         topk=2048, seed=3, outliers=0.01, no_slot_rows=()),
    "spec_verify": dict(fmt="fp8_mx", R=128, qlen=(1, 4), seq=(4096, 65536), pad_rows=4,
                        topk=2048, seed=4, outliers=0.0, no_slot_rows=()),
    "long_mxfp4": dict(fmt="mxfp4", R=8, qlen=(1, 1), seq=(131072, 131072), pad_rows=0,
                       topk=2048, seed=5, outliers=0.0, no_slot_rows=(7,)),
}


def _round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of float32 draws (round to nearest even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Float32 values of BF16 bit patterns (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, scale=1.0, shift=0.0, outliers=0.0):
    x = rng.standard_normal(shape, dtype=np.float32) * np.float32(scale) + np.float32(shift)
    if outliers > 0.0:
        hit = rng.random(shape) < outliers
        x = np.where(hit, x * np.float32(20.0), x).astype(np.float32)
    return _round_to_bf16_bits(x)


@dataclass
class Workload:
    name: str
    fmt: str
    seed: int
    topk: int
    seq_lens: np.ndarray        # int32 [R]
    query_lens: np.ndarray      # int32 [R]
    num_rows: int               # real rows + padding rows
    q_bits: np.ndarray          # uint16 [num_rows, 32, 128] BF16 indexer queries
    wv_bits: np.ndarray         # uint16 [num_rows, 32] BF16 head-weight logits
    gamma: np.ndarray           # float32 [128], BF16-representable
    beta: np.ndarray            # float32 [128], BF16-representable
    eps: float
    num_pages: int
    max_pages: int
    block_table: np.ndarray     # int32 [R, max_pages], -1 where unused
    step_key_bits: np.ndarray   # uint16 [num_rows, 128] wk projections of the step's tokens
    step_slots: np.ndarray      # int64 [num_rows], -1 for padding
    row_request: np.ndarray = field(repr=False, default=None)   # int32 [num_rows], -1 padding
    row_position: np.ndarray = field(repr=False, default=None)  # int64 [num_rows], -1 padding

    @property
    def R(self) -> int:
        return int(self.seq_lens.shape[0])

    def prefill_count(self, q: int) -> int:
        return int(self.seq_lens[q]) - int(self.query_lens[q])

    def prefill(self, q: int):
        """(BF16 key bits [n, 128], int64 slots [n]) of request q's prefilled positions."""
        n = self.prefill_count(q)
        rng = np.random.default_rng([self.seed, 1, q])
        bits = _normal_bf16(rng, (n, DIM))
        t = np.arange(n, dtype=np.int64)
        slots = self.block_table[q, t // PAGE].astype(np.int64) * PAGE + t % PAGE
        return bits, slots

    def prefill_all(self):
        parts = [self.prefill(q) for q in range(self.R)]
        if not parts:
            return np.zeros((0, DIM), np.uint16), np.zeros((0,), np.int64)
        return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))

    def cache_bytes(self) -> int:
        return self.num_pages * PAGE * (68 if self.fmt in ("mxfp4", "mxfp4_rg") else 132)


def make_workload(name: str = "tiny_fp8", **overrides) -> Workload:
    """Build a named workload; ``overrides`` replace entries of its recipe
    (``R``, ``qlen``, ``seq``, ``pad_rows``, ``topk``, ``seed``, ``fmt``,
    ``outliers``, ``no_slot_rows``)."""
    spec = dict(CONFIGS[name])
    spec.update(overrides)
    fmt, R, seed = spec["fmt"], int(spec["R"]), int(spec["seed"])
    assert fmt in FORMATS
    rng = np.random.default_rng([seed, 0])
    qlo, qhi = spec["qlen"]
    slo, shi = spec["seq"]
    query_lens = rng.integers(qlo, qhi, size=R, endpoint=True).astype(np.int32)
    seq_lens = rng.integers(slo, shi, size=R, endpoint=True).astype(np.int32)
    seq_lens = np.maximum(seq_lens, query_lens).astype(np.int32)
    pages = [(int(s) + PAGE - 1) // PAGE for s in seq_lens]
    num_pages = max(1, sum(pages))
    max_pages = max([1] + pages)
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((R, max_pages), -1, dtype=np.int32)
    off = 0
    for q, n in enumerate(pages):
        block_table[q, :n] = perm[off:off + n]
        off += n

    real_rows = int(query_lens.sum())
    num_rows = real_rows + int(spec["pad_rows"])
    row_request = np.full(num_rows, -1, dtype=np.int32)
    row_position = np.full(num_rows, -1, dtype=np.int64)
    r = 0
    for q in range(R):
        for i in range(int(query_lens[q])):
            row_request[r] = q
            row_position[r] = int(seq_lens[q]) - int(query_lens[q]) + i
            r += 1

    q_bits = _normal_bf16(rng, (num_rows, HEADS, DIM), outliers=float(spec["outliers"]))
    wv_bits = _normal_bf16(rng, (num_rows, HEADS))
    gamma = bf16_bits_to_f32(_normal_bf16(rng, (DIM,), scale=0.1, shift=1.0))
    beta = bf16_bits_to_f32(_normal_bf16(rng, (DIM,), scale=0.1))
    step_rng = np.random.default_rng([seed, 2])
    step_key_bits = _normal_bf16(step_rng, (num_rows, DIM))

    step_slots = np.full(num_rows, -1, dtype=np.int64)
    for r in range(num_rows):
        q = int(row_request[r])
        if q < 0 or q in spec["no_slot_rows"]:
            continue
        t = int(row_position[r])
        step_slots[r] = int(block_table[q, t // PAGE]) * PAGE + t % PAGE

    return Workload(
        name=name, fmt=fmt, seed=seed, topk=int(spec["topk"]),
        seq_lens=seq_lens, query_lens=query_lens, num_rows=num_rows,
        q_bits=q_bits, wv_bits=wv_bits, gamma=gamma, beta=beta, eps=1e-6,
        num_pages=num_pages, max_pages=max_pages, block_table=block_table,
        step_key_bits=step_key_bits, step_slots=step_slots,
        row_request=row_request, row_position=row_position,
    )
