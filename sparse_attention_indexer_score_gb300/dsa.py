"""Python binding of ``libdsa.so`` (C ABI declared in ``include/dsa.h``).

Argument marshalling only: tensors become device pointers, sizes and strides
become integers, the current CUDA stream is passed through, and a negative
return code raises.  Every step of the decode step runs in the library's CUDA
kernels; there is no fallback path.  The library is loaded on first use and a
missing library raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa.so")

FORMATS = {"fp8": 0, "fp8_mx": 1, "mxfp4": 2, "mxfp4_rg": 3}
ERRORS = {-1: "invalid argument", -2: "unsupported", -3: "CUDA launch or driver error"}
STATUS_BITS = {1: "bad slot", 2: "bad page", 4: "bad geometry", 8: "timeout"}
Q_ROW_BYTES = 4096
PAGE_BYTES = {"fp8": 8448, "fp8_mx": 8448, "mxfp4": 4352, "mxfp4_rg": 4352}

_lib = None

_c = ctypes
_P = _c.c_void_p
_I64 = _c.c_int64
_SIGS = {
    "dsa_quantize_query": (_c.c_int, [_c.c_int, _P, _I64, _P, _I64, _I64, _P, _P, _P]),
    "dsa_quantize_queries_rg": (_c.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _P]),
    "dsa_selftest_wait_timeout": (_c.c_int, [_P, _P]),
    "dsa_insert_key": (_c.c_int, [_c.c_int, _P, _I64, _P, _P, _c.c_float, _P, _I64, _P, _I64, _I64, _P, _P]),
    "dsa_decode_layout": (_c.c_int, [_P, _I64, _P, _I64, _I64, _P, _P, _P]),
    "dsa_prepare_step": (_c.c_int, [_c.c_int, _P, _I64, _P, _I64, _I64, _P, _P, _P, _I64, _P, _P, _c.c_float, _P,
                                    _I64, _P, _I64, _I64, _P, _I64, _P, _I64, _I64, _P, _P, _P, _P]),
    "dsa_decode_step": (_c.c_int, [_c.c_int, _P, _I64, _P, _I64, _P, _I64, _P, _P, _c.c_float, _P, _I64, _P, _I64,
                                   _I64, _P, _I64, _P, _I64, _I64, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _I64,
                                   _I64, _P, _P, _c.c_size_t, _P, _P]),
    "dsa_decode_layout_dcp": (_c.c_int, [_P, _I64, _P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P]),
    "dsa_topk_merge": (_c.c_int, [_P, _I64, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P, _I64, _P, _P,
                                  _c.c_size_t, _P]),
    "dsa_query_norm": (_c.c_int, [_P, _I64, _P, _c.c_float, _I64, _P, _I64, _c.c_int, _P]),
    "dsa_workspace_size": (_c.c_size_t, [_c.c_int, _I64, _I64, _I64, _I64]),
    "dsa_score_paged": (_c.c_int, [_c.c_int, _P, _P, _P, _I64, _I64, _P, _I64, _I64, _P, _P, _I64, _I64, _I64,
                                   _P, _I64, _I64, _P, _P, _c.c_size_t, _P, _P]),
    "dsa_score_paged_heads": (_c.c_int, [_c.c_int, _I64, _P, _P, _P, _P, _I64, _I64, _P, _I64, _I64, _P, _P, _I64,
                                         _I64, _I64, _P, _I64, _I64, _P, _P, _c.c_size_t, _P, _P]),
    "dsa_topk_workspace_size": (_c.c_size_t, [_I64, _I64]),
    "dsa_topk": (_c.c_int, [_P, _I64, _P, _I64, _I64, _I64, _P, _P, _c.c_size_t, _P]),
    "dsa_topk_noalloc": (_c.c_int, [_P, _I64, _P, _I64, _I64, _I64, _P, _P]),
    "dsa_set_score_timing": (None, [_P, _P]),
    "dsa_timing_event_create": (_c.c_int, [_c.POINTER(_P)]),
    "dsa_timing_event_destroy": (_c.c_int, [_P]),
    "dsa_timing_elapsed_ms": (_c.c_int, [_P, _P, _c.POINTER(_c.c_float)]),
    "dsa_version": (_c.c_char_p, []),
    "dsa_probe_mma": (_c.c_int, [_c.c_int, _I64, _P, _P]),
}


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device: torch.device):
    return torch.cuda.current_stream(device).cuda_stream


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what}: {ERRORS.get(rc, rc)}")


def _fmt(fmt: str) -> int:
    if fmt not in FORMATS:
        raise ValueError(f"unknown format {fmt!r}; expected one of {sorted(FORMATS)}")
    return FORMATS[fmt]


def _query_args(q, wv, q_out, w_out):
    if q.dtype != torch.bfloat16 or q.dim() != 3 or tuple(q.shape[1:]) != (32, 128) or q.stride(2) != 1 \
            or q.stride(1) != 128:
        raise ValueError("q must be BF16 [rows, 32, 128] with contiguous heads")
    if wv.dtype != torch.bfloat16 or wv.dim() != 2 or wv.shape[1] != 32 or wv.stride(1) != 1:
        raise ValueError("wv must be BF16 [rows, 32]")
    rows = q.shape[0]
    if q_out is None:
        q_out = torch.zeros((rows, Q_ROW_BYTES), dtype=torch.uint8, device=q.device)
    if w_out is None:
        w_out = torch.empty((rows, 32), dtype=torch.bfloat16, device=q.device)
    return q_out, w_out


def _key_args(k, gamma, beta, slots):
    if k.dtype != torch.bfloat16 or k.dim() != 2 or k.shape[1] != 128 or k.stride(1) != 1:
        raise ValueError("k must be BF16 [n, 128] with contiguous rows")
    if slots.dtype != torch.int64 or slots.dim() != 1 or slots.numel() != k.shape[0] or \
            (slots.numel() and slots.stride(0) != 1):
        raise ValueError("slots must be int64 [n], one per key")
    if gamma.dtype != torch.float32 or beta.dtype != torch.float32 or gamma.numel() != 128 or beta.numel() != 128:
        raise ValueError("gamma and beta must be FP32 [128]")


def _layout_args(seq_lens, query_lens, num_rows, starts, row_ends):
    if seq_lens.dim() != 1 or query_lens.dim() != 1:
        raise ValueError("Sequence and query lengths must be one-dimensional")
    if seq_lens.dtype != torch.int32 or query_lens.dtype != torch.int32:
        raise ValueError("lengths must be int32")
    R = query_lens.numel()
    dev = query_lens.device
    if starts is None:
        starts = torch.empty(R + 1, dtype=torch.int32, device=dev)
    if row_ends is None:
        row_ends = torch.empty(max(num_rows, 0), dtype=torch.int32, device=dev)
    return starts, row_ends


def quantize_query(fmt: str, q: torch.Tensor, wv: torch.Tensor,
                   q_out: Optional[torch.Tensor] = None,
                   w_out: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """q: BF16 [rows, 32, 128] (row stride >= 4096); wv: BF16 [rows, 32].
    Returns (uint8 [rows, 4096] quantised rows, BF16 [rows, 32] head weights)."""
    q_out, w_out = _query_args(q, wv, q_out, w_out)
    rows = q.shape[0]
    rc = lib().dsa_quantize_query(_fmt(fmt), _ptr(q), q.stride(0), _ptr(wv), wv.stride(0), rows,
                                  _ptr(q_out), _ptr(w_out), _stream(q.device))
    _check(rc, "dsa_quantize_query")
    return q_out, w_out


def quantize_queries_rg(q: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """q: BF16 [rows, heads, 128], heads 16, 32 or 64, unit column stride.
    Returns (uint8 [rows, heads, 64] E2M1 payload, uint8 [rows, 1, 4, 16, 4]
    row-group block scales)."""
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[2] != 128 or q.stride(2) != 1:
        raise ValueError("q must be BF16 [rows, heads, 128] with contiguous heads")
    rows, heads = q.shape[0], q.shape[1]
    payload = torch.empty((rows, heads, 64), dtype=torch.uint8, device=q.device)
    scales = torch.empty((rows, 1, 4, 16, 4), dtype=torch.uint8, device=q.device)
    rc = lib().dsa_quantize_queries_rg(_ptr(q), q.stride(0), q.stride(1), heads, rows, _ptr(payload),
                                       _ptr(scales), _stream(q.device))
    _check(rc, "dsa_quantize_queries_rg")
    return payload, scales


def selftest_wait_timeout(status: torch.Tensor) -> None:
    """Runs the failure-detection self-check: a bounded wait that runs out
    (about one second) and sets the timeout bit of ``status`` (int32 [1])."""
    if status.dtype != torch.int32 or status.numel() < 1 or not status.is_cuda:
        raise ValueError("status must be an int32 CUDA tensor")
    _check(lib().dsa_selftest_wait_timeout(_ptr(status), _stream(status.device)), "dsa_selftest_wait_timeout")


def insert_key(fmt: str, k: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float,
               slots: torch.Tensor, cache: torch.Tensor, page_stride: int, num_pages: int,
               status: Optional[torch.Tensor] = None) -> None:
    """k: BF16 [n, 128]; gamma, beta: FP32 [128]; slots: int64 [n]; cache: uint8 buffer."""
    _key_args(k, gamma, beta, slots)
    rc = lib().dsa_insert_key(_fmt(fmt), _ptr(k), k.stride(0), _ptr(gamma), _ptr(beta), float(eps),
                              _ptr(slots), k.shape[0], _ptr(cache), int(page_stride), int(num_pages),
                              _ptr(status), _stream(k.device))
    _check(rc, "dsa_insert_key")


def decode_layout(seq_lens: torch.Tensor, query_lens: torch.Tensor, num_rows: int,
                  starts: Optional[torch.Tensor] = None,
                  row_ends: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """int32 seq_lens [>= R], query_lens [R] -> (starts int32 [R + 1], row_ends int32 [num_rows])."""
    starts, row_ends = _layout_args(seq_lens, query_lens, num_rows, starts, row_ends)
    R = query_lens.numel()
    dev = query_lens.device
    rc = lib().dsa_decode_layout(_ptr(seq_lens), seq_lens.numel(), _ptr(query_lens), R, int(num_rows),
                                 _ptr(starts), _ptr(row_ends), _stream(dev))
    _check(rc, "dsa_decode_layout")
    return starts, row_ends


def decode_layout_dcp(seq_lens: torch.Tensor, query_lens: torch.Tensor, num_rows: int, dcp_rank: int,
                      dcp_world_size: int, interleave: int = 1) -> Tuple[torch.Tensor, torch.Tensor]:
    """decode_layout with rank-local row bounds under DCP."""
    starts, row_ends = _layout_args(seq_lens, query_lens, num_rows, None, None)
    rc = lib().dsa_decode_layout_dcp(_ptr(seq_lens), seq_lens.numel(), _ptr(query_lens), query_lens.numel(),
                                     int(num_rows), int(dcp_rank), int(dcp_world_size), int(interleave),
                                     _ptr(starts), _ptr(row_ends), _stream(query_lens.device))
    _check(rc, "dsa_decode_layout_dcp")
    return starts, row_ends


def topk_merge(scores: torch.Tensor, idx: torch.Tensor, world: int, k: int, interleave: int, k_out: int,
               rank: Optional[int] = None, workspace: Optional[torch.Tensor] = None):
    """scores FP32 [rows, >= world*k] and idx int32 [rows, >= world*k] (rank w's
    candidates at columns w*k ..) -> (int32 [rows, k_out] global positions,
    int32 [rows, k_out] local slots of ``rank`` or None)."""
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be FP32 [rows, world * k]")
    if idx.dtype != torch.int32 or idx.dim() != 2 or idx.stride(1) != 1 or idx.shape[0] != scores.shape[0]:
        raise ValueError("idx must be int32 [rows, world * k]")
    rows = scores.shape[0]
    dev = scores.device
    if workspace is None:
        workspace = new_workspace(topk_workspace_size(rows, k_out), dev)
    out = torch.empty((rows, k_out), dtype=torch.int32, device=dev)
    out_local = torch.empty((rows, k_out), dtype=torch.int32, device=dev) if rank is not None else None
    rc = lib().dsa_topk_merge(_ptr(scores), scores.stride(0), _ptr(idx), idx.stride(0), rows, int(world), int(k),
                              int(interleave), int(k_out), _ptr(out), int(rank or 0), _ptr(out_local),
                              _ptr(workspace), workspace.numel(), _stream(dev))
    _check(rc, "dsa_topk_merge")
    return out, out_local


NORM_VARIANTS = {"auto": -1, "row": 0, "tiled": 1}


def query_norm(x: torch.Tensor, w: torch.Tensor, eps: float, variant: str = "auto",
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """QueryNorm: x BF16 [batch, >= 1536] (columns 0..1535 are q_a), w BF16 [1536]
    -> q_c BF16 [batch, 1536] (or ``out``).  variant: "row", "tiled" or "auto"."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] < 1536 or x.stride(1) != 1:
        raise ValueError("x must be BF16 [batch, >= 1536] with contiguous columns")
    if w.dtype != torch.bfloat16 or w.numel() != 1536:
        raise ValueError("w must be BF16 [1536]")
    if variant not in NORM_VARIANTS:
        raise ValueError(f"variant must be one of {sorted(NORM_VARIANTS)}")
    if out is None:
        out = torch.empty((x.shape[0], 1536), dtype=torch.bfloat16, device=x.device)
    rc = lib().dsa_query_norm(_ptr(x), x.stride(0), _ptr(w), float(eps), x.shape[0], _ptr(out), out.stride(0),
                              NORM_VARIANTS[variant], _stream(x.device))
    _check(rc, "dsa_query_norm")
    return out


def prepare_step(fmt: str, q: torch.Tensor, wv: torch.Tensor, k: torch.Tensor, gamma: torch.Tensor,
                 beta: torch.Tensor, eps: float, slots: torch.Tensor, cache: torch.Tensor, page_stride: int,
                 num_pages: int, seq_lens: torch.Tensor, query_lens: torch.Tensor, num_rows: int,
                 q_out: Optional[torch.Tensor] = None, w_out: Optional[torch.Tensor] = None,
                 starts: Optional[torch.Tensor] = None, row_ends: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None):
    """quantize_query + insert_key + decode_layout in one launch (same arguments
    and results).  Returns (q_rows, w, starts, row_ends)."""
    q_out, w_out = _query_args(q, wv, q_out, w_out)
    _key_args(k, gamma, beta, slots)
    starts, row_ends = _layout_args(seq_lens, query_lens, num_rows, starts, row_ends)
    rc = lib().dsa_prepare_step(_fmt(fmt), _ptr(q), q.stride(0), _ptr(wv), wv.stride(0), q.shape[0],
                                _ptr(q_out), _ptr(w_out), _ptr(k), k.stride(0), _ptr(gamma), _ptr(beta), float(eps),
                                _ptr(slots), k.shape[0], _ptr(cache), int(page_stride), int(num_pages),
                                _ptr(seq_lens), seq_lens.numel(), _ptr(query_lens), query_lens.numel(),
                                int(num_rows), _ptr(starts), _ptr(row_ends), _ptr(status), _stream(q.device))
    _check(rc, "dsa_prepare_step")
    return q_out, w_out, starts, row_ends


def decode_step(fmt: str, q: torch.Tensor, wv: torch.Tensor, k: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor,
                eps: float, slots: torch.Tensor, cache: torch.Tensor, page_stride: int, num_pages: int,
                seq_lens: torch.Tensor, query_lens: torch.Tensor, block_table: torch.Tensor, max_query_len: int,
                top_k: int = 0, want_logits: bool = False, workspace: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, q_out: Optional[torch.Tensor] = None,
                w_out: Optional[torch.Tensor] = None, starts: Optional[torch.Tensor] = None,
                row_ends: Optional[torch.Tensor] = None, topk_out: Optional[torch.Tensor] = None):
    """prepare_step then score_paged on its outputs, in one call
    (``dsa_decode_step``: every argument checked before the first launch).  Returns (q_rows, w, starts, row_ends, logits or
    None, top-k or None)."""
    num_rows = q.shape[0]
    q_out, w_out = _query_args(q, wv, q_out, w_out)
    _key_args(k, gamma, beta, slots)
    starts, row_ends = _layout_args(seq_lens, query_lens, num_rows, starts, row_ends)
    if block_table.dtype != torch.int32 or (block_table.dim() == 2 and block_table.numel() and block_table.stride(1) != 1):
        raise ValueError("block_table must be int32 with contiguous rows")
    R = query_lens.numel()
    max_pages = block_table.shape[1] if block_table.dim() == 2 else 0
    width = max_pages * 64
    dev = q.device
    logits = torch.empty((num_rows, width), dtype=torch.float32, device=dev) if want_logits else None
    if top_k > 0 and topk_out is None:
        topk_out = torch.empty((num_rows, top_k), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(fmt, num_rows, R, max_pages, top_k), dev)
    rc = lib().dsa_decode_step(
        _fmt(fmt), _ptr(q), q.stride(0), _ptr(wv), wv.stride(0), _ptr(k), k.stride(0), _ptr(gamma), _ptr(beta),
        float(eps), _ptr(slots), k.shape[0], _ptr(cache), int(page_stride), int(num_pages), _ptr(seq_lens),
        seq_lens.numel(), _ptr(query_lens), R, num_rows, _ptr(block_table),
        block_table.stride(0) if block_table.dim() == 2 else 0, max_pages, int(max_query_len), _ptr(q_out),
        _ptr(w_out), _ptr(starts), _ptr(row_ends), _ptr(logits), logits.stride(0) if logits is not None else 0,
        int(top_k), _ptr(topk_out), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev))
    _check(rc, "dsa_decode_step")
    return q_out, w_out, starts, row_ends, logits, topk_out


def workspace_size(fmt: str, rows: int, num_requests: int, max_pages: int, k: int) -> int:
    return int(lib().dsa_workspace_size(_fmt(fmt), rows, num_requests, max_pages, k))


def topk_workspace_size(rows: int, k: int) -> int:
    return int(lib().dsa_topk_workspace_size(rows, k))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled workspace (the library leaves it zero-filled after each call)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def score_paged(fmt: str, q_rows: torch.Tensor, w: torch.Tensor, cache: torch.Tensor, page_stride: int,
                num_pages: int, block_table: torch.Tensor, starts: torch.Tensor, row_ends: torch.Tensor,
                max_query_len: int, k: int = 0, want_logits: bool = False,
                workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                logits: Optional[torch.Tensor] = None, topk_out: Optional[torch.Tensor] = None):
    """Paged logits (+ top-k).  Returns (logits FP32 [rows, max_pages*64] or None,
    top-k int32 [rows, k] or None)."""
    rows = row_ends.numel()
    R = starts.numel() - 1
    max_pages = block_table.shape[1] if block_table.dim() == 2 else 0
    width = max_pages * 64
    dev = q_rows.device
    if block_table.dtype != torch.int32 or starts.dtype != torch.int32 or row_ends.dtype != torch.int32:
        raise ValueError("block_table, starts and row_ends must be int32")
    if block_table.dim() == 2 and block_table.numel() and block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    if want_logits and logits is None:
        logits = torch.empty((rows, width), dtype=torch.float32, device=dev)
    if k > 0 and topk_out is None:
        topk_out = torch.empty((rows, k), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(workspace_size(fmt, rows, R, max_pages, k), dev)
    rc = lib().dsa_score_paged(
        _fmt(fmt), _ptr(q_rows), _ptr(w), _ptr(cache), int(page_stride), int(num_pages),
        _ptr(block_table), block_table.stride(0) if block_table.dim() == 2 else 0, max_pages,
        _ptr(starts), _ptr(row_ends), R, rows, int(max_query_len),
        _ptr(logits), logits.stride(0) if logits is not None else 0,
        int(k), _ptr(topk_out), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev))
    _check(rc, "dsa_score_paged")
    return logits, topk_out


def score_paged_heads(fmt: str, payload: torch.Tensor, scales: torch.Tensor, w: torch.Tensor, cache: torch.Tensor,
                      page_stride: int, num_pages: int, block_table: torch.Tensor, starts: torch.Tensor,
                      row_ends: torch.Tensor, max_query_len: int, k: int = 0, want_logits: bool = False,
                      workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """Paged logits (+ top-k) of MXFP4 queries of 16, 32 or 64 heads:
    payload uint8 [rows, heads, 64] and scales uint8 [rows, 1, 4, 16, 4] from
    ``quantize_queries_rg``, w BF16 [rows, heads].  Returns (logits or None,
    top-k or None) as ``score_paged``."""
    if payload.dtype != torch.uint8 or payload.dim() != 3 or payload.shape[2] != 64 or not payload.is_contiguous():
        raise ValueError("payload must be contiguous uint8 [rows, heads, 64]")
    rows, heads = payload.shape[0], payload.shape[1]
    if scales.dtype != torch.uint8 or scales.numel() != rows * 256 or not scales.is_contiguous():
        raise ValueError("scales must be contiguous uint8 [rows, 1, 4, 16, 4]")
    if w.dtype != torch.bfloat16 or tuple(w.shape) != (rows, heads) or not w.is_contiguous():
        raise ValueError("w must be contiguous BF16 [rows, heads]")
    if row_ends.numel() != rows:
        raise ValueError("row_ends must hold one bound per query row")
    R = starts.numel() - 1
    max_pages = block_table.shape[1] if block_table.dim() == 2 else 0
    width = max_pages * 64
    dev = payload.device
    logits = torch.empty((rows, width), dtype=torch.float32, device=dev) if want_logits else None
    top = torch.empty((rows, k), dtype=torch.int32, device=dev) if k > 0 else None
    if workspace is None:
        workspace = new_workspace(workspace_size(fmt, rows, R, max_pages, k), dev)
    rc = lib().dsa_score_paged_heads(
        _fmt(fmt), heads, _ptr(payload), _ptr(scales), _ptr(w), _ptr(cache), int(page_stride), int(num_pages),
        _ptr(block_table), block_table.stride(0) if block_table.dim() == 2 else 0, max_pages,
        _ptr(starts), _ptr(row_ends), R, rows, int(max_query_len),
        _ptr(logits), logits.stride(0) if logits is not None else 0,
        int(k), _ptr(top), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev))
    _check(rc, "dsa_score_paged_heads")
    return logits, top


def topk(logits: torch.Tensor, row_ends: torch.Tensor, k: int, width: Optional[int] = None,
         workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Top-k positions of each row of FP32 logits [rows, >= width] (valid below row_ends)."""
    if logits.dtype != torch.float32 or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be FP32 [rows, width] with contiguous rows")
    rows = logits.shape[0]
    width = logits.shape[1] if width is None else int(width)
    if out is None:
        out = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    if workspace is None:
        workspace = new_workspace(topk_workspace_size(rows, k), logits.device)
    rc = lib().dsa_topk(_ptr(logits), logits.stride(0), _ptr(row_ends), rows, width, int(k), _ptr(out),
                        _ptr(workspace), workspace.numel(), _stream(logits.device))
    _check(rc, "dsa_topk")
    return out


class TimingEvent:
    """A CUDA event of the library's own runtime (for ``set_score_timing``)."""

    def __init__(self):
        h = _P()
        _check(lib().dsa_timing_event_create(ctypes.byref(h)), "dsa_timing_event_create")
        self.handle = h.value

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.dsa_timing_event_destroy(self.handle)
            self.handle = None

    def elapsed_ms(self, end: "TimingEvent") -> float:
        ms = _c.c_float()
        _check(lib().dsa_timing_elapsed_ms(self.handle, end.handle, ctypes.byref(ms)), "dsa_timing_elapsed_ms")
        return float(ms.value)


TOPK_NOALLOC_MAX_ROWS = 64


def topk_noalloc(logits: torch.Tensor, row_ends: torch.Tensor, k: int, width: Optional[int] = None,
                 out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """``topk`` without a workspace, for callers that cannot allocate device
    memory: the library's own static scratch (at most 64 rows) is used instead.
    Pass ``out`` to avoid the one allocation this wrapper would make."""
    if logits.dtype != torch.float32 or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be FP32 [rows, width] with contiguous rows")
    rows = logits.shape[0]
    if rows > TOPK_NOALLOC_MAX_ROWS:
        raise ValueError(f"topk_noalloc handles at most {TOPK_NOALLOC_MAX_ROWS} rows per call, got {rows}")
    width = logits.shape[1] if width is None else int(width)
    if out is None:
        out = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    rc = lib().dsa_topk_noalloc(_ptr(logits), logits.stride(0), _ptr(row_ends), rows, width, int(k), _ptr(out),
                                _stream(logits.device))
    _check(rc, "dsa_topk_noalloc")
    return out


def set_score_timing(before: Optional[TimingEvent], after: Optional[TimingEvent]) -> None:
    """Record `before`/`after` around the scoring kernel of later score_paged calls."""
    if before is None or after is None:
        lib().dsa_set_score_timing(None, None)
    else:
        lib().dsa_set_score_timing(before.handle, after.handle)


MMA_KINDS = {"fp8": 0, "mxf4": 1}
MMA_K = {"fp8": 32, "mxf4": 64}


def probe_mma(kind: str, iters: int, status: Optional[torch.Tensor] = None,
              device: Optional[torch.device] = None) -> None:
    """Launches the tensor-core rate probe (``dsa_probe_mma``) on the current
    stream: one CTA per SM, ``iters`` MMAs of 128 x 128 x K each."""
    if kind not in MMA_KINDS:
        raise ValueError(f"kind must be one of {sorted(MMA_KINDS)}")
    dev = device or torch.device("cuda", torch.cuda.current_device())
    _check(lib().dsa_probe_mma(MMA_KINDS[kind], int(iters), _ptr(status), _stream(dev)), "dsa_probe_mma")


def version() -> str:
    return lib().dsa_version().decode()
