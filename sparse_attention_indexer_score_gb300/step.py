"""One decode step of the indexer on the GPU, end to end through the C ABI.

``DecodeIndexer`` owns the device state a serving loop keeps between steps
(the paged key cache, the block table, a zero-filled workspace) and runs the
step on the current stream with one decode_step call: quantize_query +
insert_key + decode_layout in one launch -> plan -> scoring -> top-k.  ``GraphedStep``
captures a step with its host copies as one CUDA graph.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import dsa


@dataclass
class StepOutput:
    q_rows: torch.Tensor        # uint8 [rows, 4096]
    w: torch.Tensor             # bf16 [rows, 32]
    starts: torch.Tensor        # int32 [R + 1]
    row_ends: torch.Tensor      # int32 [rows]
    topk: Optional[torch.Tensor]
    logits: Optional[torch.Tensor]


class DecodeIndexer:
    def __init__(self, fmt: str, num_pages: int, block_table: torch.Tensor, gamma: torch.Tensor,
                 beta: torch.Tensor, eps: float, max_rows: int, topk: int, device="cuda",
                 page_stride: Optional[int] = None):
        self.fmt = fmt
        self.device = torch.device(device)
        self.page_stride = int(page_stride or dsa.PAGE_BYTES[fmt])
        self.num_pages = int(num_pages)
        self.cache = torch.zeros(max(1, self.num_pages) * self.page_stride, dtype=torch.uint8, device=self.device)
        self.block_table = block_table.to(self.device, torch.int32).contiguous()
        self.gamma = gamma.to(self.device, torch.float32).contiguous()
        self.beta = beta.to(self.device, torch.float32).contiguous()
        self.eps = float(eps)
        self.k = int(topk)
        R = self.block_table.shape[0]
        max_pages = self.block_table.shape[1]
        self.workspace = dsa.new_workspace(dsa.workspace_size(fmt, max_rows, R, max_pages, self.k), self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def insert(self, keys: torch.Tensor, slots: torch.Tensor) -> None:
        dsa.insert_key(self.fmt, keys, self.gamma, self.beta, self.eps, slots, self.cache, self.page_stride,
                       self.num_pages, self.status)

    def step(self, q: torch.Tensor, wv: torch.Tensor, keys: torch.Tensor, slots: torch.Tensor,
             seq_lens: torch.Tensor, query_lens: torch.Tensor, max_query_len: int,
             want_logits: bool = False, topk_out: Optional[torch.Tensor] = None,
             q_out: Optional[torch.Tensor] = None, w_out: Optional[torch.Tensor] = None) -> StepOutput:
        q_rows, w, starts, row_ends, logits, top = dsa.decode_step(
            self.fmt, q, wv, keys, self.gamma, self.beta, self.eps, slots, self.cache, self.page_stride,
            self.num_pages, seq_lens, query_lens, self.block_table, max_query_len, top_k=self.k,
            want_logits=want_logits, workspace=self.workspace, status=self.status, q_out=q_out, w_out=w_out,
            topk_out=topk_out)
        return StepOutput(q_rows, w, starts, row_ends, top, logits)

    def status_bits(self) -> int:
        return int(self.status.item())


class _Staging:
    """One step's pinned host staging buffer with its named input views, the
    device copy, and the top-k on the device and in pinned host memory."""

    NAMES = ("q", "wv", "keys", "slots", "seq_lens", "query_lens")
    ALIGN = 256

    def __init__(self, ix: DecodeIndexer, like: dict):
        offs, total = {}, 0
        for name in self.NAMES:
            t = like[name]
            offs[name] = total
            total += -(-t.numel() * t.element_size() // self.ALIGN) * self.ALIGN
        self.nbytes = total
        self.host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dev_buf = torch.empty(total, dtype=torch.uint8, device=ix.device)

        def view(buf, name):
            t = like[name]
            n = t.numel() * t.element_size()
            return buf[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)

        self.inputs = {name: view(self.host_buf, name) for name in self.NAMES}
        self.dev = {name: view(self.dev_buf, name) for name in self.NAMES}
        rows = like["q"].shape[0]
        self.topk = torch.empty((rows, ix.k), dtype=torch.int32, device=ix.device)
        self.host_topk = torch.empty((rows, ix.k), dtype=torch.int32).pin_memory()
        for name in self.NAMES:
            self.inputs[name].copy_(like[name])

    def compute(self, ix: DecodeIndexer, max_query_len: int) -> None:
        d = self.dev
        ix.step(d["q"], d["wv"], d["keys"], d["slots"], d["seq_lens"], d["query_lens"], max_query_len,
                topk_out=self.topk)


class GraphedStep:
    """A decode step captured as one CUDA graph, as a serving loop runs it: one
    host-to-device copy of the step's inputs from a pinned staging buffer, the
    step itself (prepare_step, scoring, top-k), and one copy of the top-k
    positions back to a pinned host buffer.

    ``inputs`` holds pinned views ``q``, ``wv``, ``keys``, ``slots``,
    ``seq_lens`` and ``query_lens`` into the staging buffer, shaped and typed
    like the ``like`` tensors given; the caller fills them, calls ``replay()``
    (current stream) and synchronises before reading ``host_topk``.
    """

    NAMES = _Staging.NAMES

    def __init__(self, ix: DecodeIndexer, like: dict, max_query_len: int):
        self.ix = ix
        self.max_query_len = int(max_query_len)
        self.st = _Staging(ix, like)
        self.inputs, self.host_topk, self.staging_bytes = self.st.inputs, self.st.host_topk, self.st.nbytes
        self._run()                      # first use outside capture (library and allocator set up)
        torch.cuda.synchronize(ix.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._run()

    def _run(self) -> None:
        self.st.dev_buf.copy_(self.st.host_buf, non_blocking=True)
        self.st.compute(self.ix, self.max_query_len)
        self.st.host_topk.copy_(self.st.topk, non_blocking=True)

    def replay(self) -> None:
        self.graph.replay()


class StepPipeline:
    """Decode steps with their host copies overlapped, as a serving loop runs
    them back to back: step i's inputs are copied in (one copy from a pinned
    staging buffer, on an input stream) while step i - 1 computes, and step
    i's top-k is copied back (on an output stream) while step i + 1 computes.
    Two staging sets alternate; each step's compute is a CUDA graph replayed
    on the stream current at construction, and events order the three
    streams, so every step still copies its own inputs in and its own result
    out.

    caches: optional list of key-cache tensors laid out like ``ix.cache``;
    step i reads caches[i % len(caches)] (one graph per set and cache).
    A serving loop passes none: every step reads the indexer's own cache.
    ``inputs(i)`` / ``host_topk(i)`` are the pinned views of step i's set.
    ``run(n)`` issues n steps and returns the timing events (start, end)
    bracketing them on the device.
    """

    def __init__(self, ix: DecodeIndexer, like: dict, max_query_len: int, caches=None):
        self.ix = ix
        self.sets = [_Staging(ix, like) for _ in range(2)]
        self.staging_bytes = self.sets[0].nbytes
        caches = list(caches) if caches else [ix.cache]
        own = ix.cache
        dev = ix.device
        self.compute = torch.cuda.current_stream(dev)
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        for st in self.sets:             # first use outside capture
            st.dev_buf.copy_(st.host_buf)
            st.compute(ix, max_query_len)
        torch.cuda.synchronize(dev)
        self.graphs = []                 # [cache][set]
        for c in caches:
            ix.cache = c
            row = []
            for st in self.sets:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    st.compute(ix, max_query_len)
                row.append(g)
            self.graphs.append(row)
        ix.cache = own
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.out_done = [torch.cuda.Event() for _ in range(2)]
        for e in self.computed + self.out_done:
            e.record(self.compute)

    def inputs(self, i: int) -> dict:
        return self.sets[i % 2].inputs

    def host_topk(self, i: int) -> torch.Tensor:
        return self.sets[i % 2].host_topk

    def run(self, n: int):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.compute):
            start.record(self.compute)
            self.s_in.wait_event(start)
            self.s_out.wait_event(start)
            for i in range(n):
                k = i % 2
                st = self.sets[k]
                with torch.cuda.stream(self.s_in):
                    self.s_in.wait_event(self.computed[k])      # the set's previous step has read its inputs
                    st.dev_buf.copy_(st.host_buf, non_blocking=True)
                    self.in_ready[k].record(self.s_in)
                self.compute.wait_event(self.in_ready[k])
                self.compute.wait_event(self.out_done[k])       # its previous top-k has left the device
                self.graphs[i % len(self.graphs)][k].replay()
                self.computed[k].record(self.compute)
                with torch.cuda.stream(self.s_out):
                    self.s_out.wait_event(self.computed[k])
                    st.host_topk.copy_(st.topk, non_blocking=True)
                    self.out_done[k].record(self.s_out)
            self.compute.wait_stream(self.s_in)
            self.compute.wait_stream(self.s_out)
            end.record(self.compute)
        return start, end
