"""Benchmark of the DSA lightning-indexer decode step on GB300.

One step = the whole hot path over one batch of seeded synthetic inputs, one
decode_step call: quantize_query + insert_key + decode_layout in one launch ->
the scoring plan -> the scoring kernel -> top-k selection.  The headline
workload is ``spec_verify`` (128 requests x 1..4 verify rows, 4096..65536
keys, FP8 keys with UE8M0 scales, top-2048), the largest one that the step
runs on one GPU; ``fp8_decode``, ``mxfp4_decode`` and ``long_mxfp4`` follow,
each with an object of the same keys under ``configs``.

Prints one JSON line.  ``value`` is scored keys per second (sum of the row
bounds of a step / device time of a step) with inputs resident in HBM.  The K
timed steps run as one captured CUDA graph, replayed until at least 100 ms
have been timed, each replay between CUDA events; the median replay gives the
step time.  The key cache is replicated until the replicas exceed three times
the L2 size and the steps use them in turn, so every step reads its keys from
HBM.  ``e2e`` is the same metric through the public API with every step
copying its inputs in from pinned host memory and its top-k back
(``StepPipeline``; ``e2e_graphed`` and ``e2e_eager`` run the step one at a
time).  ``--fmt`` runs workloads in another cache format (e.g. ``mxfp4_rg``);
``--op`` times QueryNorm or the DCP top-k merge instead of the step.
``--impl reference`` times the CPU oracle on the headline workload instead.

Multi-GPU (``torchrun``): every rank runs its own replica of the workload
(the step has no exchange); the timing is the max over ranks and ``value``
sums the keys of all ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import numpy as np  # noqa: E402

METRIC = "indexer scored keys/sec and cache GB/s (score+top-k) vs roofline, 1 GB300"
UNIT = "keys/s"
STEP_KERNELS = 4   # decode_step: prepare (quantize + insert + layout), plan, score, select
FP4_FORMATS = ("mxfp4", "mxfp4_rg")


def workload_desc(wl) -> str:
    kind = {"fp8": "FP8 E4M3 keys, FP32 scales (132 B/token)",
            "fp8_mx": "FP8 E4M3 keys, UE8M0 scales (132 B/token)",
            "mxfp4": "MXFP4 keys (68 B/token)",
            "mxfp4_rg": "MXFP4 keys, row-group page layout (68 B/token)"}[wl.fmt]
    return (f"{wl.name}: {wl.R} requests, {int(wl.query_lens.sum())} rows (+{wl.num_rows - int(wl.query_lens.sum())}"
            f" padding), seq {int(wl.seq_lens.min())}..{int(wl.seq_lens.max())}, {kind}, top-{wl.topk}")


def algorithmic_bytes(wl, row_ends) -> dict:
    """Bytes the step must move at least: unique cache bytes of the scored keys
    (each request's keys once), the quantised query rows and head weights, the
    block-table entries read, and the top-k indices written."""
    per_token = 68 if wl.fmt in FP4_FORMATS else 132
    starts = np.concatenate([[0], np.cumsum(wl.query_lens)])
    keys_unique = 0
    pages = 0
    for q in range(wl.R):
        e = row_ends[starts[q]:starts[q + 1]]
        m = int(e.max()) if e.size else 0
        keys_unique += m
        pages += (m + 63) // 64
    q_bytes = 2176 if wl.fmt in FP4_FORMATS else 4096
    cache = keys_unique * per_token
    other = wl.num_rows * (q_bytes + 64 + 4) + pages * 4
    topk = wl.num_rows * wl.topk * 4
    return dict(cache=cache, score_kernel=cache + other, step=cache + other + topk,
                keys_unique=keys_unique, scored=int(row_ends.sum()))


class ClockSampler:
    """nvidia-smi samples of SM clocks and throttle reasons during a region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        import datetime
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10 or not parts[2].isdigit():
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if self.t0 is not None and not (self.t0 - 0.05 <= ts <= (self.t1 or ts) + 0.05):
                    continue
                rows.append(parts[1:])
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"], "samples": 0}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]), "reasons": reasons,
                "samples": len(rows)}


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1700.0, "source": "fallback"}


NOMINAL_HBM_GBS = 7900.0
# Dense tensor rate of the score kernel's MMA kind over bf16's, from the nominal
# per-GPU figures (bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s).
TENSOR_RATIO = {"fp8": 2.0, "fp8_mx": 2.0, "mxfp4": 6.0, "mxfp4_rg": 6.0}
FLOPS_PER_SCORED_KEY = 2 * 32 * 128   # one row's 32 head dot products of 128 columns


def tensor_side(scored_keys: int, kernel_ms: float, fmt: str, peaks: dict) -> dict:
    """The score kernel against the tensor-core roof: algorithmic FLOPs per
    launch over its event time, against the rate of the kernel's MMA kind
    measured on this GPU by the library's probe (``mma_tflops``), else the
    measured burst bf16 rate (the kernel is timed alone) times the nominal
    ratio of the MMA's operand type."""
    flops = FLOPS_PER_SCORED_KEY * scored_keys
    achieved = flops / (kernel_ms / 1e3) / 1e12
    kind = "mxf4" if fmt in FP4_FORMATS else "fp8"
    probe = peaks.get("mma_tflops", {}).get(kind)
    if probe:
        peak, source = probe, (f"measured on this GPU: dense tcgen05 {kind} MMA rate "
                               "(128 x 128 tiles, operands in shared memory)")
    else:
        peak = peaks["bf16_tflops"] * TENSOR_RATIO[fmt]
        source = f"{peaks['source']} burst bf16 x {TENSOR_RATIO[fmt]:g} (nominal {fmt} / bf16)"
    return {"flops_per_launch": flops, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": source}


def measure_mma_tflops(iters: int = 1 << 16, reps: int = 5) -> dict:
    """Dense tensor-core rates of the scorer's MMA kinds on this GPU, from the
    library's probe (one CTA per SM issuing back-to-back 128 x 128 x K MMAs),
    timed with CUDA events on the stream: the best of ``reps`` launches."""
    import torch
    from sparse_attention_indexer_score_gb300 import dsa
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {}
    for kind in ("fp8", "mxf4"):
        dsa.probe_mma(kind, iters, status)
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dsa.probe_mma(kind, iters, status)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        if int(status.item()) != 0:
            raise RuntimeError("the MMA probe's final wait gave up")
        out[kind] = 2 * 128 * 128 * dsa.MMA_K[kind] * iters * sms / (best / 1e3) / 1e12
    return out


def score_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("score.cu", "common.cuh", "scan.cuh"):
        h.update(open(os.path.join(ROOT, "sparse_attention_indexer_score_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_key(wl) -> str:
    """Name of a workload's entry in the traffic record: the workload's name,
    with ``/<format>`` when its cache format was overridden."""
    from synth.workloads import CONFIGS
    return wl.name if wl.fmt == CONFIGS[wl.name]["fmt"] else f"{wl.name}/{wl.fmt}"


def ncu_traffic(workload: str, units_per_launch: int):
    """DRAM bytes per launch of the scoring kernel from the committed ncu
    summary, scaled to this launch, or None when absent or stale."""
    path = os.path.join(ROOT, "profiles", "score_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(workload)
    if not e or e.get("source_hash") != score_source_hash():
        return None
    return float(e["dram_bytes"]) * units_per_launch / float(e["units"])


# ----------------------------------------------------------------- CPU oracle
def _request_problem(wl, q):
    """The oracle's inputs for request q alone: its quantised rows, their bounds,
    a compact cache holding its pages (built by the oracle's own insert)."""
    from oracle import indexer as O
    from synth import bf16_bits_to_f32
    rows = [r for r in range(wl.num_rows) if wl.row_request[r] == q]
    q_rows, w = O.quantize_query(wl.fmt, bf16_bits_to_f32(wl.q_bits[rows]), bf16_bits_to_f32(wl.wv_bits[rows]))
    _, row_ends = O.decode_layout(wl.seq_lens, wl.query_lens, wl.num_rows)
    stride = O.page_bytes(wl.fmt)
    n = (int(wl.seq_lens[q]) + 63) // 64
    remap = {int(p): i for i, p in enumerate(wl.block_table[q, :n])}
    cache = np.zeros(max(1, n) * stride, np.uint8)
    kb, sl = wl.prefill(q)
    sl2 = np.array([remap[int(s // 64)] * 64 + int(s % 64) for s in sl], dtype=np.int64)
    O.insert_key(wl.fmt, cache, stride, n, bf16_bits_to_f32(kb), wl.gamma, wl.beta, wl.eps, sl2)
    srows = [r for r in rows if wl.step_slots[r] >= 0]
    if srows:
        ss = wl.step_slots[srows]
        sl3 = np.array([remap[int(s // 64)] * 64 + int(s % 64) for s in ss], dtype=np.int64)
        O.insert_key(wl.fmt, cache, stride, n, bf16_bits_to_f32(wl.step_key_bits[srows]), wl.gamma, wl.beta,
                     wl.eps, sl3)
    return dict(q_rows=q_rows, w=w, starts=np.array([0, len(rows)], np.int32),
                row_ends=row_ends[rows], cache=cache, bt=np.arange(n, dtype=np.int32)[None, :], stride=stride)


def oracle_sample(wl, budget_s: float, rng_seed: int = 0):
    """Times the oracle's score + top-k, request by request in a seeded random
    order, until about ``budget_s`` seconds; returns (scored keys, seconds, desc).
    Building each request's cache is set-up and is not timed."""
    from oracle import indexer as O
    order = np.random.default_rng(rng_seed).permutation(wl.R)
    keys, secs, used = 0, 0.0, 0
    for q in order:
        if wl.query_lens[q] == 0:
            continue
        o = _request_problem(wl, int(q))
        t = time.perf_counter()
        s = O.score_paged(wl.fmt, o["q_rows"], o["w"], o["cache"], o["stride"], o["bt"], o["starts"], o["row_ends"])
        O.topk(s, o["row_ends"], wl.topk)
        secs += time.perf_counter() - t
        keys += int(o["row_ends"].sum())
        used += 1
        if secs >= budget_s:
            break
    return keys, secs, f"{used} of {wl.R} requests of {wl.name} (score + top-k of their rows)"


def oracle_one_core(wl, budget_s: float):
    """``oracle_sample`` on one host core: a child process whose BLAS and
    OpenMP pools hold one thread, on the same workload.  Returns (scored keys,
    seconds, desc), or None when the child fails."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, bench\nfrom synth import make_workload\n"
            f"wl = make_workload({wl.name!r}, fmt={wl.fmt!r})\n"
            f"print(json.dumps(bench.oracle_sample(wl, {float(budget_s)!r})))")
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=600)
        keys, secs, desc = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, OSError, ValueError, IndexError):
        return None
    return int(keys), float(secs), str(desc)


def run_reference(args, wl):
    """The oracle on the host cores: each step a bounded sample of the workload."""
    from oracle import indexer as O
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    per_step = max(0.5, min(8.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(wl, per_step / 4)
    keys = 0
    secs = 0.0
    desc = ""
    for i in range(args.steps):
        k, s, desc = oracle_sample(wl, per_step, rng_seed=i)
        keys += k
        secs += s
    value = keys / secs if secs > 0 else 0.0
    _, row_ends = O.decode_layout(wl.seq_lens, wl.query_lens, wl.num_rows)
    ab = algorithmic_bytes(wl, row_ends)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, ab, args.gpus),
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step about {per_step:.1f} s of oracle work: {desc}"},
    }
    print(json.dumps(line))


# ----------------------------------------------------------------- ranks
def max_over_ranks(values, device=None) -> list:
    """Element-wise maximum of ``values`` over the ranks of the default
    process group (the values themselves when there is no group)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_step_per_rank: float, steps: int, world: int, total_ms: float) -> float:
    """Units all ranks processed per second: every rank runs the same
    per-step work (weak scaling), timed by the slowest rank."""
    return units_per_step_per_rank * steps * world / (total_ms / 1e3)


# ----------------------------------------------------------------- GPU
TIMED_MS_MIN = 100.0   # every workload's timed region lasts at least this long


def measure_workload(args, wl, world, local_rank, e2e_modes=("pipelined", "graphed", "eager")):
    """Times one workload on this rank's GPU.  Returns the rank-local raw
    numbers (times in ms) and the workload's config object."""
    import torch

    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from sparse_attention_indexer_score_gb300 import dsa
    from sparse_attention_indexer_score_gb300.step import DecodeIndexer, GraphedStep, StepPipeline
    from dsa_case import bf16_tensor

    dev = torch.device("cuda", local_rank)
    ix = DecodeIndexer(wl.fmt, wl.num_pages, torch.from_numpy(wl.block_table), torch.from_numpy(wl.gamma),
                       torch.from_numpy(wl.beta), wl.eps, wl.num_rows, wl.topk, dev)
    kb, sl = wl.prefill_all()
    chunk = 1 << 20
    for i in range(0, kb.shape[0], chunk):
        ix.insert(bf16_tensor(kb[i:i + chunk], dev), torch.from_numpy(sl[i:i + chunk]).to(dev))
    del kb, sl
    # Inputs larger than L2: replicas of the key cache, one per step in turn, so
    # that every step reads its keys from HBM (no flush kernel between steps).
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20) or (126 << 20)
    cache_bytes = ix.cache.numel()
    n_rep = max(2, min(64, -(-3 * l2 // cache_bytes)))
    caches = [ix.cache] + [ix.cache.clone() for _ in range(n_rep - 1)]
    host = dict(q=bf16_tensor(wl.q_bits, "cpu"), wv=bf16_tensor(wl.wv_bits, "cpu"),
                keys=bf16_tensor(wl.step_key_bits, "cpu"), slots=torch.from_numpy(wl.step_slots),
                seq=torch.from_numpy(wl.seq_lens), qlen=torch.from_numpy(wl.query_lens))
    d = {k: v.to(dev) for k, v in host.items()}
    max_q = int(wl.query_lens.max(initial=0))
    topk_out = torch.empty((wl.num_rows, wl.topk), dtype=torch.int32, device=dev)
    q_out = torch.zeros((wl.num_rows, 4096), dtype=torch.uint8, device=dev)
    w_out = torch.empty((wl.num_rows, 32), dtype=torch.bfloat16, device=dev)

    def step(inp, r):
        ix.cache = caches[r]
        return ix.step(inp["q"], inp["wv"], inp["keys"], inp["slots"], inp["seq"], inp["qlen"], max_q,
                       topk_out=topk_out, q_out=q_out, w_out=w_out)

    out = None
    for r in range(n_rep):          # eager warm-up: lazy driver state, kernel attributes
        out = step(d, r)
    torch.cuda.synchronize()
    row_ends = out.row_ends.cpu().numpy()
    ab = algorithmic_bytes(wl, row_ends)

    # One CUDA graph per replica with the library's events around the scoring
    # kernel (the roofline timing of that kernel alone).
    kgraphs, kev = [], []
    for r in range(n_rep):
        a, b = dsa.TimingEvent(), dsa.TimingEvent()
        kg = torch.cuda.CUDAGraph()
        dsa.set_score_timing(a, b)
        with torch.cuda.graph(kg):
            step(d, r)
        dsa.set_score_timing(None, None)
        kgraphs.append(kg)
        kev.append((a, b))
    # The timed steps: one CUDA graph holding all K steps (step i reads replica
    # i mod n), so the GPU runs them back to back as a serving loop issues
    # them, with the PDL edges between steps kept.
    timed = torch.cuda.CUDAGraph()
    with torch.cuda.graph(timed):
        for i in range(args.steps):
            step(d, i % n_rep)
    for _ in range(args.warmup):    # W untimed warm-up replays (W x K steps)
        timed.replay()
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_a.record()
    timed.replay()
    t_b.record()
    torch.cuda.synchronize()
    est = max(t_a.elapsed_time(t_b), 1e-3)
    replays = max(1, min(10000, int(-(-TIMED_MS_MIN // est))))
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([replays], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        replays = int(t.item())
        dist.barrier()

    # headline: `replays` replays of exactly K steps each, each bracketed by
    # CUDA events on the stream; the median replay is the K-step time
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        clocks.mark_start()
        for a, b in evs:
            a.record()
            timed.replay()
            b.record()
        torch.cuda.synchronize()
        clocks.mark_end()
        if world > 1:
            dist.barrier()
    clk = clocks.summary()
    rep_ms = sorted(a.elapsed_time(b) for a, b in evs)
    step_ms = statistics.median(rep_ms)

    # the scoring kernel alone, one step per replay, about as long
    n_k = max(args.steps, int(TIMED_MS_MIN // max(est / args.steps, 1e-3)))
    n_k = min(n_k, 20000)
    kernel_ms = 0.0
    for i in range(n_k):
        kgraphs[i % n_rep].replay()
        a, b = kev[i % n_rep]
        kernel_ms += a.elapsed_ms(b)
    kernel_ms /= n_k

    # End to end through the public API from pinned host buffers, every step
    # copying its inputs in and its top-k back: the serving loop's pipeline
    # (StepPipeline: copies of step i +- 1 overlapped with step i's compute,
    # cycling the cache replicas), the graph-captured step replayed one at a
    # time (one GraphedStep per cache replica), and eager calls.
    pinned = {k: v.pin_memory() for k, v in host.items()}
    h_top = torch.empty((wl.num_rows, wl.topk), dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = h_top.numel() * 4
    e2e_steps = max(args.steps, min(2000, int(TIMED_MS_MIN // max(est / args.steps, 1e-3))))

    def timed_e2e(run_step):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(ev):
            a.record()
            run_step(i)
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / e2e_steps

    like = dict(q=host["q"], wv=host["wv"], keys=host["keys"], slots=host["slots"], seq_lens=host["seq"],
                query_lens=host["qlen"])
    res = {"step_ms": step_ms / args.steps, "kernel_ms": kernel_ms, "replays": replays,
           "replay_ms": [rep_ms[0], rep_ms[-1]], "clocks": clk}
    gs0 = GraphedStep(ix, like, max_q)
    h2d_graph, d2h_graph = gs0.staging_bytes, gs0.host_topk.numel() * 4
    del gs0
    if "graphed" in e2e_modes:
        gsteps = []
        for r in range(n_rep):
            ix.cache = caches[r]
            gsteps.append(GraphedStep(ix, like, max_q))      # staging buffers filled from `like`
        res["e2e_graphed_ms"] = timed_e2e(lambda i: gsteps[i % n_rep].replay())
        del gsteps
    pipe = StepPipeline(ix, like, max_q, caches=caches)
    pipe.run(2 * n_rep)                                       # warm-up
    torch.cuda.synchronize()
    p_start, p_end = pipe.run(e2e_steps)
    torch.cuda.synchronize()
    res["e2e_ms"] = p_start.elapsed_time(p_end) / e2e_steps
    del pipe
    if "eager" in e2e_modes:
        def eager_step(i):
            for k in d:
                d[k].copy_(pinned[k], non_blocking=True)
            step(d, i % n_rep)
            h_top.copy_(topk_out, non_blocking=True)
        res["e2e_eager_ms"] = timed_e2e(eager_step)
    res.update(ab=ab, n_rep=n_rep, cache_bytes=cache_bytes, l2=l2, h2d=h2d, d2h=d2h, h2d_graph=h2d_graph,
               d2h_graph=d2h_graph, e2e_steps=e2e_steps, kernel_launches=n_k)
    del kgraphs, timed, caches, ix
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def workload_config(wl, ab, gpus) -> dict:
    """The config object of a workload (the same in both arms)."""
    return {"workload": workload_desc(wl), "rows": wl.num_rows, "requests": wl.R,
            "scored_keys_per_step": ab["scored"], "unique_keys_per_step": ab["keys_unique"],
            "cache_bytes_per_step": ab["cache"], "parallelism": f"replicas x{gpus}"}


def cpu_leg(wl, seconds: float, one_core_seconds: float) -> dict:
    keys, secs, desc = oracle_sample(wl, seconds)
    out = {"value": keys / secs if secs else None, "unit": UNIT,
           "cores": int(os.environ.get("OPENBLAS_NUM_THREADS", 1)), "kind": "oracle",
           "sample": f"{desc}; {secs:.1f} s"}
    one = oracle_one_core(wl, one_core_seconds)
    if one is not None:
        k1, s1, d1 = one
        out["one_core"] = {"value": k1 / s1 if s1 else None, "unit": UNIT, "cores": 1,
                           "sample": f"{d1}; {s1:.1f} s"}
    return out


def workload_record(args, wl, res, world, peaks) -> dict:
    """The JSON object of one measured workload (all ranks' max already taken)."""
    ab = res["ab"]
    step_ms = res["step_ms"]
    kernel_ms = res["kernel_ms"]
    value = whole_job_rate(ab["scored"], 1, world, step_ms)
    achieved = ab["score_kernel"] / (kernel_ms / 1e3) / 1e9
    traffic = ncu_traffic(traffic_key(wl), ab["score_kernel"])
    rec = {
        "value": value, "unit": UNIT, "ms_per_step": step_ms,
        "dtype": "fp4_e2m1" if wl.fmt in FP4_FORMATS else "fp8_e4m3",
        "config": workload_config(wl, ab, args.gpus),
        "cache_gbs": ab["cache"] * world / (step_ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "score_kernel", "kernel_us": kernel_ms * 1e3,
                     "bytes_per_launch": ab["score_kernel"],
                     "peak_source": f"{peaks['source']} HBM copy bandwidth (of measured)",
                     "step_frac": (ab["step"] / (step_ms / 1e3) / 1e9) / peaks["hbm_gbs"],
                     "step_bytes": ab["step"],
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "tensor": tensor_side(ab["scored"], kernel_ms, wl.fmt, peaks)},
        "e2e": {"value": whole_job_rate(ab["scored"], 1, world, res["e2e_ms"]), "unit": UNIT,
                "h2d_bytes_per_step": res["h2d_graph"], "d2h_bytes_per_step": res["d2h_graph"],
                "how": ("StepPipeline: each step copies its inputs in from a pinned staging buffer and its "
                        "top-k back, overlapped with the neighbouring steps' compute on two copy streams; "
                        f"device time from the first copy in to the last copy out over {res['e2e_steps']} steps")},
        "timing": {"l2": (f"inputs larger than L2: {res['n_rep']} replicas of the key cache "
                          f"({res['n_rep'] * res['cache_bytes'] / 1e6:.0f} MB, L2 {res['l2'] / 1e6:.0f} MB) "
                          "used in turn, no flush"),
                   "launch": (f"the K = {args.steps} timed steps captured as one CUDA graph (PDL edges kept); "
                              f"{res['replays']} replays of it, each between CUDA events, median replay reported"),
                   "replay_ms_min_max": res["replay_ms"], "replays": res["replays"],
                   "kernel_launches_timed": res["kernel_launches"]},
        "clocks": res["clocks"],
    }
    if "e2e_graphed_ms" in res:
        rec["e2e_graphed"] = {"value": whole_job_rate(ab["scored"], 1, world, res["e2e_graphed_ms"]), "unit": UNIT,
                              "h2d_bytes_per_step": res["h2d_graph"], "d2h_bytes_per_step": res["d2h_graph"],
                              "how": "GraphedStep replayed one step at a time: copy in, step, copy back, serialised"}
    if "e2e_eager_ms" in res:
        rec["e2e_eager"] = {"value": whole_job_rate(ab["scored"], 1, world, res["e2e_eager_ms"]), "unit": UNIT,
                            "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                            "how": "eager public-API calls per step, the same host copies in the timed region"}
    return rec


def run_ours(args, names, rank, world, local_rank):
    import torch

    from sparse_attention_indexer_score_gb300 import build as _b
    _b.build()
    from synth import make_workload

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    peaks["mma_tflops"] = measure_mma_tflops()
    records = {}
    for i, name in enumerate(names):
        wl = make_workload(name, **({"fmt": args.fmt} if args.fmt else {}))
        modes = ("pipelined", "graphed", "eager") if i == 0 else ("pipelined",)
        res = measure_workload(args, wl, world, local_rank, modes)
        keys = ["step_ms", "kernel_ms", "e2e_ms", "e2e_graphed_ms", "e2e_eager_ms"]
        vals = max_over_ranks([res.get(k, 0.0) for k in keys], dev)
        for k, v in zip(keys, vals):
            if k in res:
                res[k] = v
        if rank == 0:
            rec = workload_record(args, wl, res, world, peaks)
            if not args.no_cpu_baseline:
                rec["cpu_baseline"] = cpu_leg(wl, args.cpu_seconds if i == 0 else args.cpu_seconds / 2,
                                              1.0 if i == 0 else 0.5)
            records[name if not args.fmt else f"{name}/{args.fmt}"] = (rec, res)
    if rank != 0:
        return
    head_name = next(iter(records))
    head, hres = records[head_name]
    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
            "config": head["config"]}
    for k in ("cache_gbs", "roofline", "e2e", "e2e_graphed", "e2e_eager", "timing", "clocks", "cpu_baseline"):
        if k in head:
            line[k] = head[k]
    line["gpu_launches"] = STEP_KERNELS * args.steps * hres["replays"]
    line["mma_peaks_tflops"] = {k: round(v, 1) for k, v in peaks["mma_tflops"].items()}
    if len(records) > 1:
        line["configs"] = {n: r for n, (r, _) in list(records.items())[1:]}
    print(json.dumps(line))


def run_query_norm(args):
    """QueryNorm (q_a RMSNorm) of a batch of 1536-column BF16 rows, both forms:
    HBM-bound (2 B read + 2 B written per element), timed with CUDA events on
    the stream over K launches after W warm-up launches."""
    import torch
    from sparse_attention_indexer_score_gb300 import build as _b
    _b.build()
    from sparse_attention_indexer_score_gb300 import dsa
    dev = torch.device("cuda", 0)
    batch = args.norm_rows
    g = torch.Generator(device="cpu").manual_seed(7)
    x = torch.randn((batch, 1536), generator=g).to(torch.bfloat16).to(dev)
    w = (1 + 0.1 * torch.randn(1536, generator=g)).to(torch.bfloat16).to(dev)
    out = torch.empty_like(x)
    peaks = measured_peaks()
    bytes_per = batch * 1536 * 2 * 2 + 1536 * 2
    lines = {}
    for variant in ("row", "tiled"):
        for _ in range(args.warmup):
            dsa.query_norm(x, w, 1e-6, variant, out)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(args.steps):
            dsa.query_norm(x, w, 1e-6, variant, out)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        gbs = bytes_per / (ms / 1e3) / 1e9
        lines[variant] = {"us": ms * 1e3, "rows_per_s": batch / (ms / 1e3), "achieved_gbs": gbs,
                          "frac": gbs / peaks["hbm_gbs"]}
    best = max(lines, key=lambda v: lines[v]["rows_per_s"])
    print(json.dumps({
        "metric": "query_norm rows/s (q_a RMSNorm, 1536 BF16 columns)", "value": lines[best]["rows_per_s"],
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic", "config": {"workload": f"query_norm {batch} rows x 1536",
                                                         "variants": lines},
        "roofline": {"bound": "hbm", "achieved": lines[best]["achieved_gbs"], "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": lines[best]["frac"], "traffic": None,
                     "bytes_per_launch": bytes_per, "variant": best},
        "gpu_launches": args.steps}))


def run_topk_merge(args):
    """The DCP top-k merge of 64 rows, 8 ranks x 2048 candidates each -> 2048:
    reads 8 B per candidate (score, local position), timed with CUDA events
    over K calls after W warm-up calls."""
    import torch
    from sparse_attention_indexer_score_gb300 import build as _b
    _b.build()
    from sparse_attention_indexer_score_gb300 import dsa
    dev = torch.device("cuda", 0)
    rows, world, k, k_out, inter = 64, 8, 2048, 2048, 64
    g = torch.Generator(device="cpu").manual_seed(9)
    scores = torch.randn((rows, world * k), generator=g).to(dev)
    idx = torch.randint(0, 1 << 16, (rows, world * k), generator=g, dtype=torch.int32).to(dev)
    ws = dsa.new_workspace(dsa.topk_workspace_size(rows, k_out), dev)
    for _ in range(args.warmup):
        dsa.topk_merge(scores, idx, world, k, inter, k_out, rank=0, workspace=ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(args.steps):
        dsa.topk_merge(scores, idx, world, k, inter, k_out, rank=0, workspace=ws)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    cands = rows * world * k
    nbytes = cands * 8 + rows * k_out * 8
    peaks = measured_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "DCP top-k merge candidates/s", "value": cands / (ms / 1e3), "unit": "candidates/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "f32",
        "data": "synthetic", "config": {"workload": f"topk_merge {rows} rows, {world} ranks x {k} -> {k_out}"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "bytes_per_launch": nbytes},
        "gpu_launches": 3 * args.steps}))


DEFAULT_CONFIGS = "spec_verify,fp8_decode,mxfp4_decode,long_mxfp4"


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--configs", default=DEFAULT_CONFIGS,
                   help="comma-separated workloads; the first is the headline, the others get objects "
                        "of their own under 'configs'")
    p.add_argument("--config", default=None, help="one workload alone (same as --configs NAME)")
    p.add_argument("--fmt", default=None, help="override the workloads' cache format (e.g. mxfp4_rg)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--op", choices=["step", "query_norm", "topk_merge", "mma_peak"], default="step",
                   help="step: the decode step (the headline); query_norm: the q_a RMSNorm alone; "
                        "topk_merge: the DCP top-k merge alone; mma_peak: the tensor-core rate probe")
    p.add_argument("--norm-rows", type=int, default=16384)
    args = p.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.op == "query_norm":
        run_query_norm(args)
        return
    if args.op == "topk_merge":
        run_topk_merge(args)
        return
    if args.op == "mma_peak":
        from sparse_attention_indexer_score_gb300 import build as _b
        _b.build()
        r = measure_mma_tflops()
        print(json.dumps({"metric": "dense tcgen05 MMA rate (128 x 128 tiles, operands in shared memory)",
                          "value": r["fp8"], "unit": "TFLOP/s", "n_gpus": 1, "dtype": "fp8_e4m3",
                          "data": "synthetic", "mxf4_tflops": r["mxf4"], "higher_is_better": True}))
        return
    names = [args.config] if args.config else [n for n in args.configs.split(",") if n]
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        if rank == 0:
            from synth import make_workload
            run_reference(args, make_workload(names[0], **({"fmt": args.fmt} if args.fmt else {})))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, names, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
