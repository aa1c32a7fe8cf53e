"""The multi-rank plumbing of bench.py, on CPU with the gloo backend: the
max-over-ranks timing, the whole-job rate, and the reference arm under
torchrun (rank 0 alone prints its line)."""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 1 + r, 10 - r, r / 2 milliseconds on the three timers
        q.put((rank, bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [2.0, 10.0, 0.5]


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]


def test_whole_job_rate_counts_every_rank():
    # 1000 keys per step per rank, 10 steps, 2 ranks, 5 ms for the slowest rank
    assert bench.whole_job_rate(1000, 10, 2, 5.0) == 1000 * 10 * 2 / 0.005
    assert bench.whole_job_rate(1000, 10, 1, 5.0) * 2 == bench.whole_job_rate(1000, 10, 2, 5.0)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--config", "tiny_fp8", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [line for line in out.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_one_core_oracle_sample_runs_in_a_child():
    """The CPU baseline's one-core figure: the oracle sample in a child process
    holding one BLAS thread scores every key of a small workload."""
    from synth import make_workload
    wl = make_workload("tiny_fp8")
    keys, secs, desc = bench.oracle_one_core(wl, 1.0)
    assert keys == int(wl.seq_lens.sum()) and secs > 0
    assert desc.startswith(f"{wl.R} of {wl.R} requests")


def test_tensor_side_of_the_roofline():
    """8192 FLOPs per scored key (32 heads x 128 columns x multiply-add) over
    the kernel time, against bf16's rate times the operand type's ratio."""
    t = bench.tensor_side(1000, 1.0, "fp8", {"bf16_tflops": 1000.0, "source": "measured"})
    assert t["flops_per_launch"] == 8_192_000
    assert abs(t["achieved"] - 8.192e-3) < 1e-12 and t["peak"] == 2000.0
    assert abs(t["frac"] - 8.192e-3 / 2000.0) < 1e-15
    assert bench.tensor_side(1, 1.0, "mxfp4_rg", {"bf16_tflops": 1.0, "source": "x"})["peak"] == 6.0


def test_traffic_record_matches_the_scoring_source_and_scales_per_unit():
    """The committed ncu traffic of the scoring kernel applies only to the
    source it was taken on (a hash of the kernel's files) and scales with the
    algorithmic bytes of the launch."""
    import json
    rec = json.load(open(os.path.join(ROOT, "profiles", "score_kernel_traffic.json")))
    e = rec["fp8_decode"]
    if e["source_hash"] == bench.score_source_hash():
        assert bench.ncu_traffic("fp8_decode", e["units"]) == e["dram_bytes"]
        assert bench.ncu_traffic("fp8_decode", 2 * e["units"]) == 2 * e["dram_bytes"]
    else:   # the kernel changed since the capture: no traffic is reported
        assert bench.ncu_traffic("fp8_decode", e["units"]) is None
    assert bench.ncu_traffic("no_such_workload", 1) is None
    # every recorded workload: traffic within 10 % above its algorithmic bytes
    for name, v in rec.items():
        assert 1.0 <= v["dram_bytes"] / v["units"] < 1.1, name


def test_traffic_key_names_format_overrides():
    from synth import make_workload
    assert bench.traffic_key(make_workload("long_mxfp4")) == "long_mxfp4"
    assert bench.traffic_key(make_workload("long_mxfp4", fmt="mxfp4_rg")) == "long_mxfp4/mxfp4_rg"
