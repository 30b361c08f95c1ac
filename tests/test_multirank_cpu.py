"""The multi-rank host logic of bench.py on CPU: two ranks over the gloo
backend (no GPU).  The data path has no collective (every rank runs its own
copy of the workload); what is shared across ranks is the timing (a max over
ranks), the whole-job value and, for the reference arm, that rank 0 alone
prints.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    saved = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = saved
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    b = _bench()
    from kimi_delta_attention_05_gb300.workloads import WORKLOADS
    # a rank-dependent local duration: the job takes the slowest rank's
    ms = b.max_over_ranks(10.0 + 5.0 * rank, world)
    inp = b.rank_inputs(WORKLOADS["tiny"], rank)
    q_sum = float(inp["q"].float().sum())
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "q_sum": q_sum,
                   "value": b.whole_job_value(64, world, ms / 100.0)}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_time_max_and_distinct_inputs(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert res[0]["ms"] == res[1]["ms"] == 15.0          # max over ranks, seen by every rank
    assert res[0]["q_sum"] != res[1]["q_sum"]             # each rank draws its own inputs
    assert res[0]["value"] == pytest.approx(64 * 2 / (0.15 * 1e-3))  # tokens of all ranks


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(3.5, 1) == 3.5
    assert b.whole_job_value(1000, 1, 2.0) == pytest.approx(5e5)


def test_reference_arm_under_torchrun_prints_once():
    """--impl reference under a two-rank torchrun: rank 0 times the oracle and
    prints one JSON line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "3", "--warmup", "3", "--cpu-seconds", "0.2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
