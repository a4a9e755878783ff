"""Multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank takes its own batch of a workload (independent heads: no collective
in the data path); the ranks exchange only the slowest step time, and the
whole-job rate is world x per-rank units / that time.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from weight_recurrence_gb300 import inputs, ranks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, ws = ranks.world_from_env()
        w = inputs.WORKLOADS["causal_tiny_f32"]
        q, k, v = inputs.workload_inputs(w, r)
        # step "times" that differ by rank: the reduction must return the slowest
        t_local = 1.0 + 0.5 * r
        t_max = ranks.reduce_max(t_local, dist, "cpu")
        # every rank's batch reaches rank 0 only for the test's comparison
        gathered = [torch.empty_like(q) for _ in range(world)]
        dist.all_gather(gathered, q)
        if r == 0:
            res = {"rank_env": [r, lr, ws], "t_max": t_max,
                   "distinct": bool(not torch.equal(gathered[0], gathered[1])),
                   "rank1_matches_seed": bool(torch.equal(gathered[1], inputs.workload_inputs(w, 1)[0])),
                   "rate": ranks.whole_job_rate(w.B * w.N, ws, t_max)}
            with open(os.path.join(outdir, "res.json"), "w") as f:
                json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = json.loads((tmp_path / "res.json").read_text())
    assert res["rank_env"] == [0, 0, 2]
    assert res["t_max"] == 1.5
    assert res["distinct"] and res["rank1_matches_seed"]
    w = inputs.WORKLOADS["causal_tiny_f32"]
    assert res["rate"] == pytest.approx(2 * w.B * w.N / 1.5)


def test_single_process_helpers():
    assert ranks.reduce_max(3.25) == 3.25
    assert ranks.whole_job_rate(100, 4, 0.5) == 800.0
    with pytest.raises(ValueError):
        ranks.whole_job_rate(100, 0, 1.0)
    with pytest.raises(ValueError):
        inputs.rank_seed(1, -1)
    assert inputs.rank_seed(5, 0) == 5
    a = inputs.workload_inputs(inputs.WORKLOADS["causal_tiny_f32"], 0)[0]
    b = inputs.qkv(1, 1, 64, 16, 16, torch.float32, 1.0, 1001)[0]
    assert torch.equal(a, b)


def test_reference_arm_under_torchrun(tmp_path):
    """bench.py --impl reference with two CPU ranks: rank 0 prints one line, rank 1 exits 0."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["cpu_baseline"]["kind"] == "oracle"
