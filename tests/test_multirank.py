"""The N > 1 host path of bench.py on the CPU: every rank runs its own replica
(own seeded batch, no collective on the data path), times are reduced to the
maximum over ranks with one all-reduce, rank 0 alone reports.  Run as world
size 2 over the gloo backend (127.0.0.1); the GPU arm's NCCL group uses the
same helpers."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from online_softmax_05_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank-specific step times: the reduction must hand every rank the maximum
        vals = [1.0 + rank, 5.0 - 2 * rank, 0.25 * (rank + 1)]
        got = bench.reduce_over_ranks(vals, dist, "cpu")
        w = WORKLOADS["tiny_b1h2t128d64"]
        q = make_inputs(w.B, w.H, w.T, w.D, seed=bench.rank_seed(w, rank))[0]
        out[rank] = {"max": got, "q_sum": float(q.float().sum())}
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_and_replica_seeds_gloo_world_2():
    port = free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_ranks, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    r0, r1 = out[0], out[1]
    assert r0["max"] == r1["max"] == [2.0, 5.0, 0.5]
    # each rank's batch is its own, and rank 0's is the single-GPU batch
    w = WORKLOADS["tiny_b1h2t128d64"]
    q0 = make_inputs(w.B, w.H, w.T, w.D, seed=w.seed)[0]
    assert r0["q_sum"] == float(q0.float().sum())
    assert r0["q_sum"] != r1["q_sum"]


def test_single_rank_helpers_without_a_group():
    assert bench.reduce_over_ranks([3, 1.5]) == [3.0, 1.5]
    # whole-job throughput: N ranks, each one step of F FLOPs in ms milliseconds
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)
    assert bench.job_tflops(4, 2e12, 1000.0) == pytest.approx(8.0)
    w = WORKLOADS["causal_b2h16t8192d128"]
    assert bench.rank_seed(w, 0) == w.seed and bench.rank_seed(w, 3) == w.seed + 3


def test_reference_arm_under_two_ranks_prints_one_line():
    # torchrun with 2 ranks: rank 0 times the CPU oracle, rank 1 exits at once
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_b1h2t128d64"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
