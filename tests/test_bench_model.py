"""The bench's counting model and its measurement bookkeeping, on the host.

FLOPs follow the pages' count ("Triton FlashAttention-2 forward",
`attention_flops`: 4·B·H·T²·D, halved under causal masking; backward 2.5×),
bytes the pages' algorithmic model (`attention_bytes`: every tensor once).
The figures for the long-context causal workload are the ones the scope
table states (549.76 GFLOP forward, ~269.5 MB)."""
import json
import os

import pytest

import bench
from online_softmax_05_gb300.inputs import WORKLOADS


def test_flops_of_the_long_context_workload():
    w = WORKLOADS["causal_b2h16t8192d128"]
    fwd, bwd = bench.workload_flops(w, True)
    assert fwd == 4 * 2 * 16 * 8192 ** 2 * 128 / 2 == pytest.approx(549.76e9, rel=1e-4)
    assert bwd == 2.5 * fwd
    fwd_nc, _ = bench.workload_flops(w, False)
    assert fwd_nc == 2 * fwd


def test_algorithmic_bytes():
    # forward: Q, K, V read and O written in bf16, LSE in fp32
    B, H, T, D = 2, 16, 8192, 128
    assert bench.algorithmic_bytes(B, H, T, D, False) == 2 * B * H * D * (T + 2 * T + T) + 4 * B * H * T
    assert bench.algorithmic_bytes(B, H, T, D, False) == pytest.approx(269.5e6, rel=1e-3)
    # backward: 8 bf16 tensors, LSE read, and the two fp32 row vectors written and read
    assert bench.algorithmic_bytes(B, H, T, D, True) == 2 * 8 * B * H * T * D + 4 * B * H * T * 5


def test_job_throughput_counts_every_rank():
    assert bench.job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
    assert bench.job_tflops(4, 1e12, 1000.0) == pytest.approx(4.0)


def test_code_only_ignores_comments_and_layout():
    a = "int f(int x) {  // doubles x\n  return 2 * x; /* no overflow check */\n}\n"
    b = "int f(int x) {\n    return 2 * x;\n}  // edited comment\n"
    c = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)


def test_traffic_records_are_used_only_for_the_code_they_were_taken_on():
    # a record is reported while the kernel's code (comments aside) is the one
    # the counters were taken on, and is null otherwise
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    seen = 0
    for kernel, by_workload in records.items():
        for workload, rec in by_workload.items():
            assert rec["workload"] == workload
            assert rec["dram_bytes_per_launch"] == pytest.approx(rec["dram_read"] + rec["dram_write"])
            current = rec["source_sha256"] == bench.source_hash(kernel)
            assert bench.recorded_traffic(kernel, workload) == (rec["dram_bytes_per_launch"] if current else None)
            seen += 1
    assert seen >= 4
    assert bench.recorded_traffic("fa_fwd_kernel", "no_such_workload") is None
