#!/usr/bin/env python3
"""Throughput of the exact-attention hot path on GB300.

One step = fa_fwd + fa_bwd (the whole path: forward with LSE, backward
preprocess, the dK/dV kernel with key tiles outer and the dQ kernel with
query tiles outer) over one batch of the
long-context causal workload B=2, H=16, T=8192, D=128 (bf16, seeded
synthetic inputs resident in HBM).  FLOPs are counted as the pages count
them: forward 4*B*H*T^2*D, halved under causal masking; backward 2.5x the
forward.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
  python bench.py --configs | --sweep | --gqa | --varlen | --decode   (one line per case)

N > 1 runs under torch.distributed.run: every rank processes its own
independent batch (replicas, no collective on the data path); the barrier and
max-over-ranks timing use NCCL.  Rank 0 prints ONE JSON line.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload, with the same metric and unit.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd & fwd+bwd (bf16, 1×GB300) and % of dense BF16 peak"
DEFAULT_WORKLOAD = "causal_b2h16t8192d128"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
DATASHEET_BF16_TFLOPS = 2250.0  # vendor dense bf16 figure per GPU, reported beside the measured peaks only
CLOCK_FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["online_softmax_05_gb300/csrc/fa_fwd.cu"],
    "fa_bwd_dkdv_kernel": ["online_softmax_05_gb300/csrc/fa_bwd.cu"],
    "fa_bwd_dq_kernel": ["online_softmax_05_gb300/csrc/fa_bwd.cu"],
    "fa_bwd_dq_convert_kernel": ["online_softmax_05_gb300/csrc/fa_bwd.cu"],
}
COMMON_SOURCES = ["online_softmax_05_gb300/csrc/fa_ptx.cuh", "online_softmax_05_gb300/csrc/fa_sched.h",
                  "online_softmax_05_gb300/csrc/fa_tmap.h"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--decode", action="store_true",
                    help="split-K decoding: B=8 H=32, 1 query row against 32768 keys, D=128 (HBM-bound)")
    ap.add_argument("--gqa", action="store_true",
                    help="grouped-query attention: B=2 Hq=16 Hkv=4 T=8192 D=128 causal, fwd and bwd TFLOP/s")
    ap.add_argument("--varlen", action="store_true",
                    help="packed variable-length forward and backward: 48 causal requests of 128..8192 tokens, H=16, D=128, "
                         "against the same batch padded to the longest request")
    ap.add_argument("--configs", action="store_true",
                    help="every specified workload (fwd, bwd; the small forward also with a cold L2): one JSON line per case")
    ap.add_argument("--only", default=None, help="with --configs: run this workload only")
    ap.add_argument("--sweep", action="store_true",
                    help="T sweep (512..8192 at 16384 tokens x 16 heads): one JSON line per case, not the bench line")
    return ap.parse_args()


def rank_seed(w, rank):
    """Each rank draws its own batch (replicas: no collective on the data path);
    rank 0's batch is the single-GPU one."""
    return w.seed + rank


def reduce_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum over ranks (the slowest rank sets every time), or
    the values unchanged without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tflops(world, step_flops, ms):
    """Whole-job throughput: every rank processes one step's worth of units in
    ms milliseconds (the maximum over ranks)."""
    return world * step_flops / (ms * 1e-3) / 1e12


def workload_flops(w, causal):
    fwd = 4.0 * w.B * w.H * w.T * w.T * w.D / (2.0 if causal else 1.0)
    return fwd, 2.5 * fwd


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def code_only(text):
    """Source text without comments and with whitespace collapsed: what the
    compiler sees, so that a comment edit does not void a measurement."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return " ".join(text.split())


def source_hash(kernel):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel] + COMMON_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel][workload]
    except Exception:
        return None
    if d.get("source_sha256") != source_hash(kernel) or d.get("workload") != workload:
        return None
    return float(d["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 25 ms).  The
    caller marks the timed region with mark(); the summary keeps the samples
    taken inside it (all samples if none fell inside)."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None
        self.marks = []

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "25", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def mark(self):
        """Host wall-clock time (local, as nvidia-smi stamps its samples)."""
        self.marks.append(datetime.datetime.now())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def parse(lines, uuid=None, window=None):
        """Rows of the sampler's CSV as a summary; window = (start, end) datetimes."""
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if uuid and uuid not in parts[1]:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None
            rows.append((ts, parts))
        inside = [r for ts, r in rows if window and ts is not None and window[0] <= ts <= window[1]]
        use = inside if inside else [r for _, r in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "in_timed_region": 0}
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = [float(r[2]) for r in use if num(r[2])]
        smax = [float(r[3]) for r in use if num(r[3])]
        power = [float(r[4]) for r in use if num(r[4])]
        reasons = sorted({name for r in use for name, v in zip(REASON_NAMES, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use), "in_timed_region": len(inside),
                "power_w_max": max(power) if power else None,
                "power_w_median": statistics.median(power) if power else None}

    def summary(self):
        lines = []
        try:
            with open(self.path) as f:
                lines = f.readlines()
            os.unlink(self.path)
        except Exception:
            pass
        window = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else None
        return self.parse(lines, self.uuid, window)


_INPUT_CACHE = {}


def time_oracle_heads(w, heads, causal, T=None):
    """Run the fp64 oracle forward + backward on the given (b, h) heads
    (optionally the first T tokens of each); returns (seconds, flops, threads)."""
    import oracle
    from online_softmax_05_gb300.inputs import to_f64, workload_inputs
    oracle.build()
    if _INPUT_CACHE.get("name") != w.name:
        _INPUT_CACHE.clear()
        _INPUT_CACHE.update(name=w.name, tensors=workload_inputs(w))
    q, k, v, do = _INPUT_CACHE["tensors"]
    T = T or w.T
    arrays = [tuple(to_f64(t[b, h, :T]) for t in (q, k, v, do)) for b, h in heads]
    t0 = time.perf_counter()
    for qf, kf, vf, df in arrays:
        oracle.attn_fwd(qf[None], kf[None], vf[None], w.scale, causal)
        oracle.attn_bwd(qf[None], kf[None], vf[None], df[None], w.scale, causal)
    sec = time.perf_counter() - t0
    fwd = 4.0 * T * T * w.D / (2.0 if causal else 1.0)
    return sec, 3.5 * fwd * len(heads), oracle.num_threads()


def run_reference(args, w, causal, rank, world):
    """Reference arm: the CPU oracle as it stands, bounded sample per step."""
    if rank != 0:
        return
    # one head per step at full T costs ~5-10 s on 16 cores; shrink the causal
    # prefix if the whole run would take more than about three minutes
    n = args.steps + args.warmup
    T_s = w.T
    if n * 6.0 > 180.0:
        T_s = max(256, int(w.T * math.sqrt(180.0 / (n * 6.0))) // 128 * 128)
    BH = w.B * w.H
    total_s, total_f, threads = 0.0, 0.0, 1
    for s in range(n):
        bh = s % BH
        sec, fl, threads = time_oracle_heads(w, [divmod(bh, w.H)], causal, T_s)
        if s >= args.warmup:
            total_s += sec
            total_f += fl
    value = total_f / total_s / 1e12
    sample = (f"per step one (b,h) head of {w.name} (round-robin over heads), "
              + ("full T" if T_s == w.T else f"first {T_s} tokens (causal prefix)")
              + ", fp64 oracle forward + backward (naive, materialises S and P)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "D": w.D, "causal": causal,
                       "passes": "fwd+bwd"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def algorithmic_bytes(B, H, T, D, bwd):
    """Bytes the pass must move at least: each tensor read or written once.
    Forward: read Q, K, V; write O (bf16) and LSE (fp32).  Backward: read Q,
    K, V, O, dO, LSE; write dQ, dK, dV; plus the fp32 per-row workspace (D
    and the log2-scaled LSE, each written once and read once)."""
    n = B * H * T * D
    if not bwd:
        return 2 * 4 * n + 4 * B * H * T
    return 2 * 8 * n + 4 * B * H * T + 4 * 4 * B * H * T


def run_configs(args):
    """Every specified workload, forward and (where specified) backward: median
    over at least 20 launches after 5 warm-ups, each between its own pair of
    events (`ms`), and the mean over the same number of launches between one
    pair of events (`ms_back_to_back`; the launches' fixed GPU-side costs then
    overlap).  The small non-causal forward (B=1 H=8 T=1024 D=64) is also
    timed with a 256 MB write between launches, so it starts with a cold L2.
    One JSON line per case, then one with the event-pair time of a one-element
    torch kernel: the floor of the per-launch method on this GPU."""
    import torch
    import online_softmax_05_gb300 as fa
    from online_softmax_05_gb300.inputs import WORKLOADS, workload_inputs
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, src = load_peaks()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    n_iter = max(20, min(args.steps, 100))
    for name, w in WORKLOADS.items():
        if args.only and name != args.only:
            continue
        q, k, v, do = (t.to(dev) for t in workload_inputs(w))
        B, H, T, D, sc = w.B, w.H, w.T, w.D, w.scale
        o = torch.empty_like(q)
        lse = torch.empty(B, H, T, device=dev)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        for causal in w.causal:
            f = lambda: fa.fa_fwd(q, k, v, o, lse, B, H, T, D, sc, int(causal), stream)
            b = lambda: fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, T, D, sc, int(causal), stream)
            passes = [("fwd", f, False)] + ([("bwd", b, False)] if w.bwd else [])
            if name == "fwd_b1h8t1024d64":
                passes.append(("fwd", f, True))
            fwd_fl = 4.0 * B * H * T * T * D / (2 if causal else 1)
            for pname, fn, flush in passes:
                for _ in range(max(5, args.warmup)):
                    assert fn() == 0
                torch.cuda.synchronize(dev)
                # all launches enqueued back to back with an event pair around each:
                # host-side launch work is hidden, each pair times one launch on the GPU
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(n_iter)]
                for e0, e1 in evs:
                    if flush:
                        flush_buf.fill_(1)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                torch.cuda.synchronize(dev)
                times = [e0.elapsed_time(e1) for e0, e1 in evs]
                assert fa.fa_get_device_status(stream) == 0
                ms = sorted(times)[len(times) // 2]
                ms_b2b = None
                if not flush:
                    e0, e1 = evs[0]
                    e0.record(stream)
                    for _ in range(n_iter):
                        fn()
                    e1.record(stream)
                    torch.cuda.synchronize(dev)
                    ms_b2b = e0.elapsed_time(e1) / n_iter
                bwd = pname == "bwd"
                fl = fwd_fl * (2.5 if bwd else 1.0)
                nbytes = algorithmic_bytes(B, H, T, D, bwd)
                line = {"config": name, "pass": pname, "causal": bool(causal), "l2": "flushed" if flush else "warm",
                        "B": B, "H": H, "T": T, "D": D, "ms": ms, "tflops": fl / ms / 1e9,
                        "frac_of_burst": fl / ms / 1e9 / peaks["bf16_tflops"], "gbs": nbytes / ms / 1e6,
                        "frac_of_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"], "iters": n_iter,
                        "ms_back_to_back": ms_b2b, "peaks": src, "dtype": "bf16", "data": "synthetic"}
                if bwd:
                    # the backward's two main kernels, timed apart in a pass of their own
                    # (events between them serialise the grids, which otherwise overlap)
                    lib = fa.load_library()
                    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_iter)]
                    for e3 in kev:  # torch times only events it has recorded once itself
                        for e in e3:
                            e.record(stream)
                    for e3 in kev:
                        lib.fa_set_timing_events(None, None, *(e.cuda_event for e in e3))
                        fn()
                    lib.fa_set_timing_events(None, None, None, None, None)
                    torch.cuda.synchronize(dev)
                    med = lambda xs: sorted(xs)[len(xs) // 2]
                    line["dkdv_ms"] = med([e[0].elapsed_time(e[1]) for e in kev])
                    line["dq_ms"] = med([e[1].elapsed_time(e[2]) for e in kev])
                print(json.dumps(line), flush=True)
    # the per-launch method's own floor: a one-element torch kernel between an event pair
    x = torch.zeros(1, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iter)]
    for e0, e1 in evs:
        e0.record(stream)
        x.add_(1)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    floor = sorted(e0.elapsed_time(e1) for e0, e1 in evs)[n_iter // 2]
    print(json.dumps({"harness": "event pair around one one-element torch kernel", "ms": floor}), flush=True)


def run_sweep(args):
    """T sweep of the forward and the backward (the short-T, memory/latency-bound
    end against the long-T compute-bound end), 16384 tokens x 16 heads per case."""
    import torch
    import online_softmax_05_gb300 as fa
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, src = load_peaks()
    for D in (64, 128):
        for causal in (0, 1):
            for T in (512, 1024, 2048, 4096, 8192):
                B, H = 16384 // T, 16
                g = torch.Generator(device="cpu").manual_seed(T + D)
                q, k, v, do = (torch.randn(B, H, T, D, generator=g).to(torch.bfloat16).to(dev) for _ in range(4))
                o = torch.empty_like(q)
                lse = torch.empty(B, H, T, device=dev)
                dq, dk, dv = (torch.empty_like(q) for _ in range(3))
                sc = D ** -0.5
                f = lambda: fa.fa_fwd(q, k, v, o, lse, B, H, T, D, sc, causal, stream)
                b = lambda: fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, T, D, sc, causal, stream)
                res = {}
                for name, fn in (("fwd", f), ("bwd", b)):
                    for _ in range(max(3, args.warmup)):
                        assert fn() == 0
                    torch.cuda.synchronize(dev)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    n = max(10, min(args.steps, 50))
                    e0.record(stream)
                    for _ in range(n):
                        fn()
                    e1.record(stream)
                    torch.cuda.synchronize(dev)
                    res[name] = e0.elapsed_time(e1) / n
                assert fa.fa_get_device_status(stream) == 0
                fwd_fl = 4.0 * B * H * T * T * D / (2 if causal else 1)
                line = {"sweep": "T", "B": B, "H": H, "T": T, "D": D, "causal": bool(causal),
                        "fwd_ms": res["fwd"], "bwd_ms": res["bwd"],
                        "fwd_tflops": fwd_fl / res["fwd"] / 1e9, "bwd_tflops": 2.5 * fwd_fl / res["bwd"] / 1e9,
                        "fwd_gbs": algorithmic_bytes(B, H, T, D, False) / res["fwd"] / 1e6,
                        "bwd_gbs": algorithmic_bytes(B, H, T, D, True) / res["bwd"] / 1e6,
                        "peak_tflops": peaks["bf16_tflops"], "peak_gbs": peaks["hbm_gbs"], "peaks": src}
                print(json.dumps(line), flush=True)


def run_decode(args, B=8, H=32, Tq=1, Tk=32768, D=128):
    """fa_decode throughput: one JSON line with GB/s against the measured HBM copy rate."""
    import torch
    import online_softmax_05_gb300 as fa
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device="cpu").manual_seed(0)
    q = torch.randn(B, H, Tq, D, generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn(B, H, Tk, D, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(B, H, Tk, D, generator=g).to(torch.bfloat16).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Tq, device=dev)
    sc = D ** -0.5
    for _ in range(max(3, args.warmup)):
        assert fa.fa_decode(q, k, v, o, lse, B, H, Tq, Tk, D, sc, stream) == 0
    torch.cuda.synchronize(dev)
    n = max(10, min(args.steps, 100))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fa.fa_decode(q, k, v, o, lse, B, H, Tq, Tk, D, sc, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    assert fa.fa_get_device_status(stream) == 0
    ms = e0.elapsed_time(e1) / n
    nbytes = 2 * (2 * B * H * Tq * D + 2 * B * H * Tk * D) + 4 * B * H * Tq
    peaks, src = load_peaks()
    gbs = nbytes / ms / 1e6
    print(json.dumps({"metric": "split-K decoding GB/s (K/V streamed once)", "value": gbs, "unit": "GB/s",
                      "ms_per_call": ms, "calls": n, "tflops": 4.0 * B * H * Tq * Tk * D / ms / 1e9,
                      "config": {"workload": f"decode_b{B}h{H}q{Tq}k{Tk}d{D}", "B": B, "H": H, "Tq": Tq, "Tk": Tk,
                                 "D": D, "l2": "no flush: K/V %.1f GB > 129 MB L2" % (nbytes / 1e9)},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": gbs / peaks["hbm_gbs"], "peak_kind": f"copy bandwidth, of {src}"},
                      "dtype": "bf16", "data": "synthetic"}), flush=True)


def run_gqa(args, B=2, Hq=16, Hkv=4, T=8192, D=128, causal=1):
    """fa_fwd_gqa / fa_bwd_gqa throughput on the long-context causal shape with 4 query heads per K/V head."""
    import torch
    import online_softmax_05_gb300 as fa
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device="cpu").manual_seed(0)
    q, do = (torch.randn(B, Hq, T, D, generator=g).to(torch.bfloat16).to(dev) for _ in range(2))
    k, v = (torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16).to(dev) for _ in range(2))
    o, dq = torch.empty_like(q), torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty(B, Hq, T, device=dev)
    sc = D ** -0.5
    f = lambda: fa.fa_fwd_gqa(q, k, v, o, lse, B, Hq, Hkv, T, D, sc, causal, stream)
    b = lambda: fa.fa_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, T, D, sc, causal, stream)
    res = {}
    for name, fn in (("fwd", f), ("bwd", b)):
        for _ in range(max(3, args.warmup)):
            assert fn() == 0
        torch.cuda.synchronize(dev)
        n = max(10, min(args.steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = e0.elapsed_time(e1) / n
    assert fa.fa_get_device_status(stream) == 0
    fwd_fl = 4.0 * B * Hq * T * T * D / (2 if causal else 1)
    peaks, src = load_peaks()
    print(json.dumps({"metric": "grouped-query attention TFLOP/s", "value": 3.5 * fwd_fl / (res["fwd"] + res["bwd"]) / 1e9,
                      "unit": "TFLOP/s", "fwd_ms": res["fwd"], "bwd_ms": res["bwd"],
                      "fwd_tflops": fwd_fl / res["fwd"] / 1e9, "bwd_tflops": 2.5 * fwd_fl / res["bwd"] / 1e9,
                      "config": {"workload": f"gqa_b{B}hq{Hq}hkv{Hkv}t{T}d{D}", "causal": bool(causal)},
                      "peak": peaks["bf16_tflops"], "peaks": src, "dtype": "bf16", "data": "synthetic"}), flush=True)


def run_varlen(args, n_seq=48, H=16, D=128, causal=1):
    """fa_fwd_varlen / fa_bwd_varlen throughput on a seeded serving mix, beside fa_fwd / fa_bwd on the padded batch."""
    import numpy as np
    import torch
    import online_softmax_05_gb300 as fa
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    lengths = np.random.default_rng(0).integers(128, 8193, size=n_seq)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    total, Tmax = int(cu[-1]), int(lengths.max())
    g = torch.Generator(device="cpu").manual_seed(0)
    q, k, v, do = (torch.randn(total, H, D, generator=g).to(torch.bfloat16).to(dev) for _ in range(4))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty(H, total, device=dev)
    cud = torch.from_numpy(cu).to(dev)
    gd = torch.Generator(device=dev).manual_seed(1)
    qp, kp, vp, dop = (torch.randn(n_seq, H, Tmax, D, generator=gd, device=dev).to(torch.bfloat16) for _ in range(4))
    op, dqp, dkp, dvp = (torch.empty_like(qp) for _ in range(4))
    lp = torch.empty(n_seq, H, Tmax, device=dev)
    sc = D ** -0.5
    calls = {
        "varlen": lambda: fa.fa_fwd_varlen(q, k, v, o, lse, cud, n_seq, Tmax, total, H, D, sc, causal, stream),
        "padded": lambda: fa.fa_fwd(qp, kp, vp, op, lp, n_seq, H, Tmax, D, sc, causal, stream),
        "varlen_bwd": lambda: fa.fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cud, n_seq, Tmax, total, H, D, sc,
                                               causal, stream),
        "padded_bwd": lambda: fa.fa_bwd(qp, kp, vp, op, dop, lp, dqp, dkp, dvp, n_seq, H, Tmax, D, sc, causal, stream),
    }
    res = {}
    for name, fn in calls.items():   # forwards first: each backward reads its forward's O and LSE
        for _ in range(max(3, args.warmup)):
            assert fn() == 0
        torch.cuda.synchronize(dev)
        n = max(10, min(args.steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = e0.elapsed_time(e1) / n
    assert fa.fa_get_device_status(stream) == 0
    L = lengths.astype(np.float64)
    useful = float(np.sum(4.0 * H * L * L * D / (2 if causal else 1)))
    peaks, src = load_peaks()
    tf = useful / res["varlen"] / 1e9
    both = res["varlen"] + res["varlen_bwd"]
    print(json.dumps({"metric": "packed variable-length forward TFLOP/s (useful work)", "value": tf,
                      "unit": "TFLOP/s", "ms_per_call": res["varlen"], "padded_ms_per_call": res["padded"],
                      "padded_useful_tflops": useful / res["padded"] / 1e9, "speedup_vs_padded": res["padded"] / res["varlen"],
                      "frac_of_burst": tf / peaks["bf16_tflops"],
                      "bwd_ms_per_call": res["varlen_bwd"], "bwd_useful_tflops": 2.5 * useful / res["varlen_bwd"] / 1e9,
                      "padded_bwd_ms_per_call": res["padded_bwd"],
                      "bwd_speedup_vs_padded": res["padded_bwd"] / res["varlen_bwd"],
                      "fwd_bwd_useful_tflops": 3.5 * useful / both / 1e9,
                      "config": {"workload": f"varlen_n{n_seq}h{H}d{D}_len128to8192", "total_tokens": total,
                                 "max_seqlen": Tmax, "causal": bool(causal), "lengths": "uniform 128..8192, seed 0",
                                 "l2": "no flush: Q/K/V %.1f GB > 129 MB L2" % (3 * total * H * D * 2 / 1e9)},
                      "peak": peaks["bf16_tflops"], "peaks": src, "dtype": "bf16", "data": "synthetic"}), flush=True)


def main():
    args = parse_args()
    if args.varlen:
        run_varlen(args)
        return
    if args.gqa:
        run_gqa(args)
        return
    if args.decode:
        run_decode(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.configs:
        run_configs(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from online_softmax_05_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    causal = w.causal[0]

    if args.impl == "reference":
        run_reference(args, w, causal, rank, world)
        return

    import torch
    import online_softmax_05_gb300 as fa
    from online_softmax_05_gb300.inputs import make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lib = fa.load_library()
    stream = torch.cuda.current_stream(dev)

    # seeded inputs, one independent batch per rank, resident in HBM
    q, k, v, do = (t.to(dev) for t in make_inputs(w.B, w.H, w.T, w.D, seed=rank_seed(w, rank), qk_std=w.qk_std,
                                                   big_row_frac=w.big_row_frac, big_row_mult=w.big_row_mult))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.T, device=dev, dtype=torch.float32)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    B, H, T, D, scale = w.B, w.H, w.T, w.D, w.scale

    def step():
        rc = fa.fa_fwd(q, k, v, o, lse, B, H, T, D, scale, int(causal), stream)
        if rc != 0:
            raise fa.FAError(rc, "fa_fwd")
        rc = fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, T, D, scale, int(causal), stream)
        if rc != 0:
            raise fa.FAError(rc, "fa_bwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status(stream) != 0:
        raise RuntimeError("device status reported a stalled kernel during warm-up")

    # Per-step events around the forward kernel and the backward's two main
    # kernels.  They are recorded in a second pass of their own: an event
    # between the dK/dV and dQ launches serialises the two grids, which
    # otherwise overlap (the dQ grid starts in the dK/dV grid's tail).
    K = args.steps
    KS = min(K, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(KS)]
    for e4 in evs:
        for e in e4:
            e.record(stream)
    torch.cuda.synchronize(dev)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    lib.fa_set_timing_events(None, None, None, None, None)
    with ClockSampler(uuid) as clocks:
        clocks.mark()
        t_start.record(stream)
        for s in range(K):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark()
    if dist is not None:
        dist.barrier()
    status = fa.fa_get_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    ms = t_start.elapsed_time(t_end) / K
    # per-kernel pass (kernels serialised by the events between them)
    for s in range(KS):
        lib.fa_set_timing_events(*(e.cuda_event for e in evs[s]))
        step()
    lib.fa_set_timing_events(None, None, None, None, None)
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_status(stream) != 0:
        raise RuntimeError("device status reported a stalled kernel in the per-kernel pass")
    fwd_ms = statistics.mean(evs[s][0].elapsed_time(evs[s][1]) for s in range(KS))
    dkdv_ms = statistics.mean(evs[s][2].elapsed_time(evs[s][3]) for s in range(KS))
    dq_ms = statistics.mean(evs[s][3].elapsed_time(evs[s][4]) for s in range(KS))
    ms, fwd_ms, dkdv_ms, dq_ms = reduce_over_ranks([ms, fwd_ms, dkdv_ms, dq_ms], dist, dev)
    bwd_ms = dkdv_ms + dq_ms

    fwd_fl, bwd_fl = workload_flops(w, causal)
    step_fl = fwd_fl + bwd_fl
    value = job_tflops(world, step_fl, ms)
    fwd_tflops_kernel = fwd_fl / (fwd_ms * 1e-3) / 1e12
    bwd_tflops_kernels = bwd_fl / (bwd_ms * 1e-3) / 1e12
    # Algorithmic FLOPs per backward kernel: of the backward's five products
    # (S, dP, dV, dK, dQ; 2.5x the forward) the dK/dV kernel performs four
    # (2x the forward) and the dQ kernel one (0.5x); the dQ kernel's
    # recomputation of S and dP is extra work and is not counted.  Where the
    # library sums dQ inside the dK/dV kernel (D = 64 on a full grid) that
    # kernel performs all five, and the second kernel only converts the float32
    # dQ accumulator to bf16 (HBM-bound: 4 bytes read, 2 written per element).
    in_place = lib.fa_bwd_sums_dq_in_place(B, H, T, D) == 1
    dkdv_tflops = (2.5 if in_place else 2.0) * fwd_fl / (dkdv_ms * 1e-3) / 1e12
    dq_tflops = 0.5 * fwd_fl / (dq_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak_sus, peak_burst = peaks["bf16_tflops_sustained"], peaks["bf16_tflops"]

    # The per-kernel pass runs KS steps (tens of milliseconds at this size), so
    # the kernels are timed as a burst: the denominator is the measured burst
    # bf16 rate.  The fraction of the seconds-long sustained rate is beside it.
    def roofline(kernel, achieved):
        return {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                "frac": achieved / peak_burst, "peak_kind": f"bf16 dense, burst, of {peak_src}",
                "frac_of_sustained": achieved / peak_sus, "traffic": recorded_traffic(kernel, w.name)}

    if in_place:
        conv_bytes = B * H * T * D * 6
        conv_gbs = conv_bytes / (dq_ms * 1e-3) / 1e9
        second = {"bound": "hbm", "kernel": "fa_bwd_dq_convert_kernel", "achieved": conv_gbs, "peak": peaks["hbm_gbs"],
                  "unit": "GB/s", "frac": conv_gbs / peaks["hbm_gbs"], "peak_kind": f"copy bandwidth, of {peak_src}",
                  "traffic": recorded_traffic("fa_bwd_dq_convert_kernel", w.name)}
    else:
        second = roofline("fa_bwd_dq_kernel", dq_tflops)
    rls = sorted([(fwd_ms, roofline("fa_fwd_kernel", fwd_tflops_kernel)),
                  (dkdv_ms, roofline("fa_bwd_dkdv_kernel", dkdv_tflops)),
                  (dq_ms, second)], key=lambda x: -x[0])

    # End to end through the public API with host buffers (pinned), copies timed.
    # Every step uploads its inputs (Q, K, V, dO) and downloads its results
    # (O, LSE, dQ, dK, dV).  Uploads and downloads run on their own streams
    # into and out of two sets of device buffers, so step k+1's upload and step
    # k-1's download overlap step k's kernels, as a caller of the API would
    # pipeline them.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (t.to("cpu").pin_memory() for t in (q, k, v, do))
        ho, hdq, hdk, hdv = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(4))
        hlse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        # the first upload and the last download are not overlapped with kernels:
        # a run of up to 50 steps spreads that pipeline fill over the steps
        n_e2e = max(3, min(K, 50))
        bufs = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv)]
        bufs.append({name: torch.empty_like(t) for name, t in bufs[0].items()})
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        d2h_done = [torch.cuda.Event() for _ in range(2)]

        def upload(bf):
            with torch.cuda.stream(s_in):
                for name, src in (("q", hq), ("k", hk), ("v", hv), ("do", hdo)):
                    bf[name].copy_(src, non_blocking=True)

        def e2e_run(n):
            upload(bufs[0])
            h2d_done[0].record(s_in)
            for st in range(n):
                b = st % 2
                bf = bufs[b]
                stream.wait_event(h2d_done[b])
                if st >= 2:
                    stream.wait_event(d2h_done[b])  # step st-2's results have left these buffers
                fa.attention_forward(bf["q"], bf["k"], bf["v"], causal=causal, scale=scale, out=bf["o"],
                                     lse=bf["lse"], stream=stream)
                fa.attention_backward(bf["q"], bf["k"], bf["v"], bf["o"], bf["lse"], bf["do"], causal=causal,
                                      scale=scale, dq=bf["dq"], dk=bf["dk"], dv=bf["dv"], stream=stream)
                comp_done[b].record(stream)
                if st + 1 < n:
                    nb = (st + 1) % 2
                    if st >= 1:
                        s_in.wait_event(comp_done[nb])  # step st-1's kernels are done with its inputs
                    upload(bufs[nb])
                    h2d_done[nb].record(s_in)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[b])
                    for dst, name in ((ho, "o"), (hlse, "lse"), (hdq, "dq"), (hdk, "dk"), (hdv, "dv")):
                        dst.copy_(bf[name], non_blocking=True)
                d2h_done[b].record(s_out)
            stream.wait_event(d2h_done[(n - 1) % 2])

        e2e_run(2)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        a.record(stream)
        s_in.wait_event(a)
        s_out.wait_event(a)
        e2e_run(n_e2e)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = reduce_over_ranks([a.elapsed_time(b) / n_e2e], dist, dev)[0]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))
        e2e = {"value": job_tflops(world, step_fl, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms,
               "steps": n_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "copies": "upload and download streams, two device buffer sets, overlapped with the kernels"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads = [(0, h) for h in range(8)]
        sec, fl, threads = time_oracle_heads(w, heads, causal)
        cpu = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"heads (b,h)={heads} of {w.name} at full T, fp64 oracle forward + backward "
                         f"(naive, materialises S and P), {sec:.1f} s; FLOPs counted as for the GPU"}

    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "D": w.D, "causal": causal,
                   "passes": "fwd+bwd", "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush: inputs + outputs + workspace per step ~0.7 GB > 129 MB L2"},
        "fwd_tflops": fwd_tflops_kernel, "fwd_ms": fwd_ms, "bwd_dkdv_ms": dkdv_ms, "bwd_dq_ms": dq_ms,
        "bwd_form": "dQ summed in the dK/dV kernel, then converted" if in_place else "dK/dV kernel, then dQ kernel",
        "bwd_tflops": bwd_tflops_kernels,
        "kernel_times": f"CUDA events around each kernel in a separate pass of {KS} steps after the timed region "
                        "(events between the backward's two grids serialise them; in the timed region the dQ grid "
                        "starts in the dK/dV grid's tail)",
        "pct_of_peak": {"fwd_bwd_of_burst": 100 * value / world / peak_burst,
                        "fwd_bwd_of_sustained": 100 * value / world / peak_sus,
                        "fwd_of_burst": 100 * fwd_tflops_kernel / peak_burst, "peaks": peak_src,
                        "fwd_bwd_of_datasheet": 100 * value / world / DATASHEET_BF16_TFLOPS,
                        "datasheet": f"{DATASHEET_BF16_TFLOPS:.0f} TFLOP/s dense bf16 per GB300 (vendor figure, "
                                     "not measured here)"},
        "roofline": rls[0][1],
        "roofline_other": [r for _, r in rls[1:]],
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 4 * K,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
