"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests.  It holds no attention arithmetic: it only draws and rounds inputs.

Recipe (the same for every workload, seed 0 unless stated):
  * torch.manual_seed(seed) on the CPU generator, then fp32 ``randn`` draws
    of shape (B, H, T, D) in the order Q, K, V, dO;
  * Q and K are multiplied by ``qk_std`` (4 for the large-logit workload);
  * then ``round(big_row_frac * B*H*T)`` (b, h, t) rows of Q, chosen by a
    ``randperm`` drawn next, are multiplied by ``big_row_mult`` (x10);
  * everything is rounded to bf16 (round-to-nearest-even) last.  The GPU and
    the oracle consume the identical bf16 bits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    D: int
    causal: tuple = (False,)
    bwd: bool = True
    qk_std: float = 1.0
    big_row_frac: float = 0.0
    big_row_mult: float = 1.0
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The five synthetic workloads the path is specified on.
WORKLOADS = {
    "tiny_b1h2t128d64": Workload("tiny_b1h2t128d64", 1, 2, 128, 64, causal=(False, True), bwd=True,
                                 note="tiny reference case, both masks, fwd+bwd"),
    "fwd_b1h8t1024d64": Workload("fwd_b1h8t1024d64", 1, 8, 1024, 64, causal=(False,), bwd=False,
                                 note="non-causal forward + LSE, latency/HBM bound"),
    "causal_b4h16t2048d64": Workload("causal_b4h16t2048d64", 4, 16, 2048, 64, causal=(True,), bwd=True,
                                     note="causal fwd+bwd, D=64"),
    "causal_b2h16t8192d128": Workload("causal_b2h16t8192d128", 2, 16, 8192, 128, causal=(True,), bwd=True,
                                      note="long-context causal fwd+bwd, D=128 (throughput target)"),
    "ragged_b8h32t3000d128": Workload("ragged_b8h32t3000d128", 8, 32, 3000, 128, causal=(False,), bwd=True,
                                      qk_std=4.0, big_row_frac=0.01, big_row_mult=10.0,
                                      note="T not a tile multiple, large logits, 1% of Q rows x10"),
}


def make_inputs(B: int, H: int, T: int, D: int, seed: int = 0, qk_std: float = 1.0,
                big_row_frac: float = 0.0, big_row_mult: float = 1.0):
    """Return bf16 CPU tensors (q, k, v, do), each contiguous (B, H, T, D)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, T, D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if qk_std != 1.0:
        q.mul_(qk_std)
        k.mul_(qk_std)
    n_big = int(round(big_row_frac * B * H * T))
    if n_big > 0:
        idx = torch.randperm(B * H * T, generator=g)[:n_big]
        q.view(-1, D)[idx] *= big_row_mult
    return tuple(t.to(torch.bfloat16).contiguous() for t in (q, k, v, do))


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.H, w.T, w.D, seed=w.seed, qk_std=w.qk_std,
                       big_row_frac=w.big_row_frac, big_row_mult=w.big_row_mult)


def big_rows(w: Workload):
    """Flat (b*H*T + h*T + t) indices of the rows of Q that were scaled up."""
    n_big = int(round(w.big_row_frac * w.B * w.H * w.T))
    if n_big == 0:
        return torch.empty(0, dtype=torch.int64)
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.T, w.D)
    for _ in range(4):
        torch.randn(shape, generator=g, dtype=torch.float32)
    return torch.randperm(w.B * w.H * w.T, generator=g)[:n_big]


def to_f64(t: torch.Tensor):
    """bf16 (or any) CPU tensor -> float64 numpy array holding the same values."""
    return t.detach().to("cpu").to(torch.float64).numpy()
