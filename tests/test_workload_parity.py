"""Parity on the three large specified workloads, every element of every head.

Each workload runs once on the GPU at its full size, in the launch
configuration the bench times (the forward, then the backward on the
forward's O and LSE).  The fp64 oracle then recomputes every head, a chunk of
whole heads per test, and every element of O, LSE, dQ, dK and dV in the chunk
is compared:

  O    max-abs <= 1e-2 (plus half a bf16 ulp where |O_ref| >= 4)
  LSE  max-abs <= 1e-3
  dQ, dK, dV   max-abs <= 2e-2 * max|grad|

The gradient bound takes max|grad| over the chunk's whole heads.  That is
never looser than the bound over the whole tensor, so a chunk that passes
also passes the per-tensor bound.  The chunks of a workload together cover
all of its heads, so every row that was scaled x10 in the large-logit
workload is compared ("Lab 06 - Attention kernels", section "Tests": the
kernels are checked against the naive reference; "Triton FlashAttention-2
forward", section "Accuracy check").
"""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import WORKLOADS, big_rows, to_f64, workload_inputs
from tests.tolerances import LSE_TOL, grad_bound, o_bound


def _chunks(name, n_chunks):
    w = WORKLOADS[name]
    bh = w.B * w.H
    step = bh // n_chunks
    return [(name, lo, lo + step) for lo in range(0, bh, step)]


# (workload, first head, end head) over flattened b*H + h
CHUNKS = (_chunks("causal_b4h16t2048d64", 2) + _chunks("causal_b2h16t8192d128", 4)
          + _chunks("ragged_b8h32t3000d128", 8))


def test_chunks_cover_every_head_and_every_x10_row():
    # host-only: the chunk list is what makes the comparison complete
    for name in {c[0] for c in CHUNKS}:
        w = WORKLOADS[name]
        heads = sorted(h for c in CHUNKS if c[0] == name for h in range(c[1], c[2]))
        assert heads == list(range(w.B * w.H)), name
        for flat in big_rows(w).tolist():
            assert flat // w.T in heads


_cache = {}


def _gpu_outputs(name):
    """Inputs and the CUDA path's outputs for workload `name`, on the CPU.
    Only one workload is kept at a time."""
    if name in _cache:
        return _cache[name]
    _cache.clear()
    from online_softmax_05_gb300 import build
    build.build()
    fa.load_library()
    w = WORKLOADS[name]
    causal = w.causal[0]
    q, k, v, do = workload_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=w.scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    out = dict(q=q, k=k, v=v, do=do, o=o.cpu(), lse=lse.cpu(), dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu())
    del qd, kd, vd, dod, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    _cache[name] = out
    return out


def _heads(t, w, lo, hi):
    """Heads lo..hi-1 of a (B, H, T, ...) tensor, flattened to (hi - lo, T, ...)."""
    return t.reshape(w.B * w.H, *t.shape[2:])[lo:hi]


@pytest.mark.gpu
@pytest.mark.slow
@pytest.mark.parametrize("name,lo,hi", CHUNKS, ids=[f"{n}-heads{lo}to{hi - 1}" for n, lo, hi in CHUNKS])
def test_workload_every_element(name, lo, hi):
    w = WORKLOADS[name]
    causal = w.causal[0]
    g = _gpu_outputs(name)
    q, k, v, do = (to_f64(_heads(g[x], w, lo, hi)) for x in ("q", "k", "v", "do"))

    # forward: O and LSE of every row
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.scale, causal)
    o = to_f64(_heads(g["o"], w, lo, hi))
    lse = _heads(g["lse"], w, lo, hi).double().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    o_excess = np.abs(o - o_ref) - o_bound(o_ref)
    worst = np.unravel_index(np.argmax(o_excess), o_excess.shape)
    assert o_excess.max() <= 0, f"O: head {lo + worst[0]} row {worst[1]} col {worst[2]} " \
                                f"err {abs(o[worst] - o_ref[worst]):.4g} ref {o_ref[worst]:.4g}"
    lse_err = np.abs(lse - lse_ref)
    assert lse_err.max() <= LSE_TOL, f"LSE: max err {lse_err.max():.4g} at head {lo + lse_err.argmax() // w.T}"
    del o, o_ref, lse, lse_ref

    # backward: every element of dQ, dK, dV
    rq, rk, rv, _ = oracle.attn_bwd(q, k, v, do, w.scale, causal)
    for gname, ref in (("dq", rq), ("dk", rk), ("dv", rv)):
        got = to_f64(_heads(g[gname], w, lo, hi))
        assert np.isfinite(got).all(), gname
        err = np.abs(got - ref)
        bound = grad_bound(ref)
        where = np.unravel_index(np.argmax(err), err.shape)
        assert err.max() <= bound, f"{gname}: max err {err.max():.4g} > {bound:.4g} at head {lo + where[0]} " \
                                   f"row {where[1]}"
