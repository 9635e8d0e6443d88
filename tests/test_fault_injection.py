"""Failure detection without a GPU fault: every in-kernel wait is bounded.

A host-side test hook tells one kernel's load warp to skip one tile copy:
  mode 1  the forward's load warp, its first K/V copy (a small grid's split
          items and a full grid's pairs of query tiles);
  mode 2  the first dK/dV CTA of the backward, its third Q copy (at D = 64
          on a full grid that CTA also sums dQ, so reduce-adds are in flight);
  mode 3  the first dQ CTA of the backward, its first K copy.
The waits that need the missing tile run out after a short limit, the CTA
records FA_ERR_DEVICE_TIMEOUT, drains its copies and MMAs in flight, frees
its tensor memory and exits.  The context stays usable: the status word is
cleared by the read, and the next call (on every SM, so also on the SM whose
CTA gave up) runs and matches the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import make_inputs, to_f64
from tests.tolerances import grad_bound, o_ok


@pytest.fixture(scope="module")
def lib():
    from online_softmax_05_gb300 import build
    build.build()
    return fa.load_library()


def _inject(lib, mode, fn):
    """Run fn() with the hook set and a 100 ms wait limit; restore both."""
    assert lib.fa_debug_set_wait_timeout_ns(100_000_000) == 0
    assert lib.fa_debug_inject(mode) == 0
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        lib.fa_debug_inject(0)
        lib.fa_debug_set_wait_timeout_ns(2_000_000_000)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,T", [(1, 2, 300), (4, 16, 1280)], ids=["split_items", "paired_items"])
def test_skipped_copy_reports_timeout_and_recovers(lib, B, H, T):
    # a small grid runs one query tile per item, its key tiles split between the
    # two softmax warpgroups; a full grid runs pairs of query tiles
    D = 64
    q, k, v, _ = make_inputs(B, H, T, D, seed=1)
    dev = torch.device("cuda")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, T, device=dev)
    assert fa.fa_get_device_status() == 0

    def call():
        assert fa.fa_fwd(qd, kd, vd, o, lse, B, H, T, D, 1 / math.sqrt(D), 0, torch.cuda.current_stream()) == 0

    _inject(lib, 1, call)
    assert fa.fa_get_device_status() == -7
    assert fa.fa_get_device_status() == 0   # the status word was cleared
    o2, lse2 = fa.attention_forward(qd, kd, vd, causal=False)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for b, h in ((0, 0), (B - 1, H - 1)):
        o_ref, lse_ref = oracle.attn_fwd(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]), 1 / math.sqrt(D), False)
        assert o_ok(to_f64(o2[b, h].cpu()), o_ref)
        assert np.abs(lse2[b, h].cpu().double().numpy() - lse_ref).max() <= 1e-3


@pytest.mark.gpu
@pytest.mark.parametrize("mode", [2, 3], ids=["dkdv_q_copy", "dq_k_copy"])
@pytest.mark.parametrize("D,causal", [(64, True), (128, False)])
def test_backward_skipped_copy_reports_timeout_and_recovers(lib, mode, D, causal):
    # mode 3's dQ kernel runs at D = 64 only in deterministic mode
    if mode == 3 and D == 64:
        assert lib.fa_set_deterministic(1) == 0
    try:
        _backward_skip(lib, mode, D, causal, 1, 2, 300)
    finally:
        lib.fa_set_deterministic(0)


@pytest.mark.gpu
def test_fused_backward_skipped_copy_reports_timeout_and_recovers(lib):
    # D = 64 on a grid of at least one dK/dV CTA per SM (4 x 16 heads x 10 key
    # tiles): the CTA that gives up has already added dQ tiles into the
    # accumulator and must wait for those reduce-adds before it exits
    _backward_skip(lib, 2, 64, True, 4, 16, 1280)


def _backward_skip(lib, mode, D, causal, B, H, T):
    scale = 1 / math.sqrt(D)
    q, k, v, do = make_inputs(B, H, T, D, seed=3)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    grads = [torch.empty_like(qd) for _ in range(3)]

    def call():
        rc = fa.fa_bwd(qd, kd, vd, o, dod, lse, *grads, B, H, T, D, scale, int(causal), torch.cuda.current_stream())
        assert rc == 0

    _inject(lib, mode, call)
    assert fa.fa_get_device_status() == -7
    assert fa.fa_get_device_status() == 0
    # The next backward is correct, and so is one whose grids cover every SM
    # (512 dK/dV CTAs, a persistent dQ grid), so the SM whose CTA gave up
    # allocates tensor memory again.
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    rq, rk, rv, _ = oracle.attn_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert np.abs(to_f64(g.cpu()) - r).max() <= grad_bound(r), name
    q, k, v, do = make_inputs(4, 16, 1024, D, seed=5)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for b, h in ((0, 0), (3, 15)):
        rq, rk, rv, _ = oracle.attn_bwd(*(to_f64(t[b, h]) for t in (q, k, v, do)), scale, causal)
        for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            assert np.abs(to_f64(g[b, h].cpu()) - r).max() <= grad_bound(r), (name, b, h)
