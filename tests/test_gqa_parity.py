"""Grouped-query attention (fa_fwd_gqa / fa_bwd_gqa) against the fp64
oracle: query head h reads key/value head h // (Hq // Hkv); dK, dV sum over
each group.  Same tolerances as plain attention.  Groups of 1 (plain), 2 and
8 (pairs of query heads share a CTA's K/V tiles) and 3 (odd: consecutive
tiles of one head per CTA)."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import to_f64
from tests.tolerances import LSE_TOL, grad_bound, o_ok


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_05_gb300 import build
    build.build()
    fa.load_library()


def make(B, Hq, Hkv, T, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, T, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16)
    do = torch.randn(B, Hq, T, D, generator=g).to(torch.bfloat16)
    return q, k, v, do


def run(q, k, v, do, causal, scale):
    dev = torch.device("cuda")
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, T, device=dev)
    st = torch.cuda.current_stream()
    assert fa.fa_fwd_gqa(qd, kd, vd, o, lse, B, Hq, Hkv, T, D, scale, int(causal), st) == 0
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    assert fa.fa_bwd_gqa(qd, kd, vd, o, dod, lse, dq, dk, dv, B, Hq, Hkv, T, D, scale, int(causal), st) == 0
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    return [to_f64(t.cpu()) for t in (o, dq, dk, dv)] + [lse.cpu().double().numpy()]


@pytest.mark.gpu
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (6, 2), (8, 1)])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T", [65, 200, 383])
def test_gqa_matches_oracle(Hq, Hkv, D, causal, T):
    q, k, v, do = make(1, Hq, Hkv, T, D, seed=Hq * 100 + Hkv * 10 + T + D)
    scale = 1.0 / math.sqrt(D)
    o, dq, dk, dv, lse = run(q, k, v, do, causal, scale)
    qf, kf, vf, df = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref = oracle.attn_fwd_gqa(qf, kf, vf, scale, causal)
    assert o_ok(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL
    rq, rk, rv, _ = oracle.attn_bwd_gqa(qf, kf, vf, df, scale, causal)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert np.abs(g - r).max() <= grad_bound(r), name


@pytest.mark.gpu
def test_gqa_group_of_one_equals_plain_entry_points():
    q, k, v, do = make(2, 3, 3, 300, 128, seed=9)
    o, dq, dk, dv, lse = run(q, k, v, do, True, 0.1)
    dev = torch.device("cuda")
    o2, lse2 = fa.attention_forward(q.to(dev), k.to(dev), v.to(dev), causal=True, scale=0.1)
    dq2, dk2, dv2 = fa.attention_backward(q.to(dev), k.to(dev), v.to(dev), o2, lse2, do.to(dev), causal=True, scale=0.1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o, to_f64(o2.cpu()))
    np.testing.assert_array_equal(lse, lse2.cpu().double().numpy())
    np.testing.assert_array_equal(dk, to_f64(dk2.cpu()))
    np.testing.assert_array_equal(dv, to_f64(dv2.cpu()))
    assert np.abs(dq - to_f64(dq2.cpu())).max() <= 1e-2 * np.abs(dq).max()  # fp32 reductions in any order


@pytest.mark.gpu
def test_gqa_longer_sequence():
    q, k, v, do = make(1, 8, 2, 1024, 128, seed=10)
    scale = 1.0 / math.sqrt(128)
    o, dq, dk, dv, lse = run(q, k, v, do, True, scale)
    qf, kf, vf, df = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref = oracle.attn_fwd_gqa(qf, kf, vf, scale, True)
    assert o_ok(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL
    rq, rk, rv, _ = oracle.attn_bwd_gqa(qf, kf, vf, df, scale, True)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert np.abs(g - r).max() <= grad_bound(r), name


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_fused_backward_full_grid(causal):
    # D = 64 with at least one dK/dV CTA per SM (4 batches x 4 K/V heads x 10
    # key tiles = 160): the backward sums dQ with reduce-adds inside the dK/dV
    # kernel, walking the query tiles of all 4 query heads of each group.
    # Batches are independent, so the oracle checks the first and the last.
    B, Hq, Hkv, T, D = 4, 16, 4, 1280, 64
    q, k, v, do = make(B, Hq, Hkv, T, D, seed=12)
    scale = D ** -0.5
    o, dq, dk, dv, lse = run(q, k, v, do, causal, scale)
    for b in (0, B - 1):
        qf, kf, vf, df = (to_f64(t[b:b + 1]) for t in (q, k, v, do))
        rq, rk, rv, _ = oracle.attn_bwd_gqa(qf, kf, vf, df, scale, causal)
        for name, g, r in (("dq", dq[b:b + 1], rq), ("dk", dk[b:b + 1], rk), ("dv", dv[b:b + 1], rv)):
            assert np.abs(g - r).max() <= grad_bound(r), (name, b)


@pytest.mark.gpu
@pytest.mark.slow
def test_gqa_long_context_whole_groups():
    # The long-context causal shape with 4 query heads per K/V head (B=2,
    # Hq=16, Hkv=4, T=8192, D=128) at full size.  Two whole groups are compared
    # element by element: K/V head 0 of batch 0 and K/V head 3 of batch 1, with
    # their 4 query heads each (O, LSE, dQ of the query heads; dK, dV summed
    # over the group).
    B, Hq, Hkv, T, D = 2, 16, 4, 8192, 128
    q, k, v, do = make(B, Hq, Hkv, T, D, seed=13)
    scale = D ** -0.5
    o, dq, dk, dv, lse = run(q, k, v, do, True, scale)
    g = Hq // Hkv
    for b, kvh in ((0, 0), (1, Hkv - 1)):
        hs = slice(kvh * g, (kvh + 1) * g)
        qf, df = (to_f64(t[b:b + 1, hs]) for t in (q, do))
        kf, vf = (to_f64(t[b:b + 1, kvh:kvh + 1]) for t in (k, v))
        o_ref, lse_ref = oracle.attn_fwd_gqa(qf, kf, vf, scale, True)
        assert o_ok(o[b:b + 1, hs], o_ref), (b, kvh)
        assert np.abs(lse[b:b + 1, hs] - lse_ref).max() <= LSE_TOL, (b, kvh)
        rq, rk, rv, _ = oracle.attn_bwd_gqa(qf, kf, vf, df, scale, True)
        for name, got, r in (("dq", dq[b:b + 1, hs], rq), ("dk", dk[b:b + 1, kvh:kvh + 1], rk),
                             ("dv", dv[b:b + 1, kvh:kvh + 1], rv)):
            assert np.abs(got - r).max() <= grad_bound(r), (name, b, kvh)
