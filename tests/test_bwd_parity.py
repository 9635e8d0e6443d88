"""Backward parity: dQ, dK, dV from the CUDA path (fa_fwd then fa_bwd through
the C ABI) against the fp64 oracle's analytic gradients on the same bf16
inputs, max-abs <= 2e-2 * max|grad| per tensor.  Small shapes compare every
element (the full-size workloads are compared element by element in
test_workload_parity.py); a 32731-token head and a 2900-token batch compare
sampled rows the oracle computes one by one (rows of dQ need one row of P,
rows of dK/dV one column)."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import WORKLOADS, make_inputs, to_f64, workload_inputs
from tests.tolerances import LSE_TOL, grad_bound, o_ok


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_05_gb300 import build
    build.build()
    fa.load_library()


def run_fwd_bwd(q, k, v, do, causal, scale):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    return tuple(to_f64(t.cpu()) for t in (dq, dk, dv))


def check(name, g, r):
    bound = grad_bound(r)
    err = np.abs(g - r).max()
    assert np.isfinite(g).all(), name
    assert err <= bound, f"{name}: max err {err:.4g} > {bound:.4g}"


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 200, 255, 257, 383, 500])
def test_backward_small_shapes_full_compare(T, causal, D):
    B, H = 1, 2
    q, k, v, do = make_inputs(B, H, T, D, seed=100 + T + D)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, scale)
    rq, rk, rv, _ = oracle.attn_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    check("dq", dq, rq)
    check("dk", dk, rk)
    check("dv", dv, rv)


@pytest.mark.gpu
@pytest.mark.parametrize("scale", [0.0, -0.07, 0.3])
def test_backward_unusual_scales(scale):
    B, H, T, D = 1, 1, 200, 64
    q, k, v, do = make_inputs(B, H, T, D, seed=9)
    for causal in (False, True):
        dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, scale)
        rq, rk, rv, _ = oracle.attn_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
        if scale != 0.0:
            check("dq", dq, rq)
            check("dk", dk, rk)
        else:  # scale 0: dQ and dK are exactly zero
            assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
        check("dv", dv, rv)


@pytest.mark.gpu
def test_backward_tiny_workload_both_masks():
    w = WORKLOADS["tiny_b1h2t128d64"]
    q, k, v, do = workload_inputs(w)
    for causal in w.causal:
        dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, w.scale)
        rq, rk, rv, _ = oracle.attn_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), w.scale, causal)
        check("dq", dq, rq)
        check("dk", dk, rk)
        check("dv", dv, rv)


@pytest.mark.gpu
def test_backward_head_pair_schedule_odd_tile_count():
    # Non-causal, K and V of all heads well above half of L2: the dQ kernel
    # walks (tile n-1-r, tile r) pairs head by head.  T = 2900 gives 23 query
    # tiles, so tile 11 has no partner; rows of every tile boundary and of the
    # unpaired tile are compared, on the first, a middle and the last head.
    B, H, T, D = 8, 32, 2900, 128
    q, k, v, do = make_inputs(B, H, T, D, seed=29)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = run_fwd_bwd(q, k, v, do, False, scale)
    rng = np.random.default_rng(11)
    middle = 11 * 128
    for bh in (0, B * H // 2 + 3, B * H - 1):
        b, h = divmod(bh, H)
        rows = sorted({0, 127, 128, middle, middle + 77, middle + 127, T - 1} | set(rng.integers(0, T, 12).tolist()))
        rq, rk, rv, _, _ = oracle.attn_bwd_rows(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]),
                                                to_f64(do[b, h]), scale, False, rows, rows)
        check(f"dq[{bh}]", dq[b, h, rows], rq)
        check(f"dk[{bh}]", dk[b, h, rows], rk)
        check(f"dv[{bh}]", dv[b, h, rows], rv)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_work_partition_does_not_change_bits_backward(D, causal, deterministic_backward):
    # 4 heads of T = 2048 make few dK/dV CTAs, launched key tile major; 32 x 4
    # heads make many, launched head by head; the dQ kernel hands its items out
    # in whatever order CTAs ask.  Each key tile's dK / dV and each query tile's
    # dQ are computed the same way wherever they run, so the shared heads'
    # gradients must agree bit for bit.
    B, H, T = 32, 4, 2048
    q, k, v, do = make_inputs(B, H, T, D, seed=23)
    dev = torch.device("cuda")
    scale = D ** -0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    big = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    small = fa.attention_backward(qd[:1].contiguous(), kd[:1].contiguous(), vd[:1].contiguous(), o[:1].contiguous(),
                                  lse[:1].contiguous(), dod[:1].contiguous(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for g_small, g_big in zip(small, big):
        assert torch.equal(g_small[0], g_big[0])


@pytest.mark.gpu
@pytest.mark.parametrize("D,causal,T", [(128, True, 32768 - 37), (64, False, 32768 - 37),
                                         pytest.param(128, True, 65536 + 61, marks=pytest.mark.slow)])
def test_long_sequence_sampled_rows(D, causal, T):
    # one head of 32731 tokens (256 tiles, the last one ragged), or of 65597
    # (513 tiles, the last one holding 61 rows): forward O and LSE and
    # backward dQ, dK, dV on sampled rows, including both ends
    q, k, v, do = make_inputs(1, 1, T, D, seed=41)
    scale = D ** -0.5
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    rng = np.random.default_rng(43)
    rows = sorted({0, 1, 127, 128, 16383, 16384, T // 2, T - 129, T - 128, T - 2, T - 1}
                  | set(rng.integers(0, T, 16).tolist()))
    qf, kf, vf, df = (to_f64(t[0, 0]) for t in (q, k, v, do))
    o_ref, lse_ref = oracle.attn_fwd_rows(qf, kf, vf, scale, causal, rows)
    o_got = to_f64(o[0, 0].cpu())[rows]
    assert o_ok(o_got, o_ref)
    assert np.abs(lse[0, 0].cpu().double().numpy()[rows] - lse_ref).max() <= LSE_TOL
    rq, rk, rv, _, _ = oracle.attn_bwd_rows(qf, kf, vf, df, scale, causal, rows, rows)
    check("dq", to_f64(dq[0, 0].cpu())[rows], rq)
    check("dk", to_f64(dk[0, 0].cpu())[rows], rk)
    check("dv", to_f64(dv[0, 0].cpu())[rows], rv)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_fused_backward_against_the_two_kernel_form(causal):
    # D = 64 by default computes dQ inside the dK/dV kernel and sums the key
    # tiles' contributions with float32 reduce-adds.  dK and dV come from the
    # same per-key-tile arithmetic as the two-kernel form and must match it bit
    # for bit.  dQ is built from the dK/dV kernel's own dS (rounded to bf16
    # there, not in a second kernel), so the two forms' dQ are each checked
    # against the oracle; two fused runs differ only in the order of the same
    # float32 sums.  The batch's grid covers every SM (64 heads).
    from tests.tolerances import same_up_to_sum_order
    B, H, T, D = 4, 16, 1000, 64
    q, k, v, do = make_inputs(B, H, T, D, seed=27)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal)
    fused = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal)
    fused2 = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal)
    lib = fa.load_library()
    assert lib.fa_set_deterministic(1) == 0
    try:
        two = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal)
    finally:
        lib.fa_set_deterministic(0)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    assert torch.equal(fused[1], two[1]) and torch.equal(fused[2], two[2])
    assert same_up_to_sum_order(fused[0], fused2[0])
    for b, h in ((0, 0), (1, 7), (3, 15)):
        rq, rk, rv, _ = oracle.attn_bwd(*(to_f64(t[b, h]) for t in (q, k, v, do)), D ** -0.5, causal)
        check("dq fused", to_f64(fused[0][b, h].cpu()), rq)
        check("dq two-kernel", to_f64(two[0][b, h].cpu()), rq)

