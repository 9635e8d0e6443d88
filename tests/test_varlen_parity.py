"""Packed variable-length forward (fa_fwd_varlen) against the fp64 oracle.
Sequences of mixed length (empty, one token, tile multiples +-1, longer than
a tile pair) share one launch; each attends only to itself.  Same tolerances
as the dense forward."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import to_f64
from tests.tolerances import LSE_TOL, o_ok


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_05_gb300 import build
    build.build()
    fa.load_library()


def packed(lengths, H, D, seed, qk_std=1.0):
    total = int(sum(lengths))
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn(total, H, D, generator=g) for _ in range(3))
    q.mul_(qk_std)
    k.mul_(qk_std)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), cu


def run(q, k, v, cu, max_seqlen, causal, scale, expect_status=0):
    dev = torch.device("cuda")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    cud = torch.from_numpy(cu).to(dev)
    total, H, D = q.shape
    o = torch.zeros_like(qd)
    lse = torch.zeros(H, total, device=dev)
    rc = fa.fa_fwd_varlen(qd, kd, vd, o, lse, cud, cu.size - 1, max_seqlen, total, H, D, scale, int(causal),
                          torch.cuda.current_stream())
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == expect_status
    return to_f64(o.cpu()), lse.cpu().double().numpy()


LENGTHS = {
    "tile_edges": [1, 127, 128, 129, 300],
    "with_empty": [0, 513, 7, 0, 256],
    "one_long": [1000],
    "many_short": [3, 60, 64, 65, 17, 200, 1, 90],
}


@pytest.mark.gpu
@pytest.mark.parametrize("mix", sorted(LENGTHS))
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_oracle(mix, D, causal):
    lengths = LENGTHS[mix]
    H = 3
    q, k, v, cu = packed(lengths, H, D, seed=len(lengths) * 7 + D + int(causal))
    scale = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, cu, max(lengths), causal, scale)
    o_ref, lse_ref = oracle.attn_fwd_varlen(to_f64(q), to_f64(k), to_f64(v), cu, scale, causal)
    assert o_ok(o, o_ref), np.abs(o - o_ref).max()
    assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_large_logits(causal):
    # sharp softmax rows (qk std 4): the running max moves by large steps
    lengths = [200, 385, 64]
    q, k, v, cu = packed(lengths, 2, 128, seed=11, qk_std=4.0)
    scale = 1.0 / math.sqrt(128)
    o, lse = run(q, k, v, cu, 400, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd_varlen(to_f64(q), to_f64(k), to_f64(v), cu, scale, causal)
    assert o_ok(o, o_ref), np.abs(o - o_ref).max()
    assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
def test_varlen_loose_max_seqlen_gives_same_bits():
    # max_seqlen only bounds the work list; a larger bound changes nothing
    lengths = [130, 5, 257]
    q, k, v, cu = packed(lengths, 2, 128, seed=3)
    a = run(q, k, v, cu, 257, True, 0.1)
    b = run(q, k, v, cu, 4096, True, 0.1)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_single_sequence_equals_dense_forward(causal):
    T, H, D = 700, 4, 128
    q, k, v, cu = packed([T], H, D, seed=5)
    o, lse = run(q, k, v, cu, T, causal, 0.09)
    dev = torch.device("cuda")
    qd, kd, vd = (t.permute(1, 0, 2).contiguous().unsqueeze(0).to(dev) for t in (q, k, v))
    od = torch.empty_like(qd)
    ld = torch.empty(1, H, T, device=dev)
    assert fa.fa_fwd(qd, kd, vd, od, ld, 1, H, T, D, 0.09, int(causal), torch.cuda.current_stream()) == 0
    torch.cuda.synchronize()
    # The packed forward walks pairs of query tiles; the dense call on one head
    # group this small gives each query tile an SM and splits its key tiles
    # between the two softmax warpgroups, so the two agree to rounding (and each
    # matches the oracle)
    od = to_f64(od[0].permute(1, 0, 2).cpu())
    ld = ld[0].cpu().double().numpy()
    o_ref, lse_ref = oracle.attn_fwd_varlen(to_f64(q), to_f64(k), to_f64(v), cu, 0.09, causal)
    assert o_ok(o, o_ref) and o_ok(od, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL and np.abs(ld - lse_ref).max() <= LSE_TOL
    assert np.abs(o - od).max() <= 2 ** -5 and np.abs(lse - ld).max() <= 1e-5


@pytest.mark.gpu
def test_sequence_longer_than_max_seqlen_is_reported():
    # the second sequence (300 tokens) breaks the promised bound of 200: it is
    # skipped and FA_ERR_SEQLEN is recorded; the first sequence is still right
    lengths = [100, 300]
    q, k, v, cu = packed(lengths, 2, 64, seed=9)
    o, lse = run(q, k, v, cu, 200, True, 0.125, expect_status=-11)
    o_ref, lse_ref = oracle.attn_fwd_varlen(to_f64(q), to_f64(k), to_f64(v), cu, 0.125, True)
    assert o_ok(o[:100], o_ref[:100])
    assert np.abs(lse[:, :100] - lse_ref[:, :100]).max() <= LSE_TOL
    assert fa.fa_get_device_status() == 0   # the status word was cleared by the read


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_serving_mix_sampled_rows(causal):
    # a serving-sized batch: 24 requests of 33..4000 tokens (about 38k tokens),
    # 16 heads, D = 128; rows sampled per sequence and head against the oracle
    rs = np.random.default_rng(17)
    lengths = [int(x) for x in rs.integers(33, 4001, size=24)]
    H, D = 16, 128
    q, k, v, cu = packed(lengths, H, D, seed=23)
    scale = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, cu, max(lengths), causal, scale)
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    for s, L in enumerate(lengths):
        a = int(cu[s])
        rows = np.unique(np.concatenate([[0, L - 1], rs.integers(0, L, size=4)]))
        for h in (0, (s * 5) % H, H - 1):
            o_ref, lse_ref = oracle.attn_fwd_rows(qf[a:a + L, h], kf[a:a + L, h], vf[a:a + L, h], scale, causal,
                                                  rows)
            assert o_ok(o[a + rows, h], o_ref), (s, h)
            assert np.abs(lse[h, a + rows] - lse_ref).max() <= LSE_TOL, (s, h)


# ---------------------------------------------------------------- backward
from tests.tolerances import grad_bound  # noqa: E402


def run_bwd(q, k, v, do, cu, max_seqlen, causal, scale, expect_status=0):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    cud = torch.from_numpy(cu).to(dev)
    o, lse = fa.attention_forward_varlen(qd, kd, vd, cud, max_seqlen, causal=causal, scale=scale)
    dq, dk, dv = (torch.zeros_like(qd) for _ in range(3))
    total, H, D = q.shape
    rc = fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, cud, cu.size - 1, max_seqlen, total, H, D, scale,
                          int(causal), torch.cuda.current_stream())
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == expect_status
    return tuple(to_f64(t.cpu()) for t in (dq, dk, dv))


def packed4(lengths, H, D, seed, qk_std=1.0):
    q, k, v, cu = packed(lengths, H, D, seed, qk_std)
    g = torch.Generator().manual_seed(seed + 1000)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    return q, k, v, do, cu


def check_grads(got, ref, rows=slice(None)):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        bound = grad_bound(r[rows])
        err = np.abs(g[rows] - r[rows]).max()
        assert np.isfinite(g[rows]).all(), name
        assert err <= bound, f"{name}: max err {err:.4g} > {bound:.4g}"


@pytest.mark.gpu
@pytest.mark.parametrize("mix", sorted(LENGTHS))
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_matches_oracle(mix, D, causal):
    lengths = LENGTHS[mix]
    q, k, v, do, cu = packed4(lengths, 3, D, seed=len(lengths) * 5 + D + int(causal))
    scale = 1.0 / math.sqrt(D)
    got = run_bwd(q, k, v, do, cu, max(lengths), causal, scale)
    ref = oracle.attn_bwd_varlen(to_f64(q), to_f64(k), to_f64(v), to_f64(do), cu, scale, causal)
    check_grads(got, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_large_logits(causal):
    lengths = [200, 385, 64]
    q, k, v, do, cu = packed4(lengths, 2, 128, seed=12, qk_std=4.0)
    scale = 1.0 / math.sqrt(128)
    got = run_bwd(q, k, v, do, cu, 400, causal, scale)
    ref = oracle.attn_bwd_varlen(to_f64(q), to_f64(k), to_f64(v), to_f64(do), cu, scale, causal)
    check_grads(got, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_single_sequence_equals_dense(causal):
    T, H, D = 700, 4, 128
    q, k, v, do, cu = packed4([T], H, D, seed=6)
    got = run_bwd(q, k, v, do, cu, T, causal, 0.09)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.permute(1, 0, 2).contiguous().unsqueeze(0).to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=0.09)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=0.09)
    torch.cuda.synchronize()
    # the dense forward of this small head group splits each query tile's key
    # tiles between two warpgroups, so its O and LSE (the backward's inputs)
    # differ from the packed forward's in rounding: the gradients agree within
    # the gradient tolerance
    for g, d in zip(got, (dq, dk, dv)):
        d = to_f64(d[0].permute(1, 0, 2).cpu())
        assert np.abs(g - d).max() <= grad_bound(d)


@pytest.mark.gpu
def test_varlen_backward_sequence_longer_than_max_seqlen_is_reported():
    # the second sequence (300 tokens) breaks the promised bound of 200: its
    # gradients are left unwritten (zeros here) and FA_ERR_SEQLEN is recorded
    lengths = [100, 300]
    q, k, v, do, cu = packed4(lengths, 2, 64, seed=9)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    cud = torch.from_numpy(cu).to(dev)
    # forward and backward with a bound that covers the first sequence only
    o, lse = fa.attention_forward_varlen(qd, kd, vd, cud, 200, causal=True, scale=0.125)
    assert fa.fa_get_device_status() == -11
    dq, dk, dv = (torch.zeros_like(qd) for _ in range(3))
    total, H, D = q.shape
    assert fa.fa_bwd_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, cud, 2, 200, total, H, D, 0.125, 1,
                            torch.cuda.current_stream()) == 0
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == -11
    ref = oracle.attn_bwd_varlen(to_f64(q), to_f64(k), to_f64(v), to_f64(do), cu, 0.125, True)
    got = tuple(to_f64(t.cpu()) for t in (dq, dk, dv))
    check_grads(got, ref, rows=slice(0, 100))
    for g in got:
        assert not g[100:].any()
    assert fa.fa_get_device_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_serving_mix_sampled_rows(causal):
    # 16 requests of 33..3000 tokens, 16 heads, D = 128; rows of dQ, dK and dV
    # sampled per sequence and head against the oracle
    rs = np.random.default_rng(19)
    lengths = [int(x) for x in rs.integers(33, 3001, size=16)]
    H, D = 16, 128
    q, k, v, do, cu = packed4(lengths, H, D, seed=31)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = run_bwd(q, k, v, do, cu, max(lengths), causal, scale)
    qf, kf, vf, dof = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    for s, L in enumerate(lengths):
        a = int(cu[s])
        rows = np.unique(np.concatenate([[0, L - 1], rs.integers(0, L, size=3)]))
        for h in (0, (s * 7) % H, H - 1):
            sl = slice(a, a + L)
            rq, rk, rv, _, _ = oracle.attn_bwd_rows(qf[sl, h], kf[sl, h], vf[sl, h], dof[sl, h], scale, causal,
                                                    rows, rows)
            for name, g, r in (("dq", dq[a + rows, h], rq), ("dk", dk[a + rows, h], rk), ("dv", dv[a + rows, h], rv)):
                assert np.abs(g - r).max() <= grad_bound(r), (name, s, h)


@pytest.mark.gpu
@pytest.mark.slow
def test_serving_pack_whole_sequences():
    # The packed batch the bench times: 48 causal requests of 128..8192 tokens
    # (numpy seed 0), 16 heads, D = 128, inputs seed 0.  Forward and backward
    # run on the whole pack; the longest, the shortest and the median-length
    # request are compared against the oracle in full, every head and row.
    n_seq, H, D = 48, 16, 128
    lengths = np.random.default_rng(0).integers(128, 8193, size=n_seq)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    total, Tmax = int(cu[-1]), int(lengths.max())
    g = torch.Generator().manual_seed(0)
    q, k, v, do = (torch.randn(total, H, D, generator=g).to(torch.bfloat16) for _ in range(4))
    scale = D ** -0.5
    o, lse = run(q, k, v, cu, Tmax, True, scale)
    dq, dk, dv = run_bwd(q, k, v, do, cu, Tmax, True, scale)
    order = np.argsort(lengths, kind="stable")
    for s in (int(order[-1]), int(order[0]), int(order[n_seq // 2])):
        a, L = int(cu[s]), int(lengths[s])
        sl = slice(a, a + L)
        # (L, H, D) -> (1, H, L, D) for the dense oracle
        qf, kf, vf, df = (to_f64(t[sl]).transpose(1, 0, 2)[None] for t in (q, k, v, do))
        o_ref, lse_ref = oracle.attn_fwd(qf, kf, vf, scale, True)
        assert o_ok(o[sl].transpose(1, 0, 2)[None], o_ref), s
        assert np.abs(lse[:, sl][None] - lse_ref).max() <= LSE_TOL, s
        ref = oracle.attn_bwd(qf, kf, vf, df, scale, True)[:3]
        check_grads([t[sl].transpose(1, 0, 2)[None] for t in (dq, dk, dv)], ref)
