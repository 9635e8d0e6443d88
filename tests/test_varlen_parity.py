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
    np.testing.assert_array_equal(o, to_f64(od[0].permute(1, 0, 2).cpu()))
    np.testing.assert_array_equal(lse, ld[0].cpu().double().numpy())


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
