"""Forward parity: the CUDA forward (through the C ABI) against the fp64 CPU
oracle on the same bf16 inputs.  Tolerances: O max-abs <= 1e-2, LSE max-abs
<= 1e-3.  Shapes here are checked element by element over every output; the
full-size workloads are compared element by element in
test_workload_parity.py, and a 32731-token head on sampled rows in
test_bwd_parity.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import WORKLOADS, make_inputs, to_f64, workload_inputs

from tests.tolerances import LSE_TOL, O_TOL, o_ok


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_05_gb300 import build
    build.build()
    fa.load_library()


def run_fwd(q, k, v, causal, scale):
    dev = torch.device("cuda")
    o, lse = fa.attention_forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    return to_f64(o.cpu()), lse.cpu().double().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 383, 500])
def test_forward_small_shapes_full_compare(T, causal, D):
    B, H = 1, 2
    q, k, v, _ = make_inputs(B, H, T, D, seed=T + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    assert o_ok(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
@pytest.mark.parametrize("scale", [0.0, -0.07, 0.3])
def test_forward_unusual_scales(scale):
    B, H, T, D = 1, 1, 300, 64
    q, k, v, _ = make_inputs(B, H, T, D, seed=5)
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, causal, scale)
        o_ref, lse_ref = oracle.attn_fwd(to_f64(q), to_f64(k), to_f64(v), scale, causal)
        assert o_ok(o, o_ref)
        assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129, 200, 3000])
def test_mask_probe_uniform_scores(T, causal, D):
    # Q = 0 makes every visible score 0, so P is uniform over the visible keys.
    # With V[j] = e_{j mod D}: O[i, c] = #{visible j : j = c mod D} / #visible and
    # LSE_i = log(#visible).  Which O entries are nonzero is an integer fact and
    # must match exactly; the values match the closed form within tolerance.
    B, H = 1, 1
    q = torch.zeros(B, H, T, D, dtype=torch.bfloat16)
    k = torch.randn(B, H, T, D, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    v = torch.zeros(B, H, T, D, dtype=torch.bfloat16)
    v[0, 0, torch.arange(T), torch.arange(T) % D] = 1.0
    o, lse = run_fwd(q, k, v, causal, 0.125)
    i = np.arange(T)
    n_vis = (i + 1) if causal else np.full(T, T)
    counts = np.zeros((T, D))
    for c in range(D):
        # keys j < n_vis with j % D == c
        counts[:, c] = np.maximum(0, (n_vis - 1 - c) // D + 1)
    want = counts / n_vis[:, None]
    np.testing.assert_array_equal(o[0, 0] != 0, want != 0)
    assert np.abs(o[0, 0] - want).max() <= O_TOL
    assert np.abs(lse[0, 0] - np.log(n_vis)).max() <= 1e-5


@pytest.mark.gpu
def test_forward_large_logits_growing_max():
    # keys whose scores grow by hundreds from tile to tile: the deferred rescale must stay exact
    B, H, T, D = 1, 2, 640, 128
    g = torch.Generator().manual_seed(11)
    q = torch.randn(B, H, T, D, generator=g)
    k = torch.randn(B, H, T, D, generator=g) * torch.linspace(0.1, 30.0, T)[None, None, :, None]
    v = torch.randn(B, H, T, D, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, causal, 1.0 / math.sqrt(D))
        o_ref, lse_ref = oracle.attn_fwd(to_f64(q), to_f64(k), to_f64(v), 1.0 / math.sqrt(D), causal)
        assert o_ok(o, o_ref)
        assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny_b1h2t128d64", "fwd_b1h8t1024d64"])
def test_forward_workload_full_compare(name):
    w = WORKLOADS[name]
    q, k, v, _ = workload_inputs(w)
    for causal in w.causal:
        o, lse = run_fwd(q, k, v, causal, w.scale)
        o_ref, lse_ref = oracle.attn_fwd(to_f64(q), to_f64(k), to_f64(v), w.scale, causal)
        assert o_ok(o, o_ref)
        assert np.abs(lse - lse_ref).max() <= LSE_TOL



@pytest.mark.gpu
@pytest.mark.parametrize("D,T", [(64, 1024), (128, 2048), (128, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_work_partition_keeps_parity(D, T, causal):
    # One batch of 4 heads has few work items, so each query tile gets an SM of
    # its own and its two softmax warpgroups split the key tiles (their states
    # merged at the end); inside a batch of 16 x 4 heads the same heads are
    # walked as pairs of query tiles by persistent CTAs.  Both must match the
    # oracle on the shared heads, and agree with each other to rounding.
    H = 4
    q, k, v, _ = make_inputs(16, H, T, D, seed=21)
    dev = torch.device("cuda")
    scale = D ** -0.5
    o_small, l_small = fa.attention_forward(q[:1].to(dev), k[:1].to(dev), v[:1].to(dev), causal=causal, scale=scale)
    o_big, l_big = fa.attention_forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(to_f64(q[0]), to_f64(k[0]), to_f64(v[0]), scale, causal)
    for o, lse in ((o_small[0], l_small[0]), (o_big[0], l_big[0])):
        assert o_ok(to_f64(o.cpu()), o_ref)
        assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= LSE_TOL
    assert (o_small[0].float() - o_big[0].float()).abs().max().item() <= 2 ** -5

