"""Split-K decoding forward (fa_decode) against the fp64 oracle for queries
attending to a longer key sequence.  O max-abs <= 1e-2 (bf16 half-ulp added
above |O| >= 4), LSE max-abs <= 1e-3, every element compared."""
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


def make(B, H, Tq, Tk, D, seed, qk_std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Tq, D, generator=g) * qk_std).to(torch.bfloat16)
    k = (torch.randn(B, H, Tk, D, generator=g) * qk_std).to(torch.bfloat16)
    v = torch.randn(B, H, Tk, D, generator=g).to(torch.bfloat16)
    return q, k, v


def run(q, k, v, scale):
    dev = torch.device("cuda")
    o, lse = fa.attention_decode(q.to(dev), k.to(dev), v.to(dev), scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    return to_f64(o.cpu()), lse.cpu().double().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Tq", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("Tk", [1, 7, 255, 256, 257, 1000, 4109])
def test_decode_matches_oracle(Tq, Tk, D):
    B, H = 2, 3
    q, k, v = make(B, H, Tq, Tk, D, seed=Tq * 1000 + Tk + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, scale)
    o_ref, lse_ref = oracle.attn_fwd_cross(to_f64(q), to_f64(k), to_f64(v), scale)
    assert o_ok(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
@pytest.mark.parametrize("scale", [0.0, -0.2])
def test_decode_unusual_scales(scale):
    q, k, v = make(1, 2, 2, 700, 128, seed=3)
    o, lse = run(q, k, v, scale)
    o_ref, lse_ref = oracle.attn_fwd_cross(to_f64(q), to_f64(k), to_f64(v), scale)
    assert o_ok(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
def test_decode_large_logits():
    # scores with standard deviation ~30: near one-hot rows, the max moves between key chunks
    q, k, v = make(2, 4, 4, 5000, 128, seed=4, qk_std=4.0)
    o, lse = run(q, k, v, 1.0 / math.sqrt(128))
    o_ref, lse_ref = oracle.attn_fwd_cross(to_f64(q), to_f64(k), to_f64(v), 1.0 / math.sqrt(128))
    assert o_ok(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
def test_decode_long_cache():
    # one new token per head against a 32768-token cache
    B, H, Tq, Tk, D = 2, 8, 1, 32768, 128
    q, k, v = make(B, H, Tq, Tk, D, seed=5)
    o, lse = run(q, k, v, 1.0 / math.sqrt(D))
    o_ref, lse_ref = oracle.attn_fwd_cross(to_f64(q), to_f64(k), to_f64(v), 1.0 / math.sqrt(D))
    assert o_ok(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= LSE_TOL


@pytest.mark.gpu
def test_decode_equals_forward_when_lengths_match():
    # the same attention through both paths (T_q = T_k = 8, no mask)
    q, k, v = make(1, 2, 8, 8, 64, seed=6)
    o_dec, lse_dec = run(q, k, v, 0.125)
    dev = torch.device("cuda")
    o_fwd, lse_fwd = fa.attention_forward(q.to(dev), k.to(dev), v.to(dev), causal=False, scale=0.125)
    torch.cuda.synchronize()
    assert np.abs(o_dec - to_f64(o_fwd.cpu())).max() <= 1e-2
    assert np.abs(lse_dec - lse_fwd.cpu().double().numpy()).max() <= 1e-3


@pytest.mark.gpu
@pytest.mark.slow
def test_decode_bench_shape_every_head():
    # the shape the bench times: one new token for each of B=8 x H=32 heads
    # against a 32768-token cache, D = 128 (its own split of the keys across
    # CTAs); every head compared, 32 heads at a time on the host
    B, H, Tq, Tk, D = 8, 32, 1, 32768, 128
    q, k, v = make(B, H, Tq, Tk, D, seed=8)
    scale = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, scale)
    q3, k3, v3 = (t.reshape(B * H, 1, -1, D) for t in (q, k, v))
    o3, lse3 = o.reshape(B * H, 1, Tq, D), lse.reshape(B * H, 1, Tq)
    for lo in range(0, B * H, 32):
        hs = slice(lo, lo + 32)
        o_ref, lse_ref = oracle.attn_fwd_cross(to_f64(q3[hs]), to_f64(k3[hs]), to_f64(v3[hs]), scale)
        assert o_ok(o3[hs], o_ref), lo
        assert np.abs(lse3[hs] - lse_ref).max() <= LSE_TOL, lo
