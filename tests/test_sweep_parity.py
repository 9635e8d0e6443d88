"""Parity at the shapes of the T sweep (`bench.py --sweep`): 16384 tokens x 16
heads per case, T from 512 to 8192 (B = 16384 / T), D in {64, 128}, with and
without causal masking.  Each case runs the forward and the backward at full
size, in the launch configuration the sweep times; the first and the last
head are compared with the fp64 oracle element by element (O, LSE, dQ, dK,
dV), at the tolerances of every other parity test."""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import make_inputs, to_f64
from tests.tolerances import LSE_TOL, grad_bound, o_ok

CASES = [(D, causal, T) for D in (64, 128) for causal in (False, True) for T in (512, 1024, 2048, 4096, 8192)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_05_gb300 import build
    build.build()
    fa.load_library()


@pytest.mark.gpu
@pytest.mark.slow
@pytest.mark.parametrize("D,causal,T", CASES, ids=[f"d{D}-{'causal' if c else 'full'}-t{T}" for D, c, T in CASES])
def test_sweep_shape_first_and_last_head(D, causal, T):
    B, H = 16384 // T, 16
    q, k, v, do = make_inputs(B, H, T, D, seed=T + D)
    scale = D ** -0.5
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for b, h in ((0, 0), (B - 1, H - 1)):
        qf, kf, vf, df = (to_f64(t[b, h]) for t in (q, k, v, do))
        o_ref, lse_ref = oracle.attn_fwd(qf, kf, vf, scale, causal)
        assert o_ok(to_f64(o[b, h].cpu()), o_ref), (b, h)
        assert np.abs(lse[b, h].cpu().double().numpy() - lse_ref).max() <= LSE_TOL, (b, h)
        rq, rk, rv, _ = oracle.attn_bwd(qf, kf, vf, df, scale, causal)
        for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            assert np.abs(to_f64(g[b, h].cpu()) - r).max() <= grad_bound(r), (name, b, h)
