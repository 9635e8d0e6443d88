"""The autograd entry point (FlashAttention.apply / flash_attention): its
gradients are the library's backward, checked against the fp64 oracle and
bitwise against the direct C-ABI calls; the (B, T, D) form equals one head of
the (B, H, T, D) form; CPU tensors are refused (there is no CPU path)."""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import make_inputs, to_f64

from tests.tolerances import grad_bound, o_ok, same_gradients, same_up_to_sum_order


def test_cpu_tensors_are_refused():
    q = torch.zeros(1, 2, 16, 64, dtype=torch.bfloat16, requires_grad=True)
    with pytest.raises(ValueError):
        fa.flash_attention(q, q, q)
    with pytest.raises(ValueError):
        fa.FlashAttention.apply(q[0], q[0], q[0], True)


def leaf(t):
    return t.to("cuda").requires_grad_(True)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_oracle_and_direct_calls(D, causal):
    from online_softmax_05_gb300 import build
    build.build()
    B, H, T = 2, 3, 200
    q, k, v, do = make_inputs(B, H, T, D, seed=61)
    scale = D ** -0.5
    ql, kl, vl = leaf(q), leaf(k), leaf(v)
    o = fa.FlashAttention.apply(ql, kl, vl, causal)
    (o.float() * do.to("cuda").float()).sum().backward()
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    # the same numbers as the direct calls
    o2, lse2 = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    g2 = fa.attention_backward(q.cuda(), k.cuda(), v.cuda(), o2, lse2, do.cuda(), causal=causal, scale=scale)
    assert torch.equal(o.detach(), o2)
    assert same_gradients((ql.grad, kl.grad, vl.grad), g2, D)
    # and within tolerance of the oracle
    qf, kf, vf, df = (to_f64(t) for t in (q, k, v, do))
    o_ref, _ = oracle.attn_fwd(qf, kf, vf, scale, causal)
    assert o_ok(to_f64(o.detach().cpu()), o_ref)
    refs = oracle.attn_bwd(qf, kf, vf, df, scale, causal)[:3]
    for got, ref in zip((ql.grad, kl.grad, vl.grad), refs):
        assert np.abs(to_f64(got.cpu()) - ref).max() <= grad_bound(ref)


@pytest.mark.gpu
def test_three_dimensional_form_is_one_head():
    from online_softmax_05_gb300 import build
    build.build()
    q, k, v, do = make_inputs(2, 1, 300, 64, seed=62)
    q3, k3, v3 = leaf(q[:, 0]), leaf(k[:, 0]), leaf(v[:, 0])
    o3 = fa.flash_attention(q3, k3, v3, causal=True)
    (o3.float() * do[:, 0].cuda().float()).sum().backward()
    q4, k4, v4 = leaf(q), leaf(k), leaf(v)
    o4 = fa.flash_attention(q4, k4, v4, causal=True)
    (o4.float() * do.cuda().float()).sum().backward()
    torch.cuda.synchronize()
    assert o3.shape == (2, 300, 64)
    assert torch.equal(o3.detach(), o4.detach()[:, 0])
    assert same_up_to_sum_order(q3.grad, q4.grad[:, 0])   # D = 64: dQ sums in varying order
    for a, b in ((k3, k4), (v3, v4)):
        assert torch.equal(a.grad, b.grad[:, 0])
