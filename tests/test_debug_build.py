"""The debug build of the library (libfa_debug.so, the same sources compiled
with FA_DEBUG): every kernel checks its run-time tile coordinates, ring
stages, per-row vector offsets and tensor-memory columns before it uses
them.  A failed check skips the access and is reported as
FA_ERR_DEBUG_CHECK, never as a trap.

Host side: the debug library exports every symbol include/fa.h declares and
says it is the debug build.  GPU side: the small parity cases (both masks,
both head dimensions, ragged tails, grouped heads, a packed batch) run
through the debug library with no check failing, and its results equal the
product library's bit for bit (the checks change no arithmetic; dQ of the
D = 64 backward up to the order of its float32 sums)."""
import ctypes
import math
import os

import numpy as np
import pytest
import torch

import oracle
import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import make_inputs, to_f64
from tests.test_abi import declared_functions
from tests.tolerances import LSE_TOL, grad_bound, o_ok, same_gradients

PKG = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "online_softmax_05_gb300")


@pytest.fixture(scope="module")
def dlib():
    from online_softmax_05_gb300 import build
    try:
        build.build()
    except RuntimeError as e:
        pytest.skip(f"the CUDA libraries cannot be built here: {e}")
    lib = ctypes.CDLL(os.path.join(PKG, "libfa_debug.so"))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_bwd.argtypes = [vp] * 9 + [i, i, i, i, f, i, vp]
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_bwd_gqa.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp]
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_bwd_varlen.argtypes = [vp] * 10 + [i, i, i, i, i, f, i, vp]
    lib.fa_get_device_status.argtypes = [vp]
    return lib


def test_debug_library_exports_every_symbol_and_says_so(dlib):
    for n in declared_functions():
        assert hasattr(dlib, n), n
    assert dlib.fa_debug_checks_enabled() == 1
    assert fa.load_library().fa_debug_checks_enabled() == 0


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T", [1, 65, 128, 300, 1000])
def test_debug_build_runs_small_cases_clean(dlib, T, causal, D):
    B, H = 2, 3
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = make_inputs(B, H, T, D, seed=7 + T)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, T, device=dev)
    dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
    assert dlib.fa_fwd(_p(qd), _p(kd), _p(vd), _p(o), _p(lse), B, H, T, D, scale, int(causal), stream) == 0
    assert dlib.fa_bwd(_p(qd), _p(kd), _p(vd), _p(o), _p(dod), _p(lse), _p(dq), _p(dk), _p(dv), B, H, T, D, scale,
                       int(causal), stream) == 0
    assert dlib.fa_get_device_status(stream) == 0
    # the product library computes the same bits
    o2, lse2 = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    g2 = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert same_gradients((dq, dk, dv), g2, D)
    # and the oracle agrees
    o_ref, lse_ref = oracle.attn_fwd(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    assert o_ok(to_f64(o.cpu()), o_ref)
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= LSE_TOL
    rq, rk, rv, _ = oracle.attn_bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.abs(to_f64(g.cpu()) - r).max() <= grad_bound(r)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_debug_build_grouped_and_packed_clean(dlib, causal):
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    D, T, B, Hq, Hkv = 128, 700, 2, 8, 2
    scale = D ** -0.5
    g = torch.Generator().manual_seed(3)
    q = torch.randn(B, Hq, T, D, generator=g).to(torch.bfloat16).to(dev)
    k, v = (torch.randn(B, Hkv, T, D, generator=g).to(torch.bfloat16).to(dev) for _ in range(2))
    do = torch.randn(B, Hq, T, D, generator=g).to(torch.bfloat16).to(dev)
    o, lse = torch.empty_like(q), torch.empty(B, Hq, T, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert dlib.fa_fwd_gqa(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, T, D, scale, int(causal), stream) == 0
    assert dlib.fa_bwd_gqa(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv), B, Hq, Hkv, T, D,
                           scale, int(causal), stream) == 0
    assert dlib.fa_get_device_status(stream) == 0
    # packed batch: lengths 1, 300, 0, 129 with max_seqlen 300
    cu = torch.tensor([0, 1, 301, 301, 430], dtype=torch.int32, device=dev)
    total, H = 430, 4
    qp, kp, vp_, dop = (torch.randn(total, H, D, generator=g).to(torch.bfloat16).to(dev) for _ in range(4))
    op, lsep = torch.empty_like(qp), torch.empty(H, total, device=dev)
    dqp, dkp, dvp = (torch.empty_like(qp) for _ in range(3))
    assert dlib.fa_fwd_varlen(_p(qp), _p(kp), _p(vp_), _p(op), _p(lsep), _p(cu), 4, 300, total, H, D, scale,
                              int(causal), stream) == 0
    assert dlib.fa_bwd_varlen(_p(qp), _p(kp), _p(vp_), _p(op), _p(dop), _p(lsep), _p(dqp), _p(dkp), _p(dvp), _p(cu),
                              4, 300, total, H, D, scale, int(causal), stream) == 0
    assert dlib.fa_get_device_status(stream) == 0
    o_ref, _ = oracle.attn_fwd_varlen(to_f64(qp.cpu()), to_f64(kp.cpu()), to_f64(vp_.cpu()), cu.cpu().numpy(), scale,
                                      causal)
    assert o_ok(to_f64(op.cpu()), o_ref)


@pytest.mark.gpu
@pytest.mark.slow
@pytest.mark.parametrize("name", ["causal_b4h16t2048d64", "causal_b2h16t8192d128", "ragged_b8h32t3000d128"])
def test_debug_build_full_size_workloads_clean(dlib, name):
    # every run-time index of the full-size launches (the configurations the
    # bench times) passes its check, and the debug build computes the product
    # build's bits
    from online_softmax_05_gb300.inputs import WORKLOADS, workload_inputs
    w = WORKLOADS[name]
    causal = int(w.causal[0])
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in workload_inputs(w))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, H, T, D = w.B, w.H, w.T, w.D
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    assert dlib.fa_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, T, D, w.scale, causal, stream) == 0
    assert dlib.fa_bwd(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv), B, H, T, D, w.scale,
                       causal, stream) == 0
    assert dlib.fa_get_device_status(stream) == 0
    o2, lse2 = fa.attention_forward(q, k, v, causal=bool(causal), scale=w.scale)
    g2 = fa.attention_backward(q, k, v, o, lse, do, causal=bool(causal), scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert same_gradients((dq, dk, dv), g2, D)
