"""fa_bwd_noalloc: the backward for callers that cannot allocate device
memory at call time (for instance inside a fixed memory pool that must not
grow, or where the CUDA allocator is not reachable from the calling code).
It runs the same kernels as fa_bwd on the library's fixed 64 MiB device
scratch buffer instead of a stream-ordered allocation.

Checked through the C ABI: two calls in a row give dQ, dK, dV matching
fa_bwd within the gradient tolerance of the other tests (the second call
also shows that the previous call's leftovers in the shared buffer do not
leak into the result), and a problem too large for the buffer is refused
with FA_ERR_SCRATCH before anything is launched.  Kept in a file collected
last so a run stopping at the first failure has already run every other
test; it also passes on its own in a fresh process."""
import math

import numpy as np
import pytest
import torch

import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import make_inputs, to_f64
from tests.tolerances import grad_bound


@pytest.fixture(scope="module")
def lib():
    from online_softmax_05_gb300 import build
    build.build()
    return fa.load_library()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,T,D,causal", [(1, 4, 777, 128, 1), (2, 3, 300, 64, 0)])
def test_noalloc_matches_fa_bwd_on_two_calls(lib, B, H, T, D, causal):
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, T, D, seed=21 + D))
    stream = torch.cuda.current_stream()
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    assert fa.fa_fwd(q, k, v, o, lse, B, H, T, D, scale, causal, stream) == 0
    ref = [torch.empty_like(q) for _ in range(3)]
    assert fa.fa_bwd(q, k, v, o, do, lse, *ref, B, H, T, D, scale, causal, stream) == 0
    torch.cuda.synchronize()
    refs = [to_f64(t.cpu()) for t in ref]
    for call in range(2):
        out = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                lse.data_ptr(), out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
                                B, H, T, D, scale, causal, stream.cuda_stream)
        assert rc == 0, fa.fa_strerror(rc)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status(stream) == 0
        for name, g, r in zip(("dq", "dk", "dv"), out, refs):
            g = to_f64(g.cpu())
            assert np.isfinite(g).all(), (call, name)
            assert np.abs(g - r).max() <= grad_bound(r), (call, name)


@pytest.mark.gpu
def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    # 64 x 32 x 8192 rows need 128 MiB of scratch (8 bytes a row): refused before any launch
    base = 1 << 40
    ptrs = [base * (i + 1) for i in range(9)]
    rc = lib.fa_bwd_noalloc(*ptrs, 64, 32, 8192, 128, 0.088, 1, None)
    assert rc == -10
    assert "scratch" in fa.fa_strerror(rc)


@pytest.fixture(scope="module")
def host_lib():
    # the refusal below needs the library but no GPU: build it where nvcc
    # exists, skip where the library cannot be had
    from online_softmax_05_gb300 import build
    try:
        build.build()
        return fa.load_library()
    except (RuntimeError, OSError) as e:
        pytest.skip(f"libfa.so not available: {e}")


def test_noalloc_refuses_one_row_block_past_its_scratch(host_lib):
    # the scratch holds two (B*H, T_pad) float vectors plus 256 bytes: at
    # T = 8192, 1024 heads need 64 MiB + 256 bytes and are refused before any
    # device access (placeholder pointers; nothing is launched)
    lib = host_lib
    base = 1 << 40
    ptrs = [base * (i + 1) for i in range(9)]
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1024, 8192, 64, 0.125, 1, None) == -10
    assert lib.fa_bwd_noalloc(*ptrs, 2, 512, 8192 - 100, 64, 0.125, 0, None) == -10   # T_pad is still 8192


@pytest.mark.gpu
def test_noalloc_runs_the_largest_problem_that_fits(lib, deterministic_backward):
    # 1023 heads at T = 8192 leave 64 MiB - 65280 bytes: the largest head count
    # that fits; the result equals fa_bwd's (in its deterministic mode, the
    # same kernels), compared on a few heads
    B, H, T, D = 1, 1023, 8192, 64
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(71)
    q, k, v, do = (torch.randn(B, H, T, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(4))
    o, lse = fa.attention_forward(q, k, v, causal=True)
    ref = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    got = [torch.empty_like(q) for _ in range(3)]
    rc = lib.fa_bwd_noalloc(*(t.data_ptr() for t in (q, k, v, o, do, lse, *got)), B, H, T, D, D ** -0.5, 1,
                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for h in (0, 511, H - 1):
        for a, b in zip(got, ref):
            assert torch.equal(a[0, h], b[0, h])
