"""Bring-up checks of the hardware encodings the kernels rely on (test-only
libfa_probe.so): TMA 128-byte-swizzle tile loads with zero fill past the
tensor, and tcgen05.mma with K-major / MN-major shared-memory operands and an
A operand read from tensor memory, against a float64 matmul."""
import ctypes
import os

import numpy as np
import pytest
import torch

PKG = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "online_softmax_05_gb300")


@pytest.fixture(scope="module")
def plib():
    from online_softmax_05_gb300 import build
    build.build()
    lib = ctypes.CDLL(os.path.join(PKG, "libfa_probe.so"))
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.probe_mma.argtypes = [i, i, i, i, vp, vp, vp]
    lib.probe_mma.restype = i
    lib.probe_tma.argtypes = [vp, i, i, i, i, i, i, vp]
    lib.probe_tma.restype = i
    return lib


@pytest.mark.gpu
@pytest.mark.parametrize("a_mode,b_mode,N,K", [
    (0, 0, 128, 64), (0, 0, 128, 128), (0, 0, 64, 64), (0, 0, 64, 128),   # S = Q K^T form
    (0, 1, 128, 128), (0, 1, 64, 128),                                    # P V with V MN-major
    (2, 1, 128, 128), (2, 1, 64, 128), (2, 1, 128, 64),                   # P from TMEM
    (1, 1, 128, 128), (1, 1, 64, 128),                                    # dS^T stored, used as MN-major A
    (2, 0, 128, 128),
])
def test_mma_probe(plib, a_mode, b_mode, N, K):
    M = 128
    g = torch.Generator().manual_seed(1000 + 10 * a_mode + b_mode + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    A_glob = A.t().contiguous() if a_mode == 1 else A
    B_glob = B if b_mode == 1 else B.t().contiguous()
    dev = torch.device("cuda")
    a_d, b_d = A_glob.to(dev), B_glob.to(dev)
    out = torch.full((M, N), float("nan"), device=dev)
    rc = plib.probe_mma(a_mode, b_mode, N, K, a_d.data_ptr(), b_d.data_ptr(), out.data_ptr())
    assert rc == 0
    want = A.double().numpy() @ B.double().numpy()
    got = out.cpu().double().numpy()
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-3)


@pytest.mark.gpu
@pytest.mark.parametrize("D,row0,bh", [(128, 128, 1), (64, 0, 0), (64, 128, 1)])
def test_tma_probe_swizzle_and_zero_fill(plib, D, row0, bh):
    BH, T, box = 2, 200, 128
    x = torch.arange(BH * T * D, dtype=torch.int32).remainder(30000).to(torch.int16).reshape(BH, T, D)
    src = x.view(torch.bfloat16).cuda()
    dst = torch.zeros(box * D * 2, dtype=torch.uint8, device="cuda")
    assert plib.probe_tma(src.data_ptr(), BH, T, D, box, row0, bh, dst.data_ptr()) == 0
    got = dst.cpu().numpy().view(np.int16)
    want = np.zeros(box * D, dtype=np.int16)
    xs = x.numpy()
    for a in range(D // 64):
        for r in range(box):
            row = row0 + r
            for c in range(8):
                vals = xs[bh, row, 64 * a + 8 * c: 64 * a + 8 * c + 8] if row < T else np.zeros(8, np.int16)
                off = (a * box * 128 + r * 128 + ((c ^ (r % 8)) * 16)) // 2
                want[off:off + 8] = vals
    np.testing.assert_array_equal(got, want)


@pytest.mark.gpu
def test_tmem_16x256b_load_and_16x128b_store_layout(plib):
    """tcgen05.ld.16x256b.x8: thread t, register j = 4k + i holds lane
    t/4 (+8 for i >= 2), column 8k + 2 (t % 4) + (i % 2).
    tcgen05.st.16x128b.x8: thread t, register j = 2k + i lands in lane
    t/4 (+8 for i = 1), column 4k + t % 4."""
    ld = (ctypes.c_uint32 * (128 * 64))()
    st = (ctypes.c_uint32 * (128 * 32))()
    plib.probe_tmem_layout.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)]
    assert plib.probe_tmem_layout(ld, st) == 0
    ld = np.array(ld, dtype=np.uint32).reshape(4, 32, 2, 32)
    for w in range(4):
        for t in range(32):
            for half in range(2):
                for j in range(32):
                    k, i = divmod(j, 4)
                    lane = 32 * w + 16 * half + t // 4 + (8 if i >= 2 else 0)
                    col = 8 * k + 2 * (t % 4) + (i % 2)
                    assert ld[w, t, half, j] == (lane << 16) | col, (w, t, half, j, hex(ld[w, t, half, j]))
    st = np.array(st, dtype=np.uint32).reshape(128, 32)
    for w in range(4):
        for t in range(32):
            for j in range(16):
                k, i = divmod(j, 2)
                lane = 32 * w + t // 4 + (8 if i == 1 else 0)
                col = 4 * k + t % 4
                assert st[lane, col] == (w << 24) | (t << 16) | j, (w, t, j, hex(st[lane, col]))
