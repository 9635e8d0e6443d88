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
def test_mma_chain_length_report(plib, capsys):
    """Cycles per 128xNx16 bf16 tcgen05.mma when n = 256 instructions run as
    chains of `chain` instructions on one accumulator, alternating between two
    accumulators chain by chain (the shape of the attention kernels' products:
    a chain per product, K / 16 instructions long).  Checks the long chains
    of the dense K-major form stream within 30 % of 8192 FLOP/clk."""
    plib.probe_mma_chain.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_longlong)]
    kinds = {0: "SS, A and B K-major", 1: "SS, A K-major, B MN-major", 2: "TS (A in TMEM), B MN-major"}
    rows = []
    for N in (64, 128):
        for kind in kinds:
            for chain in (1, 2, 4, 8, 16, 32):
                o = (ctypes.c_longlong * 1)()
                assert plib.probe_mma_chain(N, 256, chain, kind, o) == 0
                assert plib.probe_mma_chain(N, 256, chain, kind, o) == 0
                rows.append((N, kinds[kind], chain, o[0] / 256.0))
    with capsys.disabled():
        print("\n  N  form                          chain  cycles/MMA")
        for N, name, chain, c in rows:
            print(f"{N:4d}  {name:28s} {chain:6d} {c:10.1f}")
    for N, name, chain, c in rows:
        if N == 128 and name == kinds[0] and chain == 32:
            assert c <= 1.3 * 64


@pytest.mark.gpu
def test_mma_sequence_report(plib, capsys):
    """Cycles per 128x128x16 MMA for loops of three 8-instruction chains shaped
    like the attention kernels' (see probe_mma_seq_kernel): plain, with a
    commit after each chain, with commit + satisfied wait + fence, and the
    dQ kernel's SS / TS / SS rotation; on one SM and on every SM at once.
    Then the first and the fourth with pseudo-random operands instead of 1.0
    everywhere, and the wait / fence pair taken apart: the wait alone, the
    fence alone, and the wait issued before the last two MMAs of the
    previous chain; then the loop run by the whole warp with elect.sync
    choosing the issuing lane, and descriptor offsets known only at run
    time (as the kernels' ring stages are); and the warp-wide dQ loop while
    the other three warps stream TMEM loads or shared-memory loads."""
    import torch
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    plib.probe_mma_seq.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_longlong)]
    names = {0: "3 accumulators, SS chains", 1: "+ commit after each chain",
             2: "+ satisfied wait and fence", 3: "dQ loop: SS, TS, SS",
             4: "3 accumulators, random operands", 7: "dQ loop, random operands",
             2 | 8: "wait without fence", 2 | 16: "fence without wait",
             2 | 24: "wait early, fence after chain", 3 | 24: "dQ loop, wait early",
             2 | 32: "wait + fence, whole warp", 3 | 32: "dQ loop, whole warp",
             2 | 64: "wait + fence, run-time offsets", 3 | 64: "dQ loop, run-time offsets",
             2 | 96: "whole warp, run-time offsets", 3 | 96: "dQ loop, warp, run-time offsets",
             3 | 120: "dQ loop, warp, rt off, early",
             3 | 96 | 128: "dQ loop (warp) + TMEM loads", 3 | 96 | 256: "dQ loop (warp) + smem loads"}
    res = {}
    for ctas, n_iter in ((1, 32), (n_sm, 32), (n_sm, 2048)):
        for mode in names:
            o = (ctypes.c_longlong * ctas)()
            assert plib.probe_mma_seq(mode, n_iter, ctas, o) == 0
            assert plib.probe_mma_seq(mode, n_iter, ctas, o) == 0
            res[(ctas, n_iter, mode)] = float(np.median(np.array(o[:])) / (n_iter * 24))
    with capsys.disabled():
        print(f"\n  loop                              1 SM   {n_sm} SMs  {n_sm} SMs x 2048 iterations")
        for mode, name in names.items():
            print(f"  {name:32s} {res[(1, 32, mode)]:6.1f} {res[(n_sm, 32, mode)]:8.1f} {res[(n_sm, 2048, mode)]:8.1f}")
    assert res[(1, 32, 0)] <= 1.3 * 64



@pytest.mark.gpu
def test_exp2_and_bf16_pack_rate_report(plib, capsys):
    """Throughput on one SM (1 to 32 warps) of the softmax's special-function
    work (see probe_exp2_rate_kernel): ex2.approx alone, exp2 as an FMA
    polynomial, cvt.rn.bf16x2.f32 packs alone, and ex2 with packs in the
    softmax's 2:1 mix.  Reported as operations per clock per SM; in the mixed
    mode an ex2 and half a pack count as one step, so if the packs took no
    issue or pipe time of their own it would match the ex2-alone rate."""
    plib.probe_exp2_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_longlong),
                                     ctypes.c_void_p]
    iters = 256
    ops = {0: 8, 1: 8, 2: 4, 3: 8}   # counted operations per round per thread
    names = {0: "ex2.approx", 1: "exp2 polynomial (FMA)", 2: "bf16x2 pack", 3: "ex2 + pack (2:1)"}
    res = {}
    for warps in (4, 8, 16, 32):
        for mode in names:
            o = (ctypes.c_longlong * 32)()
            assert plib.probe_exp2_rate(mode, iters, warps, o, None) == 0
            assert plib.probe_exp2_rate(mode, iters, warps, o, None) == 0
            cyc = max(o[:warps])
            res[(warps, mode)] = warps * 32 * iters * ops[mode] / cyc
    with capsys.disabled():
        print("\n  per SM and clock           4 warps  8 warps 16 warps 32 warps")
        for mode, name in names.items():
            print(f"  {name:24s}" + "".join(f"{res[(w, mode)]:9.1f}" for w in (4, 8, 16, 32)))
    assert all(v > 0 for v in res.values())

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
