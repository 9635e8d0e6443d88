"""The kernels' causal tile skip, tile classes and element masks, evaluated
through the library's host-side schedule queries, equal a brute-force mask
bit for bit ("Lab 06", section 3 and "Common bugs": skip, full and diag
tiles; the last key tile needed holds the tile's last row; keys >= T masked).
"""
import ctypes

import numpy as np
import pytest

import online_softmax_05_gb300 as fa


@pytest.fixture(scope="module")
def lib():
    from online_softmax_05_gb300 import build
    build.build()
    return fa.load_library()


def tiles(lib, D):
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert lib.fa_sched_tile_rows(D, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == 0
    return a.value, b.value, c.value


def brute_visible(T, causal, n_rows, n_keys, pad_rows_visible):
    i = np.arange(n_rows)[:, None]
    j = np.arange(n_keys)[None, :]
    vis = (j < T) & (i >= 0)
    if causal:
        vis = vis & (j <= i)
    if not pad_rows_visible:
        vis = vis & (i < T)
    return vis


T_VALUES = [1, 2, 7, 33, 63, 64, 65, 127, 128, 129, 191, 200, 255, 256, 257, 300, 383, 513]


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("T", T_VALUES)
def test_forward_keep_equals_brute_force(lib, T, causal):
    bm, bn, _ = tiles(lib, 64)
    n_rows = -(-T // bm) * bm
    n_keys = -(-T // bn) * bn
    got = np.array([[lib.fa_sched_fwd_keep(T, causal, i, j) for j in range(n_keys)] for i in range(n_rows)])
    want = brute_visible(T, causal, n_rows, n_keys, pad_rows_visible=True)
    # rows past T are padding: only rows < T are specified
    np.testing.assert_array_equal(got[:T], want[:T].astype(int))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("T", T_VALUES)
def test_backward_keep_equals_brute_force(lib, T, causal, D):
    _, bn, bmb = tiles(lib, D)
    n_rows = -(-T // bmb) * bmb
    n_keys = -(-T // bn) * bn
    got = np.array([[lib.fa_sched_bwd_keep(T, D, causal, i, j) for j in range(n_keys)] for i in range(n_rows)])
    want = brute_visible(T, causal, n_rows, n_keys, pad_rows_visible=False)
    np.testing.assert_array_equal(got, want.astype(int))


def tile_class_brute(vis_tile):
    if not vis_tile.any():
        return 0
    return 1 if vis_tile.all() else 2


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("T", T_VALUES)
def test_forward_tile_classes_are_exact(lib, T, causal):
    # skip iff no real row sees a key of the tile; full iff every real row sees every key
    bm, bn, _ = tiles(lib, 64)
    nq, nk = -(-T // bm), -(-T // bn)
    vis = brute_visible(T, causal, nq * bm, nk * bn, pad_rows_visible=True)
    for qt in range(nq):
        rows = slice(qt * bm, min((qt + 1) * bm, T))
        for kt in range(nk + 1):
            want = 0 if kt >= nk else tile_class_brute(vis[rows, kt * bn:(kt + 1) * bn])
            assert lib.fa_sched_fwd_tile_class(T, causal, qt, kt) == want, (qt, kt)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("T", T_VALUES)
def test_backward_tile_classes_are_exact(lib, T, causal, D):
    _, bn, bmb = tiles(lib, D)
    nq, nk = -(-T // bmb), -(-T // bn)
    vis = brute_visible(T, causal, nq * bmb, nk * bn, pad_rows_visible=False)
    for kt in range(nk + 1):
        for qt in range(nq + 1):
            if kt >= nk or qt >= nq:
                want = 0
            else:
                want = tile_class_brute(vis[qt * bmb:(qt + 1) * bmb, kt * bn:(kt + 1) * bn])
            assert lib.fa_sched_bwd_tile_class(T, D, causal, qt, kt) == want, (qt, kt)


def test_causal_skip_halves_the_work(lib):
    # "about half the work": visited tile pairs at T = 8192 vs the full grid
    T = 8192
    bm, bn, _ = tiles(lib, 128)
    n = T // bm
    visited = sum(lib.fa_sched_fwd_tile_class(T, 1, qt, kt) != 0 for qt in range(n) for kt in range(n))
    assert visited == n * (n + 1) // 2
