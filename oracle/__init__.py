"""CPU oracle for exact scaled-dot-product attention (fp64, naive, materialising).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never calls it; the oracle and the CUDA path share no code (only the
seeded input generators in ``online_softmax_05_gb300.inputs`` serve both).

The arithmetic lives in ``attn_ref.c`` (plain C + OpenMP, IEEE double,
compiled without fast-math and without FMA contraction); this module builds
it and marshals numpy arrays.  Each function names the page section it
follows (pages: "Lab 06 - Attention kernels: online softmax -> FlashAttention
-> Triton" sections 2-4; "Triton FlashAttention-2 forward", section "The
kernel"; "Flash Attention and Kernel Optimization", section "Causal masking").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.POINTER(ctypes.c_long)


def build(force: bool = False) -> str:
    """Compile attn_ref.c into liboracle.so (gcc, -O2, OpenMP, no fast-math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_online_softmax_stats.argtypes = [_D, ctypes.c_long, ctypes.c_long, _D, _D]
        lib.oracle_attn_fwd.argtypes = [_D, _D, _D, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                        ctypes.c_double, ctypes.c_int, _D, _D]
        lib.oracle_attn_probs.argtypes = [_D, _D, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                          ctypes.c_int, _D]
        lib.oracle_attn_bwd.argtypes = [_D, _D, _D, _D, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                        ctypes.c_double, ctypes.c_int, _D, _D, _D, _D]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd_rows.argtypes = [_D, _D, _D, _D, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_long, _L, ctypes.c_long, _L,
                                             _D, _D, _D, _D, _D]
        lib.oracle_attn_bwd_rows.restype = ctypes.c_int
        lib.oracle_attn_fwd_rows.argtypes = [_D, _D, _D, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_long, _L, _D, _D]
        lib.oracle_attn_fwd_cross.argtypes = [_D, _D, _D, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                              ctypes.c_double, _D, _D]
        lib.oracle_flash_fwd_tiled.argtypes = [_D, _D, _D, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                               ctypes.c_int, ctypes.c_long, ctypes.c_long, _D, _D]
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _lp(a: np.ndarray):
    return a.ctypes.data_as(_L)


def num_threads() -> int:
    """OpenMP threads the oracle uses (set OMP_NUM_THREADS to change)."""
    return int(_load().oracle_num_threads())


def online_softmax_stats(x, block: int):
    """Running (m, l) over ``x`` visited in blocks ("Lab 06", section 2).

    Returns (m, l) with logsumexp(x) = m + log(l).
    """
    x = _f64(x).ravel()
    m = np.zeros(1)
    l = np.zeros(1)
    _load().oracle_online_softmax_stats(_p(x), x.size, int(block), _p(m), _p(l))
    return float(m[0]), float(l[0])


def attn_fwd(q, k, v, scale: float, causal: bool):
    """Naive forward over [..., T, D] inputs; returns (O [..., T, D], LSE [..., T]).

    "Lab 06", sections 1 and 3 (definition the tiled recurrence reaches).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, D = q.shape[-2], q.shape[-1]
    nbh = q.size // (T * D) if q.size else 0
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:-1])
    if nbh:
        _load().oracle_attn_fwd(_p(q), _p(k), _p(v), nbh, T, D, float(scale), int(bool(causal)), _p(o), _p(lse))
    return o, lse


def attn_probs(q, k, scale: float, causal: bool) -> np.ndarray:
    """Materialised P [T, T] of one head (rows sum to 1, masked entries 0)."""
    q, k = _f64(q), _f64(k)
    T, D = q.shape
    P = np.zeros((T, T))
    _load().oracle_attn_probs(_p(q), _p(k), T, D, float(scale), int(bool(causal)), _p(P))
    return P


def attn_bwd(q, k, v, dout, scale: float, causal: bool):
    """Analytic gradients ("Lab 06", section 4); returns (dQ, dK, dV, Dvec)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, D = q.shape[-2], q.shape[-1]
    nbh = q.size // (T * D) if q.size else 0
    dq, dk, dv = np.zeros(q.shape), np.zeros(q.shape), np.zeros(q.shape)
    dvec = np.zeros(q.shape[:-1])
    if nbh:
        rc = _load().oracle_attn_bwd(_p(q), _p(k), _p(v), _p(dout), nbh, T, D, float(scale), int(bool(causal)),
                                     _p(dq), _p(dk), _p(dv), _p(dvec))
        if rc != 0:
            raise MemoryError("oracle_attn_bwd: could not allocate T x T scratch")
    return dq, dk, dv, dvec


def attn_fwd_rows(q, k, v, scale: float, causal: bool, rows):
    """O and LSE of selected rows of ONE head [T, D]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, D = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.zeros((rows.size, D))
    lse = np.zeros(rows.size)
    _load().oracle_attn_fwd_rows(_p(q), _p(k), _p(v), T, D, float(scale), int(bool(causal)), rows.size,
                                 _lp(rows), _p(o), _p(lse))
    return o, lse


def attn_bwd_rows(q, k, v, dout, scale: float, causal: bool, rows_q, rows_k):
    """Selected rows of dQ (rows_q) and dK/dV (rows_k) of ONE head, plus LSE and D of every row."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, D = q.shape
    rq = np.ascontiguousarray(np.asarray(rows_q, dtype=np.int64))
    rk = np.ascontiguousarray(np.asarray(rows_k, dtype=np.int64))
    dq = np.zeros((rq.size, D))
    dk = np.zeros((rk.size, D))
    dv = np.zeros((rk.size, D))
    lse = np.zeros(T)
    dvec = np.zeros(T)
    _load().oracle_attn_bwd_rows(_p(q), _p(k), _p(v), _p(dout), T, D, float(scale), int(bool(causal)),
                                 rq.size, _lp(rq), rk.size, _lp(rk), _p(dq), _p(dk), _p(dv), _p(lse), _p(dvec))
    return dq, dk, dv, lse, dvec


def flash_fwd_tiled(q, k, v, scale: float, causal: bool, bq: int, bk: int):
    """The tiled online-softmax forward of "Lab 06", section 3, for ONE head, in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, D = q.shape
    o = np.zeros((T, D))
    lse = np.zeros(T)
    _load().oracle_flash_fwd_tiled(_p(q), _p(k), _p(v), T, D, float(scale), int(bool(causal)), int(bq), int(bk),
                                   _p(o), _p(lse))
    return o, lse


def attn_fwd_cross(q, k, v, scale: float):
    """Tq queries attend to all Tk keys of their head, no mask ([..., Tq, D] / [..., Tk, D]).

    "Lab 06", "Check yourself" item 2 (decoding against a long cache)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, D = q.shape[-2], q.shape[-1]
    Tk = k.shape[-2]
    nbh = q.size // (Tq * D) if q.size else 0
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:-1])
    if nbh:
        _load().oracle_attn_fwd_cross(_p(q), _p(k), _p(v), nbh, Tq, Tk, D, float(scale), _p(o), _p(lse))
    return o, lse


def attn_fwd_gqa(q, k, v, scale: float, causal: bool):
    """Grouped-query forward: q [B, Hq, T, D], k/v [B, Hkv, T, D], query head h
    using key/value head h // (Hq // Hkv) ("Lab 06", "Check yourself" item 7).
    By definition: repeat each key/value head over its group, then attn_fwd."""
    g = q.shape[1] // k.shape[1]
    return attn_fwd(q, np.repeat(_f64(k), g, axis=1), np.repeat(_f64(v), g, axis=1), scale, causal)


def attn_bwd_gqa(q, k, v, dout, scale: float, causal: bool):
    """Gradients of the grouped-query forward: those of the repeated problem,
    with dK and dV summed over the query heads of each group."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    dq, dk_r, dv_r, dvec = attn_bwd(q, np.repeat(_f64(k), g, axis=1), np.repeat(_f64(v), g, axis=1), dout, scale,
                                    causal)
    return dq, dk_r.reshape(B, Hkv, g, T, D).sum(axis=2), dv_r.reshape(B, Hkv, g, T, D).sum(axis=2), dvec


def attn_bwd_varlen(q, k, v, dout, cu_seqlens, scale: float, causal: bool):
    """Gradients of attn_fwd_varlen: q/k/v/dout [total, H, D].  By definition:
    attn_bwd on each sequence's slice (no row of one sequence depends on
    another's).  Returns (dQ, dK, dV), each [total, H, D]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    total, H, D = q.shape
    cu = [int(c) for c in np.asarray(cu_seqlens).ravel()]
    dq, dk, dv = np.zeros((total, H, D)), np.zeros((total, H, D)), np.zeros((total, H, D))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if b <= a:
            continue
        t = lambda x: x[a:b].transpose(1, 0, 2)
        g = attn_bwd(t(q), t(k), t(v), t(dout), scale, causal)
        dq[a:b], dk[a:b], dv[a:b] = (x.transpose(1, 0, 2) for x in g[:3])
    return dq, dk, dv


def attn_fwd_varlen(q, k, v, cu_seqlens, scale: float, causal: bool):
    """Packed variable-length forward: q/k/v [total, H, D]; sequence s is rows
    cu_seqlens[s]:cu_seqlens[s+1] and attends only to itself, causal mask
    aligned to its own first token ("Triton FlashAttention-2 forward",
    "Exercises", the cu_seqlens packing).  By definition: attn_fwd on each
    sequence's slice.  Returns (O [total, H, D], LSE [H, total])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    total, H, D = q.shape
    cu = [int(c) for c in np.asarray(cu_seqlens).ravel()]
    o = np.zeros((total, H, D))
    lse = np.zeros((H, total))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if b <= a:
            continue
        os_, ls_ = attn_fwd(q[a:b].transpose(1, 0, 2), k[a:b].transpose(1, 0, 2), v[a:b].transpose(1, 0, 2),
                            scale, causal)
        o[a:b] = os_.transpose(1, 0, 2)
        lse[:, a:b] = ls_
    return o, lse
