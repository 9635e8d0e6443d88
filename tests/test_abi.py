"""The C-ABI library loads, exports every symbol include/fa.h declares, and
rejects bad arguments with the documented codes before touching a GPU."""
import ctypes
import os
import re

import pytest

import online_softmax_05_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fa_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from online_softmax_05_gb300 import build
    build.build()
    return fa.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_strerror", "fa_get_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_covers_codes(lib):
    for code in range(0, -13, -1):
        s = fa.fa_strerror(code)
        assert s and "unknown" not in s
    assert "unknown" in fa.fa_strerror(-1234)


def _fwd(**kw):
    a = dict(q=0x1000, k=0x2000_0000, v=0x4000_0000, o=0x6000_0000, lse=0x8000_0000, B=1, H=1, T=16, D=64,
             scale=0.125, causal=0)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["T"], a["D"], a["scale"],
                     a["causal"], None)


def _bwd(**kw):
    base = 0x1000_0000
    a = dict(q=base, k=2 * base, v=3 * base, o=4 * base, dO=5 * base, lse=6 * base, dq=7 * base, dk=8 * base,
             dv=9 * base, B=1, H=1, T=16, D=128, scale=0.1, causal=1)
    a.update(kw)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["dO"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"],
                     a["H"], a["T"], a["D"], a["scale"], a["causal"], None)


def test_argument_errors_fwd(lib):
    assert _fwd(q=None) == -1
    assert _fwd(lse=None) == -1
    assert _fwd(B=0) == -2
    assert _fwd(T=0) == -2
    assert _fwd(H=-3) == -2
    assert _fwd(B=1 << 16, H=1 << 16, T=1) == -2
    assert _fwd(D=96) == -3
    assert _fwd(D=256) == -3
    assert _fwd(q=0x1008) == -4
    assert _fwd(causal=2) == -8
    assert _fwd(scale=float("nan")) == -8
    assert _fwd(scale=float("inf")) == -8
    assert _fwd(o=0x1000) == -8          # output aliases q
    assert _fwd(lse=0x6000_0010) == -8   # lse inside o


def test_argument_errors_bwd(lib):
    assert _bwd(dv=None) == -1
    assert _bwd(T=0) == -2
    assert _bwd(D=32) == -3
    assert _bwd(dk=0x8000_0004) == -4
    assert _bwd(causal=-1) == -8
    assert _bwd(dq=0x1000_0000) == -8     # dq aliases q
    assert _bwd(dk=0x7000_0000) == -8     # dk aliases dq


def test_tile_rows(lib):
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert lib.fa_sched_tile_rows(128, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == 0
    assert (a.value, b.value, c.value) == (128, 128, 128)
    assert lib.fa_sched_tile_rows(64, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == 0
    assert (a.value, b.value, c.value) == (128, 128, 128)
    assert lib.fa_sched_tile_rows(80, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == -3


def test_debug_knob_validation(lib):
    assert lib.fa_debug_set_wait_timeout_ns(0) == -8
    assert lib.fa_debug_inject(7) == -8
    assert lib.fa_debug_inject(0) == 0
    assert lib.fa_debug_set_wait_timeout_ns(2_000_000_000) == 0
    assert lib.fa_set_deterministic(2) == -8
    assert lib.fa_set_deterministic(0) == 0


def test_backward_plan_query_argument_errors(lib):
    # host-only: sizes are checked before the device is looked at
    assert lib.fa_bwd_sums_dq_in_place(0, 1, 128, 64) == -2
    assert lib.fa_bwd_sums_dq_in_place(1, 1, 0, 64) == -2
    assert lib.fa_bwd_sums_dq_in_place(1, 1, 128, 96) == -3


def test_argument_errors_decode(lib):
    base = 0x1000_0000
    q, k, v, o, lse = base, 2 * base, 3 * base, 4 * base, 5 * base
    f = lambda **kw: fa.fa_decode(kw.get("q", q), k, v, kw.get("o", o), lse, kw.get("B", 1), 2, kw.get("Tq", 1),
                                  kw.get("Tk", 100), kw.get("D", 128), kw.get("scale", 0.1), None)
    assert f(q=None) == -1
    assert f(Tq=0) == -2
    assert f(Tk=0) == -2
    assert f(Tq=9) == -3
    assert f(D=96) == -3
    assert f(scale=float("nan")) == -8
    assert f(q=base + 8) == -4
    assert f(o=q) == -8


def test_argument_errors_gqa(lib):
    base = 0x1000_0000
    p = [base * (i + 1) for i in range(9)]
    assert fa.fa_fwd_gqa(p[0], p[1], p[2], p[3], p[4], 1, 6, 4, 64, 128, 0.1, 0, None) == -2   # 6 % 4 != 0
    assert fa.fa_fwd_gqa(p[0], p[1], p[2], p[3], p[4], 1, 4, 0, 64, 128, 0.1, 0, None) == -2
    assert fa.fa_bwd_gqa(*p, 1, 4, 8, 64, 128, 0.1, 0, None) == -2                               # Hkv > Hq
    assert fa.fa_bwd_gqa(*p[:8], None, 1, 4, 2, 64, 128, 0.1, 0, None) == -1


def test_argument_errors_varlen(lib):
    base = 0x1000_0000
    q, k, v, o, lse, cu = (base * (i + 1) for i in range(6))
    f = lambda **kw: fa.fa_fwd_varlen(kw.get("q", q), k, v, kw.get("o", o), lse, kw.get("cu", cu),
                                      kw.get("n_seq", 3), kw.get("max_seqlen", 100), kw.get("total", 250), 2,
                                      kw.get("D", 128), kw.get("scale", 0.1), kw.get("causal", 1), None)
    assert f(cu=None) == -1
    assert f(n_seq=0) == -2
    assert f(max_seqlen=0) == -2
    assert f(total=0) == -2
    assert f(D=80) == -3
    assert f(causal=2) == -8
    assert f(scale=float("inf")) == -8
    assert f(cu=cu + 2) == -4
    assert f(q=base + 8) == -4
    assert f(o=k) == -8


def test_argument_errors_bwd_varlen(lib):
    base = 0x1000_0000
    p = [base * (i + 1) for i in range(10)]   # q k v o dO lse dq dk dv cu

    def f(**kw):
        a = dict(zip("q k v o dO lse dq dk dv cu".split(), p))
        a.update(kw)
        return fa.fa_bwd_varlen(a["q"], a["k"], a["v"], a["o"], a["dO"], a["lse"], a["dq"], a["dk"], a["dv"], a["cu"],
                                a.get("n_seq", 3), a.get("max_seqlen", 100), a.get("total", 250), 2, a.get("D", 128),
                                a.get("scale", 0.1), a.get("causal", 0), None)
    assert f(cu=None) == -1
    assert f(dq=None) == -1
    assert f(n_seq=0) == -2
    assert f(max_seqlen=-1) == -2
    assert f(total=0) == -2
    assert f(D=96) == -3
    assert f(cu=p[9] + 1) == -4
    assert f(dk=p[7] + 8) == -4
    assert f(causal=3) == -8
    assert f(scale=float("nan")) == -8
    assert f(dq=p[0]) == -8          # dq aliases q
    assert f(dv=p[7]) == -8          # dv aliases dk
