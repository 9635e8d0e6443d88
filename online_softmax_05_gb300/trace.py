"""Pipeline cycle traces of the attention kernels (a developer tool).

    python -m online_softmax_05_gb300.trace [--B 2 --H 16 --T 8192 --D 128 --causal 1]

Builds a second copy of the library with the kernels' trace hooks compiled in
(-DFA_TRACE; the product library has none), runs one forward and one backward
on seeded inputs, and prints:

  * forward: per key-tile step of the first CTA's first work item, the median
    period and the offsets of the MMA warp's and softmax warpgroups' events;
  * dK/dV and dQ kernels: per query / key tile of the first CTA, the median
    period and the offsets of the MMA and compute warps' events;
  * per-CTA timeline of both backward grids (global timer): span, mean CTA
    duration, time after the last MMA issue, idle tail, and for the dK/dV
    grid a least-squares fit duration = a + b * query tiles.

Stamps are clock64 cycles of one SM (trace slots) or global-timer
nanoseconds (timeline); the traced build runs slightly slower than the
product library.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import subprocess

import numpy as np

from . import build as _b

TRACE_LIB = os.path.join(_b.BUILD, "libfa_trace.so")
FWD_SLOTS = ["mma P0 seen", "mma P1 seen", "mma S0 issued", "mma S1 issued", "sm0 S seen", "sm1 S seen",
             "sm0 max", "sm1 max", "sm0 P released", "sm1 P released", "sm0 warp3 P", "sm1 warp3 P"]
DKV_SLOTS = {0: "mma top", 1: "mma P^T seen", 7: "mma dV issued", 2: "mma S^T issued", 10: "mma dS^T seen",
             11: "mma dK issued", 8: "mma dP^T issued", 3: "cmp S^T seen", 4: "cmp P^T stored", 5: "cmp dP^T seen",
             6: "cmp dS^T stored"}
DQ_SLOTS = {12: "mma top", 13: "mma dS seen", 18: "mma dP issued", 19: "mma dQ issued", 14: "mma S issued",
            15: "cmp S seen", 16: "cmp dP seen", 17: "cmp dS stored"}


def build_trace_lib() -> str:
    os.makedirs(_b.BUILD, exist_ok=True)
    objs = []
    procs = []
    for unit in _b.PRODUCT_UNITS:
        obj = os.path.join(_b.BUILD, unit.replace(".cu", ".trace.o"))
        cmd = [_b.nvcc()] + _b.NVCC_FLAGS + ["-DFA_TRACE", "-c", os.path.join(_b.CSRC, unit), "-o", obj]
        procs.append((unit, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
        objs.append(obj)
    for unit, pr in procs:
        out, err = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError(f"nvcc failed for {unit}:\n{out}\n{err}")
    cmd = [_b.nvcc()] + _b.ARCH + ["-shared", "-cudart", "shared", "-o", TRACE_LIB] + objs
    subprocess.run(cmd, check=True, capture_output=True)
    return TRACE_LIB


def _offsets(tr, slots, ref, n):
    out = []
    for s, name in slots.items():
        d = tr[s][1:n - 1] - tr[ref][1:n - 1]
        out.append(f"    {name:16s} {np.median(d):8.0f}")
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--causal", type=int, default=1)
    a = ap.parse_args(argv)
    import torch
    lib = ctypes.CDLL(build_trace_lib())
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp] * 5 + [i] * 4 + [f, i, vp]
    lib.fa_bwd.argtypes = [vp] * 9 + [i] * 4 + [f, i, vp]
    B, H, T, D, causal = a.B, a.H, a.T, a.D, a.causal
    g = torch.Generator(device="cpu").manual_seed(0)
    q, k, v, do = (torch.randn(B, H, T, D, generator=g).to(torch.bfloat16).cuda() for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    sc = D ** -0.5
    for _ in range(2):
        assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, T, D, sc, causal, None) == 0
    torch.cuda.synchronize()
    fbuf = (ctypes.c_ulonglong * (20 * 128))()
    assert lib.fa_ftrace_read(fbuf) == 0
    ft = np.array(fbuf, dtype=np.int64).reshape(20, 128)
    for _ in range(2):
        assert lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, T, D, sc, causal, None) == 0
    torch.cuda.synchronize()
    bbuf = (ctypes.c_ulonglong * (28 * 512))()
    assert lib.fa_trace_read(bbuf) == 0
    bt = np.array(bbuf, dtype=np.int64).reshape(28, 512)
    cbuf = (ctypes.c_ulonglong * (2 * 8192 * 4))()
    assert lib.fa_cta_trace_read(cbuf) == 0
    ct = np.array(cbuf, dtype=np.int64).reshape(2, 8192, 4)

    print(f"B={B} H={H} T={T} D={D} causal={causal}  (cycles unless stated)")
    n = int((ft[0] != 0).sum())
    if n > 3:
        print(f"forward, first CTA's first item: {n} key-tile steps, period median "
              f"{np.median(np.diff(ft[0][:n])):.0f}; offsets from 'mma P0 seen':")
        print("\n".join(_offsets(ft, dict(enumerate(FWD_SLOTS)), 0, n)))
    for title, slots, ref, count in (("dK/dV", DKV_SLOTS, 0, 11), ("dQ", DQ_SLOTS, 12, 14)):
        n = int((bt[count] != 0).sum())
        if n > 3:
            per = np.diff(bt[ref][:n])
            print(f"{title} kernel, first CTA: {n} tiles traced, period median {np.median(per):.0f}; "
                  f"offsets from '{slots[ref]}':")
            print("\n".join(_offsets(bt, slots, ref, n)))
    n_kt = (T + 127) // 128
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    for kern, name, n_cta in ((0, "dK/dV", n_kt * B * H), (1, "dQ", min(n_kt * B * H, n_sm))):
        t = ct[kern, :min(n_cta, 8192)]
        t = t[t[:, 1] != 0]
        if len(t) == 0:
            continue
        sm, t0, tl, t1 = t[:, 0], t[:, 1], t[:, 2], t[:, 3]
        span = (t1.max() - t0.min()) / 1e3
        dur = (t1 - t0) / 1e3
        idle = [(t1.max() - t1[sm == s].max()) / 1e3 for s in np.unique(sm)]
        print(f"{name} grid timeline (us): {len(t)} CTAs, span {span:.1f}, CTA duration mean {dur.mean():.2f}, "
              f"after last MMA issue mean {((t1 - tl) / 1e3).mean():.2f}, idle tail mean {np.mean(idle):.1f}")
        if kern == 0 and len(t) == n_cta:
            bh_major = n_kt * B * H >= 8 * n_sm  # the grid's CTA order (key tile major below 8 waves)
            idx = np.arange(n_cta)
            kt = (idx % n_kt) if bh_major else (idx // (B * H))
            n_it = (n_kt - kt) if causal else np.full(n_cta, n_kt)
            coef, *_ = np.linalg.lstsq(np.stack([np.ones(n_cta), n_it], 1), dur, rcond=None)
            print(f"  fit: CTA duration = {coef[0]:.2f} us + {coef[1] * 1e3:.1f} ns x query tiles")


if __name__ == "__main__":
    main()
