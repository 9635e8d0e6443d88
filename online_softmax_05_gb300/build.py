"""Build the CUDA libraries in-tree with nvcc for sm_103a.

  libfa.so        the product: C-ABI entry points of include/fa.h
  libfa_debug.so  the same sources built with -DFA_DEBUG: every kernel checks
                  its run-time tile, ring-stage, vector and tensor-memory
                  indices before use and reports FA_ERR_DEBUG_CHECK instead of
                  touching memory out of bounds (tests only; slower)
  libfa_probe.so  test-only bring-up kernels (descriptor / TMA / TMEM layout checks)

Translation units compile in parallel; a unit is rebuilt only when its
source or any header under csrc/ or include/ is newer than its object.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")

LIB = os.path.join(PKG, "libfa.so")
DEBUG_LIB = os.path.join(PKG, "libfa_debug.so")
PROBE_LIB = os.path.join(PKG, "libfa_probe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     f"-I{INCLUDE}", f"-I{CSRC}", "--expt-relaxed-constexpr"]

PRODUCT_UNITS = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_decode.cu"]
PROBE_UNITS = ["fa_probe.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def _compile(unit: str, extra: list[str], force: bool, verbose: bool, debug: bool = False) -> str:
    src = os.path.join(CSRC, unit)
    obj = os.path.join(BUILD, unit.replace(".cu", ".debug.o" if debug else ".o"))
    if debug:
        extra = extra + ["-DFA_DEBUG"]
    if (not force and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime())):
        return obj
    cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj + ".tmp"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {unit}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    os.replace(obj + ".tmp", obj)
    return obj


def _link(objs: list[str], out: str, verbose: bool) -> None:
    newest = max(os.path.getmtime(o) for o in objs)
    if os.path.exists(out) and os.path.getmtime(out) >= newest:
        return
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", out + ".tmp"] + objs
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed for {out}:\n{r.stdout}\n{r.stderr}")
    os.replace(out + ".tmp", out)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, probes: bool = True,
          debug: bool = True) -> str:
    """Compile every CUDA translation unit and link libfa.so (+ libfa_debug.so, libfa_probe.so)."""
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    jobs = [(u, False) for u in PRODUCT_UNITS] + [(u, False) for u in (PROBE_UNITS if probes else [])]
    jobs += [(u, True) for u in (PRODUCT_UNITS if debug else [])]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        futs = {j: ex.submit(_compile, j[0], extra, force, verbose or ptxas_verbose, j[1]) for j in jobs}
        objs = {j: f.result() for j, f in futs.items()}
    _link([objs[(u, False)] for u in PRODUCT_UNITS], LIB, verbose)
    if debug:
        _link([objs[(u, True)] for u in PRODUCT_UNITS], DEBUG_LIB, verbose)
    if probes:
        _link([objs[(u, False)] for u in PROBE_UNITS], PROBE_LIB, verbose)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv)
    print(LIB)
