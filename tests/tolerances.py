"""Parity tolerances against the fp64 oracle (stated for this path):
O max-abs <= 1e-2, LSE max-abs <= 1e-3, dQ/dK/dV max-abs <= 2e-2 * max|grad|.

O and the gradients are returned in bf16.  Where |O_ref| >= 4 the bf16 grid
spacing is 2^-5 or coarser, so rounding the output alone can cost half an
ulp (>= 0.0156), more than the 1e-2 budget.  For those elements only, the
bound is 1e-2 plus half a bf16 ulp at |O_ref|; below 4 half an ulp is at
most 2^-8 and the plain 1e-2 applies.
"""
import numpy as np

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_REL_TOL = 2e-2
# When the exact gradient is identically zero (every row sees a single key,
# e.g. T = 1: P = 1 and dS = P (dP - D) = 0), 2e-2 * max|grad| is 0.  D and
# dP are the same fp32 sum taken in different orders, so a residual of fp32
# rounding remains; this absolute floor only matters in that degenerate case.
GRAD_ABS_FLOOR = 1e-5


def bf16_half_ulp(x):
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 2.0 ** (e - 8)   # bf16 keeps 8 significant bits: ulp = 2^(e-7)


def o_bound(o_ref):
    o_ref = np.asarray(o_ref, dtype=np.float64)
    return O_TOL + np.where(np.abs(o_ref) >= 4.0, bf16_half_ulp(o_ref), 0.0)


def o_ok(o, o_ref):
    """True iff every |O - O_ref| is within its bound."""
    return bool(np.all(np.abs(np.asarray(o) - o_ref) <= o_bound(o_ref)))


def grad_bound(g_ref):
    return max(GRAD_REL_TOL * float(np.abs(np.asarray(g_ref, dtype=np.float64)).max()), GRAD_ABS_FLOOR)


def grad_ok(g, g_ref):
    g_ref = np.asarray(g_ref, dtype=np.float64)
    return bool(np.abs(np.asarray(g) - g_ref).max() <= grad_bound(g_ref))
