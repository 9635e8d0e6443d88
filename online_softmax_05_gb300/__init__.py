"""GB300 (sm_103a) exact attention with the online-softmax recurrence.

A thin ctypes binding over ``libfa.so`` (declared in ``include/fa.h``).  It
only marshals arguments: every step of the forward and backward pass runs in
the library's CUDA kernels.  PyTorch is used for device memory and streams.
There is no CPU fallback: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["fa_fwd", "fa_bwd", "fa_fwd_gqa", "fa_bwd_gqa", "fa_fwd_varlen", "attention_forward_varlen", "fa_bwd_varlen", "attention_backward_varlen", "fa_decode", "attention_decode", "fa_bwd_noalloc", "fa_strerror", "fa_get_device_status", "fa_version",
           "attention_forward", "attention_backward", "FAError", "library_path", "load_library",
           "FlashAttention", "flash_attention"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa.so")
_lib = None
_lock = threading.Lock()

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", -1: "FA_ERR_NULL", -2: "FA_ERR_SHAPE", -3: "FA_ERR_UNSUPPORTED", -4: "FA_ERR_ALIGN",
                -5: "FA_ERR_CUDA", -6: "FA_ERR_NOMEM", -7: "FA_ERR_DEVICE_TIMEOUT", -8: "FA_ERR_ARG",
                -9: "FA_ERR_ARCH", -10: "FA_ERR_SCRATCH", -11: "FA_ERR_SEQLEN",
                -12: "FA_ERR_DEBUG_CHECK"}


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({fa_strerror(code)})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libfa.so (built in-tree by ``online_softmax_05_gb300.build``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is not built; run `python -m online_softmax_05_gb300.build` "
                               "(or __graft_entry__.build()) first. There is no CPU fallback.")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.fa_bwd.restype = i
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_gqa.restype = i
        lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_bwd_gqa.restype = i
        lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_varlen.restype = i
        lib.fa_bwd_varlen.argtypes = [vp] * 10 + [i, i, i, i, i, f, i, vp]
        lib.fa_bwd_varlen.restype = i
        lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.fa_decode.restype = i
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.fa_bwd_noalloc.restype = i
        lib.fa_strerror.argtypes = [i]
        lib.fa_strerror.restype = ctypes.c_char_p
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = i
        lib.fa_version.restype = i
        for name in ("fa_sched_fwd_tile_class", "fa_sched_fwd_keep"):
            getattr(lib, name).argtypes = [i, i, i, i]
            getattr(lib, name).restype = i
        for name in ("fa_sched_bwd_tile_class", "fa_sched_bwd_keep"):
            getattr(lib, name).argtypes = [i, i, i, i, i]
            getattr(lib, name).restype = i
        lib.fa_sched_tile_rows.argtypes = [i, ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.fa_sched_tile_rows.restype = i
        lib.fa_debug_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        lib.fa_debug_set_wait_timeout_ns.restype = i
        lib.fa_debug_inject.argtypes = [i]
        lib.fa_debug_inject.restype = i
        lib.fa_bwd_sums_dq_in_place.argtypes = [i, i, i, i]
        lib.fa_bwd_sums_dq_in_place.restype = i
        lib.fa_set_deterministic.argtypes = [i]
        lib.fa_set_deterministic.restype = i
        lib.fa_set_timing_events.argtypes = [vp, vp, vp, vp, vp]
        lib.fa_set_timing_events.restype = i
        _lib = lib
        return lib


def _ptr(x) -> int | None:
    """Device pointer of a torch tensor, or an int / None passed through."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def fa_fwd(q, k, v, o, lse, B: int, H: int, T: int, D: int, scale: float, causal: int, stream=None) -> int:
    """C-ABI ``fa_fwd``; tensors (or raw device pointers) in, status code out."""
    return load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, T, D, float(scale),
                                 int(causal), _stream(stream))


def fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B: int, H: int, T: int, D: int, scale: float, causal: int,
           stream=None) -> int:
    """C-ABI ``fa_bwd``; tensors (or raw device pointers) in, status code out."""
    return load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, H, T, D, float(scale), int(causal), _stream(stream))


def fa_fwd_gqa(q, k, v, o, lse, B: int, Hq: int, Hkv: int, T: int, D: int, scale: float, causal: int,
               stream=None) -> int:
    """C-ABI ``fa_fwd_gqa``: Hq query heads over Hkv shared key/value heads."""
    return load_library().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, T, D, float(scale),
                                     int(causal), _stream(stream))


def fa_bwd_gqa(q, k, v, o, dO, lse, dq, dk, dv, B: int, Hq: int, Hkv: int, T: int, D: int, scale: float,
               causal: int, stream=None) -> int:
    """C-ABI ``fa_bwd_gqa``; dk, dv sum over each group of query heads."""
    return load_library().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                     _ptr(dv), B, Hq, Hkv, T, D, float(scale), int(causal), _stream(stream))


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, n_seq: int, max_seqlen: int, total: int, H: int, D: int,
                  scale: float, causal: int, stream=None) -> int:
    """C-ABI ``fa_fwd_varlen``: packed (total, H, D) sequences delimited by device cu_seqlens."""
    return load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), n_seq,
                                        max_seqlen, total, H, D, float(scale), int(causal), _stream(stream))


def attention_forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale: float | None = None,
                             out=None, lse=None, stream=None):
    """O (total, H, D) and LSE (H, total) for packed sequences; cu_seqlens is an int32 CUDA tensor."""
    import torch
    total, H, D = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 3):
            raise ValueError(f"{n} must be a contiguous (total, H, D) bf16 CUDA tensor")
    if not (cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA tensor")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total), device=q.device, dtype=torch.float32) if lse is None else lse
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_fwd_varlen(q, k, v, out, lse, cu_seqlens, cu_seqlens.numel() - 1, max_seqlen, total, H, D, scale,
                       int(causal), stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_varlen")
    return out, lse


def fa_bwd_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, n_seq: int, max_seqlen: int, total: int, H: int,
                  D: int, scale: float, causal: int, stream=None) -> int:
    """C-ABI ``fa_bwd_varlen``: gradients of the packed-sequence forward."""
    return load_library().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk),
                                        _ptr(dv), _ptr(cu_seqlens), n_seq, max_seqlen, total, H, D, float(scale),
                                        int(causal), _stream(stream))


def attention_backward_varlen(q, k, v, o, lse, dO, cu_seqlens, max_seqlen: int, causal: bool = False,
                              scale: float | None = None, dq=None, dk=None, dv=None, stream=None):
    """dQ, dK, dV (total, H, D) for packed sequences (o, lse from attention_forward_varlen)."""
    import torch
    total, H, D = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO")):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 3):
            raise ValueError(f"{n} must be a contiguous (total, H, D) bf16 CUDA tensor")
    if not (cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA tensor")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_bwd_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, cu_seqlens.numel() - 1, max_seqlen, total, H, D,
                       scale, int(causal), stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd_varlen")
    return dq, dk, dv


def fa_decode(q, k, v, o, lse, B: int, H: int, Tq: int, Tk: int, D: int, scale: float, stream=None) -> int:
    """C-ABI ``fa_decode``: Tq (<= 8) query rows per head against all Tk keys, split over the keys."""
    return load_library().fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk, D, float(scale),
                                    _stream(stream))


def attention_decode(q, k, v, scale: float | None = None, out=None, lse=None, stream=None):
    """O, LSE for q (B, H, Tq, D) against k, v (B, H, Tk, D); all bf16 contiguous CUDA tensors."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    B, H, Tq, D = q.shape
    Tk = k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Tq), device=q.device, dtype=torch.float32) if lse is None else lse
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_decode(q, k, v, out, lse, B, H, Tq, Tk, D, scale, stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_decode")
    return out, lse


def fa_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B: int, H: int, T: int, D: int, scale: float, causal: int,
                   stream=None) -> int:
    """C-ABI ``fa_bwd_noalloc``: fa_bwd without any device allocation, for
    callers that cannot allocate at call time; uses the library's fixed
    64 MiB scratch buffer (one shared buffer: serialise calls)."""
    return load_library().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                                         _ptr(dk), _ptr(dv), B, H, T, D, float(scale), int(causal), _stream(stream))


def fa_strerror(code: int) -> str:
    return load_library().fa_strerror(int(code)).decode()


def fa_get_device_status(stream=None) -> int:
    return load_library().fa_get_device_status(_stream(stream))


def fa_version() -> int:
    return load_library().fa_version()


def _check(t, name):
    import torch
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
        raise ValueError(f"{name} must be a contiguous (B, H, T, D) bf16 CUDA tensor")


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None):
    """O, LSE for contiguous (B, H, T, D) bf16 CUDA tensors (outputs allocated if not given)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    B, H, T, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, T), device=q.device, dtype=torch.float32) if lse is None else lse
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_fwd(q, k, v, out, lse, B, H, T, D, scale, int(causal), stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd")
    return out, lse


def attention_backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, dq=None, dk=None,
                       dv=None, stream=None):
    """dQ, dK, dV for contiguous (B, H, T, D) bf16 CUDA tensors."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check(t, n)
    B, H, T, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    rc = fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, T, D, scale, int(causal), stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd")
    return dq, dk, dv


# ---------------------------------------------------------------- autograd
def _as_bhtd(t, name):
    """(B, H, T, D) contiguous view of a (B, H, T, D) or (B, T, D) tensor."""
    if t.dim() == 3:
        t = t.unsqueeze(1)
    elif t.dim() != 4:
        raise ValueError(f"{name} must be (B, H, T, D) or (B, T, D)")
    return t.contiguous()


_autograd_cls = None


def _make_autograd_class():
    import torch

    class FlashAttention(torch.autograd.Function):
        """Exact attention as a differentiable op on the library's kernels.

        Called as ``FlashAttention.apply(q, k, v, is_causal=False, scale=None)``,
        the form of the public interface in "Flash Attention and Kernel
        Optimization" ("Public Interface", "Autograd Wrapper and Backward
        Path"), which the "Lab 06 - Attention kernels" work order also tests
        end to end.  q, k, v: bf16 CUDA tensors (B, H, T, D), or (B, T, D) as
        one head; scale defaults to 1/sqrt(D).  The forward runs fa_fwd and
        saves O and LSE; the backward runs fa_bwd (the tiled backward kernels,
        where that page rebuilds dense attention in PyTorch).
        """

        @staticmethod
        def forward(ctx, q, k, v, is_causal=False, scale=None):
            squeeze = q.dim() == 3
            q4, k4, v4 = (_as_bhtd(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v")))
            o, lse = attention_forward(q4, k4, v4, causal=bool(is_causal), scale=scale)
            ctx.save_for_backward(q4, k4, v4, o, lse)
            ctx.is_causal, ctx.scale, ctx.squeeze = bool(is_causal), scale, squeeze
            return o.squeeze(1) if squeeze else o

        @staticmethod
        def backward(ctx, grad_o):
            q4, k4, v4, o, lse = ctx.saved_tensors
            do = _as_bhtd(grad_o, "grad of o")
            dq, dk, dv = attention_backward(q4, k4, v4, o, lse, do, causal=ctx.is_causal, scale=ctx.scale)
            if ctx.squeeze:
                dq, dk, dv = dq.squeeze(1), dk.squeeze(1), dv.squeeze(1)
            return dq, dk, dv, None, None

    return FlashAttention


def __getattr__(name):
    # FlashAttention subclasses torch.autograd.Function; it is built on first
    # use so that importing this module does not import torch
    global _autograd_cls
    if name == "FlashAttention":
        with _lock:
            if _autograd_cls is None:
                _autograd_cls = _make_autograd_class()
        return _autograd_cls
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


def flash_attention(q, k, v, causal: bool = False, scale: float | None = None):
    """O = softmax(q k^T * scale) v, differentiable (see FlashAttention)."""
    return __getattr__("FlashAttention").apply(q, k, v, causal, scale)
