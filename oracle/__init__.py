"""fp64 CPU oracle for Inkling relative attention -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``relattn_oracle.c`` (the forward: plain C, fp64, one
row at a time, two-pass softmax) and ``relattn_oracle_bwd.c`` (the backward:
the chain rule through that softmax, with P frozen); this module compiles them
with gcc and marshals arrays through ctypes.  It shares nothing with the CUDA library.  Only the test suite,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
may import it; the product path never does.

Definition followed: page "SGLang and Miles Add Day-0 Support for Inkling",
section "Attention with Relative Positional Embedding" (rel_logits and logit
equations, paragraph "Attention layout" for windows and the log-scale).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "relattn_oracle.c"), os.path.join(_HERE, "relattn_oracle_bwd.c")]
_LIB = os.path.join(_HERE, "librelattn_oracle.so")
_lock = threading.Lock()
_lib = None

F64, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/librelattn_oracle.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and all(os.path.getmtime(_LIB) >= os.path.getmtime(s) for s in _SRCS)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-fopenmp", "-shared", "-fPIC", "-std=c11",
           "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.relattn_oracle_forward.restype = ctypes.c_int
            vp, i32p, i64p, f64p = (ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_double))
            ci, cd = ctypes.c_int, ctypes.c_double
            lib.relattn_oracle_forward.argtypes = [
                ci, vp, vp, vp, vp, vp, i32p, i32p, ci, ci, ci, ci, ci, ci, ci,
                cd, cd, i64p, ctypes.c_int64, f64p, f64p, ci]
            lib.relattn_oracle_backward.restype = ctypes.c_int
            lib.relattn_oracle_backward.argtypes = [
                ci, vp, vp, vp, vp, vp, vp, i32p, i32p, ci, ci, ci, ci, ci, ci, ci,
                cd, cd, f64p, f64p, f64p, f64p, ci]
            lib.relattn_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().relattn_oracle_max_threads())


def _as_input(x):
    """Return (contiguous numpy array, dtype code).  bf16 torch tensors are
    passed as their raw bit patterns (widened to fp64 exactly in C)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            return x.to(torch.float64).numpy(), F64
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        return a, BF16
    return np.ascontiguousarray(a, dtype=np.float64), F64


def forward(q, k, v, r, P, cu_seqlens_q, cu_seqlens_k, *, alpha: float,
            window: int = 0, log_scale_base: float = 0.0, rows=None,
            threads: int = 0):
    """Evaluate the relative-attention forward in fp64.

    q [Tq,Hq,D], k/v [Tk,Hkv,D], r [Tq,Hq,r_dim], P [r_dim,E] (all bf16 torch
    tensors or float arrays of one kind); cu_seqlens_* int [B+1].
    ``rows``: optional packed query-row indices to evaluate (default: all).
    Returns (out [n,Hq,D] float64, lse [n,Hq] float64), natural-log lse.
    """
    lib = _load()
    arrs = [_as_input(x) for x in (q, k, v, r, P)]
    kinds = {a[1] for a in arrs}
    if len(kinds) != 1:
        raise TypeError("oracle inputs must all be bf16 or all be float")
    dtype = kinds.pop()
    qa, ka, va, ra, Pa = (a[0] for a in arrs)
    Tq, Hq, D = qa.shape
    Tk, Hkv, Dk = ka.shape
    if Dk != D or va.shape != ka.shape:
        raise ValueError("k/v shape mismatch")
    r_dim = ra.shape[2] if ra.ndim == 3 else 0
    if Pa.ndim != 2 or Pa.shape[0] != r_dim:
        raise ValueError("P must be [r_dim, E]")
    E = Pa.shape[1]
    cq = np.ascontiguousarray(np.asarray(
        cu_seqlens_q.cpu() if hasattr(cu_seqlens_q, "cpu") else cu_seqlens_q), dtype=np.int32)
    ck = np.ascontiguousarray(np.asarray(
        cu_seqlens_k.cpu() if hasattr(cu_seqlens_k, "cpu") else cu_seqlens_k), dtype=np.int32)
    B = cq.shape[0] - 1
    if rows is None:
        sel_p, n = None, int(cq[-1]) if B > 0 else 0
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows), dtype=np.int64)
        sel_p, n = rows_a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows_a.shape[0]
    out = np.zeros((n, Hq, D), dtype=np.float64)
    lse = np.zeros((n, Hq), dtype=np.float64)
    rc = lib.relattn_oracle_forward(
        dtype, qa.ctypes.data, ka.ctypes.data, va.ctypes.data, ra.ctypes.data,
        Pa.ctypes.data, cq.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        ck.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, Hq, Hkv, D, r_dim,
        E, int(window), float(alpha), float(log_scale_base), sel_p, n,
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out, lse


def backward(q, k, v, r, P, dout, cu_seqlens_q, cu_seqlens_k, *, alpha: float,
             window: int = 0, log_scale_base: float = 0.0, threads: int = 0):
    """Gradients of sum(dout * out) in fp64, with P frozen.

    Inputs as for ``forward`` plus dout [Tq,Hq,D] (same kind).  Returns
    (dq [Tq,Hq,D], dk [Tk,Hkv,D], dv [Tk,Hkv,D], dr [Tq,Hq,r_dim]) float64.
    """
    lib = _load()
    arrs = [_as_input(x) for x in (q, k, v, r, P, dout)]
    kinds = {a[1] for a in arrs}
    if len(kinds) != 1:
        raise TypeError("oracle inputs must all be bf16 or all be float")
    dtype = kinds.pop()
    qa, ka, va, ra, Pa, da = (a[0] for a in arrs)
    Tq, Hq, D = qa.shape
    Tk, Hkv, _ = ka.shape
    if da.shape != qa.shape or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    r_dim = ra.shape[2] if ra.ndim == 3 else 0
    if Pa.ndim != 2 or Pa.shape[0] != r_dim:
        raise ValueError("P must be [r_dim, E]")
    E = Pa.shape[1]
    cq = np.ascontiguousarray(np.asarray(
        cu_seqlens_q.cpu() if hasattr(cu_seqlens_q, "cpu") else cu_seqlens_q), dtype=np.int32)
    ck = np.ascontiguousarray(np.asarray(
        cu_seqlens_k.cpu() if hasattr(cu_seqlens_k, "cpu") else cu_seqlens_k), dtype=np.int32)
    B = cq.shape[0] - 1
    dq = np.zeros((Tq, Hq, D))
    dk = np.zeros((Tk, Hkv, D))
    dv = np.zeros((Tk, Hkv, D))
    dr = np.zeros((Tq, Hq, r_dim))
    f64p = ctypes.POINTER(ctypes.c_double)
    rc = lib.relattn_oracle_backward(
        dtype, qa.ctypes.data, ka.ctypes.data, va.ctypes.data, ra.ctypes.data,
        Pa.ctypes.data, da.ctypes.data, cq.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        ck.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), B, Hq, Hkv, D, r_dim, E,
        int(window), float(alpha), float(log_scale_base), dq.ctypes.data_as(f64p),
        dk.ctypes.data_as(f64p), dv.ctypes.data_as(f64p), dr.ctypes.data_as(f64p),
        int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return dq, dk, dv, dr
