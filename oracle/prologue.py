"""fp64 oracle of the attention prologue -- TEST INFRASTRUCTURE ONLY.

The step right before the attention forward, as described on the page "SGLang
and Miles Add Day-0 Support for Inkling":
  * section "Short Convolution (ShortConv)": a per-channel causal filter over
    the token dimension, y[t,c] = x[t,c] + sum_{d=0}^{W-1} w[c,d] x[t-d,c],
    W = 4, applied to the K and V streams right after their projections;
  * section "ShortConv Optimization", paragraph "KV ShortConv + QK-norm + KV
    store": the K / V convolution, the Q / K RMSNorm and the KV-cache write
    fused into one prologue.

Readings where the pages are silent (the same ones the CUDA kernel uses):
  * RMSNorm is per token and per head over the 128 head dims,
    x * rsqrt(mean(x^2) + eps) * gamma, with one gamma of 128 values for q
    and one for k (shared by the heads); K is normalised after its
    convolution, V only convolved, Q only normalised.
  * Positions of a chunk are bottom-right aligned in their sequence (the new
    rows are the last Lq of Lk), and the cache rows they go to are the same
    rows the attention reads.  Inputs before the chunk come from a conv state
    holding the 3 pre-convolution inputs that precede it (oldest first);
    without a state they are zero (the sequence starts with the chunk).
  * The state after the call holds the last 3 pre-convolution inputs up to
    the chunk's end.

Plain numpy, fp64, loops over sequences; written from the equations above.
Only tests/, __graft_entry__.smoke() and bench.py may import it.
"""
from __future__ import annotations

import numpy as np

W = 4   # ShortConv taps ("Current Inkling configurations use W = 4")


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        t = x.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.float()
        return t.double().numpy()
    return np.asarray(x, dtype=np.float64)


def short_conv(x, w, state=None):
    """y[t,c] = x[t,c] + sum_d w[c,d] x[t-d,c] over one sequence's rows.

    x [T, C]; w [C, W]; state [W-1, C] (the inputs before row 0, oldest first)
    or None for zeros.  Returns (y [T, C], new state [W-1, C]).
    """
    x = _f64(x)
    w = _f64(w)
    T, C = x.shape
    hist = np.zeros((W - 1, C)) if state is None else _f64(state)
    ext = np.concatenate([hist, x], axis=0)            # row W-1+t is x[t]
    y = x.copy()
    for d in range(W):
        y += w[:, d][None, :] * ext[W - 1 - d: W - 1 - d + T]
    return y, ext[-(W - 1):].copy()


def rms_norm(x, gamma, eps):
    """x [..., 128] -> x / sqrt(mean(x^2) + eps) * gamma (last axis)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(gamma)


def prologue(q, k, v, conv_k, conv_v, norm_q, norm_k, cu_seqlens_q, cu_seqlens_k, *,
             eps=1e-6, state_k=None, state_v=None):
    """The prologue of one chunk of packed sequences.

    q [Tq, Hq, 128], k / v [Tq, Hkv, 128] (this chunk's rows); conv_k / conv_v
    [Hkv*128, W]; norm_q / norm_k [128]; cu_seqlens_q / _k [B+1]; state_k /
    state_v [B, W-1, Hkv*128] or None.
    Returns dict: q_out [Tq, Hq, 128]; k_rows / v_rows [Tq, Hkv, 128] (what
    goes to the cache rows); cache_rows [Tq] (cache row of each chunk row);
    state_k / state_v [B, W-1, Hkv*128] after the chunk.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    cq = np.asarray(_f64(cu_seqlens_q), dtype=np.int64)
    ck = np.asarray(_f64(cu_seqlens_k), dtype=np.int64)
    Tq, Hkv, D = k.shape
    C = Hkv * D
    B = len(cq) - 1
    q_out = rms_norm(q, norm_q, eps)
    k_rows = np.zeros_like(k)
    v_rows = np.zeros_like(v)
    rows = np.zeros(Tq, dtype=np.int64)
    sk = np.zeros((B, W - 1, C))
    sv = np.zeros((B, W - 1, C))
    for b in range(B):
        a, e = cq[b], cq[b + 1]
        Lq, Lk = e - a, ck[b + 1] - ck[b]
        st_k = None if state_k is None else _f64(state_k)[b]
        st_v = None if state_v is None else _f64(state_v)[b]
        yk, sk[b] = short_conv(k[a:e].reshape(Lq, C), conv_k, st_k)
        yv, sv[b] = short_conv(v[a:e].reshape(Lq, C), conv_v, st_v)
        k_rows[a:e] = rms_norm(yk.reshape(Lq, Hkv, D), norm_k, eps)
        v_rows[a:e] = yv.reshape(Lq, Hkv, D)
        rows[a:e] = ck[b] + (Lk - Lq) + np.arange(Lq)
    return {"q_out": q_out, "k_rows": k_rows, "v_rows": v_rows, "cache_rows": rows,
            "state_k": sk, "state_v": sv}
