"""Algorithmic work of a relative-attention call, for roofline reporting.

Counts only what the definition needs (page "SGLang and Miles Add Day-0
Support for Inkling", section "Attention with Relative Positional
Embedding"): per head and per visible (query, key) pair, 2*128 flops for q.k
and 2*128 for the PV product; per head and per (query, distance) with
d < min(E, visible keys), 2*r_dim flops for r.P.  No dense T^2, no padded
tiles, no softmax arithmetic.  Decode bytes are the K and V rows some query of
the sequence can see (bf16), nothing else.
"""
from __future__ import annotations

import numpy as np

from .workloads import Workload


def _rows(w: Workload):
    for lq, lk in zip(w.q_lens, w.k_lens):
        p = (lk - lq) + np.arange(lq, dtype=np.int64)
        lo = np.maximum(0, p - w.window + 1) if w.window > 0 else np.zeros_like(p)
        yield p, lo, lk


def visible_pairs(w: Workload, rows=None) -> int:
    """Visible (i, j) pairs per head, over all (or the selected packed) rows."""
    tot, start = 0, 0
    for p, lo, _ in _rows(w):
        n = p - lo + 1
        if rows is not None:
            sel = rows[(rows >= start) & (rows < start + len(p))] - start
            n = n[sel]
        tot += int(n.sum())
        start += len(p)
    return tot


def band_pairs(w: Workload, rows=None) -> int:
    """(i, d) pairs per head with a bias term: d < min(E, visible keys)."""
    if w.rel_extent <= 0 or w.r_dim <= 0:
        return 0
    tot, start = 0, 0
    for p, lo, _ in _rows(w):
        n = np.minimum(p - lo + 1, w.rel_extent)
        if rows is not None:
            sel = rows[(rows >= start) & (rows < start + len(p))] - start
            n = n[sel]
        tot += int(n.sum())
        start += len(p)
    return tot


def flops(w: Workload, rows=None) -> int:
    D = w.head_dim
    return w.Hq * (4 * D * visible_pairs(w, rows) + 2 * w.r_dim * band_pairs(w, rows))


def bwd_flops(w: Workload, rows=None) -> int:
    """Backward: per head and visible pair the five products S, dP, dV, dK, dQ
    (2*128 flops each, 2.5x the forward's two), and per band (i, d) pair
    2*r_dim for dr = dR . P^T.  Recomputation beyond S is not counted."""
    D = w.head_dim
    return w.Hq * (10 * D * visible_pairs(w, rows) + 2 * w.r_dim * band_pairs(w, rows))


def kv_bytes(w: Workload) -> int:
    """bf16 K and V rows visible to at least one query of each sequence."""
    tot = 0
    for p, lo, lk in _rows(w):
        if len(p) == 0:
            continue
        tot += int(lk - lo.min()) * w.Hkv * w.head_dim * 2 * 2
    return tot


def kv_bytes_mxfp8(w: Workload) -> int:
    """The same visible K and V rows stored in MXFP8: one E4M3 byte per
    element and one E8M0 scale byte per 32 elements."""
    return kv_bytes(w) // 2 // w.head_dim * (w.head_dim + w.head_dim // 32)


def io_bytes(w: Workload) -> dict:
    """Bytes of every input and output tensor (for host<->device copies)."""
    Tq, Tk, D = sum(w.q_lens), sum(w.k_lens), w.head_dim
    inp = 2 * (Tq * w.Hq * D + 2 * Tk * w.Hkv * D + Tq * w.Hq * w.r_dim +
               w.r_dim * w.rel_extent) + 2 * 4 * (w.batch + 1)
    out = 2 * Tq * w.Hq * D + 4 * Tq * w.Hq
    return {"h2d": inp, "d2h": out}


def prologue_bytes(w: Workload, state_in: bool = False, state_out: bool = True) -> int:
    """Bytes the attention prologue must move for the chunk rows of ``w``:
    read q, k, v once and write q_out and the k / v cache rows once (bf16),
    read the conv taps and norm weights (fp32) once, and the conv states.
    The earlier rows a conv tap reads again are not counted."""
    Tq, D, C = sum(w.q_lens), w.head_dim, w.Hkv * w.head_dim
    rows = 2 * 2 * Tq * (w.Hq + 2 * w.Hkv) * D
    weights = 4 * (2 * C * 4 + 2 * D)
    state = 2 * 2 * w.batch * 3 * C
    return rows + weights + (state if state_in else 0) + (state if state_out else 0)
