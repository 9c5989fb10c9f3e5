"""Helpers shared by the GPU parity tests: run the CUDA path and the fp64
oracle on the same seeded bf16 inputs and compare element by element."""
from __future__ import annotations

import math

import numpy as np
import torch

import relative_position_biased_gb300 as rpb
from relative_position_biased_gb300 import workloads as W

OUT_TOL = 2e-2   # max |out_gpu - out_oracle|  (bf16 in, fp32 accumulate, bf16 out)
LSE_TOL = 1e-3   # max |lse_gpu - lse_oracle|  (natural log)


def run_gpu(w: W.Workload, inp, *, decode=None, num_splits=0, stream=None):
    dev = {k: v.cuda() for k, v in inp.items()}
    decode = w.is_decode if decode is None else decode
    kw = dict(max_seqlen_q=max(w.q_lens), max_seqlen_k=max(w.k_lens), alpha=w.alpha,
              window=w.window, log_scale_base=w.log_scale_base)
    args = (dev["q"], dev["k"], dev["v"], dev["r"], dev["P"], dev["cu_seqlens_q"],
            dev["cu_seqlens_k"])
    if decode:
        out, lse = rpb.decode(*args, num_splits=num_splits, **kw)
    else:
        out, lse = rpb.prefill(*args, **kw)
    torch.cuda.synchronize()
    st = rpb.relattn_get_device_error()
    assert st == rpb.RELATTN_OK, (rpb.STATUS_NAMES.get(st, st), hex(rpb.relattn_last_device_error_word()))
    return out.float().cpu().numpy(), lse.cpu().numpy()


def run_oracle(w: W.Workload, inp, rows=None):
    import oracle
    return oracle.forward(inp["q"], inp["k"], inp["v"], inp["r"], inp["P"], inp["cu_seqlens_q"],
                          inp["cu_seqlens_k"], alpha=w.alpha, window=w.window,
                          log_scale_base=w.log_scale_base, rows=rows)


def sample_rows(w: W.Workload, n_random=64, seed=1234):
    """Rows to check on large workloads: each sequence's first and last 128
    rows, rows around 1024 and 4096 (bias extent and window edges), plus
    seeded random rows."""
    rng = np.random.default_rng(seed)
    rows, start = [], 0
    for L in w.q_lens:
        local = set(range(min(128, L))) | set(range(max(0, L - 128), L))
        for c in (1023, 1024, 1025, 4095, 4096, 4097):
            if c < L:
                local.add(c)
        local |= set(int(x) for x in rng.integers(0, L, size=min(n_random, L)))
        rows += [start + x for x in sorted(local)]
        start += L
    return np.array(rows, dtype=np.int64)


def compare(w: W.Workload, inp, gpu, rows=None, out_tol=OUT_TOL, lse_tol=LSE_TOL):
    out_g, lse_g = gpu
    out_o, lse_o = run_oracle(w, inp, rows)
    if rows is not None:
        out_g = out_g[rows]
        lse_g = lse_g[:, rows]
    d_out = float(np.max(np.abs(out_g - out_o))) if out_o.size else 0.0
    d_lse = float(np.max(np.abs(lse_g.T - lse_o))) if lse_o.size else 0.0
    assert np.all(np.isfinite(out_g)) and np.all(np.isfinite(lse_g))
    assert d_out <= out_tol, f"{w.name}: max |dout| = {d_out:.3e} > {out_tol}"
    assert d_lse <= lse_tol, f"{w.name}: max |dlse| = {d_lse:.3e} > {lse_tol}"
    return d_out, d_lse


def alpha_default():
    return 1.0 / math.sqrt(W.HEAD_DIM)


def oracle_key_range_grads(w, inp, b, j0, m):
    """Exact dk / dv of keys [j0, j0 + m) of sequence b of a prefill workload
    (Lq = Lk, no log-scale), from the backward oracle run on just the query
    rows that see those keys.

    With a window W, rows [j0, j0 + m + W - 1) are the only ones that see the
    keys, and they see keys from ka = j0 - W + 1 on.  The oracle takes that
    chunk bottom-right aligned: chunk row t sits at position
    (qb - ka) - (qb - qa) + t = (qa + t) - ka, its original position less
    ka, and so does every key; every distance i - j, mask and logit is the
    original one (without a log-scale, which depends on the absolute
    position).  One virtual sequence per query head (with
    its kv head's keys) lets the oracle's per-(sequence, kv head) tasks run
    in parallel; the dk / dv of a kv head are the sums over its query heads.
    Returns (dk, dv) [m, Hkv, 128] float64.
    """
    import oracle
    L, W_ = w.q_lens[b], (w.window if w.window > 0 else w.q_lens[b])
    base = sum(w.q_lens[:b])
    qa, qb = j0, min(L, j0 + m + W_ - 1)
    ka = max(0, j0 - W_ + 1)
    group = w.Hq // w.Hkv
    qs, rs, ds, ks, vs, cq, ck = [], [], [], [], [], [0], [0]
    for h in range(w.Hq):
        g = h // group
        qs.append(inp["q"][base + qa:base + qb, h:h + 1])
        rs.append(inp["r"][base + qa:base + qb, h:h + 1])
        ds.append(inp["dout"][base + qa:base + qb, h:h + 1])
        ks.append(inp["k"][base + ka:base + qb, g:g + 1])
        vs.append(inp["v"][base + ka:base + qb, g:g + 1])
        cq.append(cq[-1] + (qb - qa))
        ck.append(ck[-1] + (qb - ka))
    cat = torch.cat
    _, dk, dv, _ = oracle.backward(cat(qs), cat(ks), cat(vs), cat(rs), inp["P"], cat(ds), cq, ck,
                                   alpha=w.alpha, window=w.window)
    nk = qb - ka
    dk = dk.reshape(w.Hq, nk, 128)[:, j0 - ka:j0 - ka + m]
    dv = dv.reshape(w.Hq, nk, 128)[:, j0 - ka:j0 - ka + m]
    # sum the query heads of each kv head -> [m, Hkv, 128]
    dk = dk.reshape(w.Hkv, group, m, 128).sum(axis=1).transpose(1, 0, 2)
    dv = dv.reshape(w.Hkv, group, m, 128).sum(axis=1).transpose(1, 0, 2)
    return dk, dv
