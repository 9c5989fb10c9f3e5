"""Pins of the fp64 backward oracle (gradients of sum(dout * out), P frozen).

Each pin ties the backward oracle to something other than its own formulas:
central finite differences of the (separately pinned) forward oracle; torch's
fp64 autograd through a dense formulation of the logits; torch's SDPA
backward when P = 0; closed forms (a single visible key); and two invariants
of the softmax (shifting every key of a sequence changes nothing, so the dk of
a sequence sum to zero; the dv of a sequence sum to the sum of dout).
"""
import numpy as np
import pytest
import torch

import oracle
from relative_position_biased_gb300 import workloads as W
from tests import parity_util as PU

ALPHA = 0.37


def _inputs(seed, lens, klens=None, Hq=4, Hkv=2, D=16, r_dim=5, E=6):
    rng = np.random.default_rng(seed)
    klens = lens if klens is None else klens
    Tq, Tk = sum(lens), sum(klens)
    x = dict(q=rng.standard_normal((Tq, Hq, D)), k=rng.standard_normal((Tk, Hkv, D)),
             v=rng.standard_normal((Tk, Hkv, D)), r=rng.standard_normal((Tq, Hq, r_dim)),
             P=rng.standard_normal((r_dim, E)) * 0.5, dout=rng.standard_normal((Tq, Hq, D)))
    x["cq"] = np.cumsum([0] + list(lens)).astype(np.int32)
    x["ck"] = np.cumsum([0] + list(klens)).astype(np.int32)
    return x


def _bwd(x, **kw):
    return oracle.backward(x["q"], x["k"], x["v"], x["r"], x["P"], x["dout"], x["cq"], x["ck"],
                           alpha=ALPHA, **kw)


def _loss(x, **kw):
    out, _ = oracle.forward(x["q"], x["k"], x["v"], x["r"], x["P"], x["cq"], x["ck"],
                            alpha=ALPHA, **kw)
    return float(np.sum(out * x["dout"]))


@pytest.mark.parametrize("kw", [dict(), dict(window=3), dict(log_scale_base=2.5),
                                dict(window=4, log_scale_base=3.0)])
def test_finite_differences_of_the_forward(kw):
    x = _inputs(1, [7, 3], [9, 3])
    grads = dict(zip(("q", "k", "v", "r"), _bwd(x, **kw)))
    rng = np.random.default_rng(2)
    h = 1e-5
    for name in ("q", "k", "v", "r"):
        a = x[name]
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in a.shape)
            keep = a[idx]
            a[idx] = keep + h
            up = _loss(x, **kw)
            a[idx] = keep - h
            dn = _loss(x, **kw)
            a[idx] = keep
            fd = (up - dn) / (2 * h)
            assert abs(fd - grads[name][idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grads[name][idx])


def _dense_torch(x, window=0, log_scale_base=0.0):
    """fp64 autograd through dense logits with the bias gathered per (i, j)."""
    t = {n: torch.tensor(x[n], dtype=torch.float64, requires_grad=n in "qkvr")
         for n in ("q", "k", "v", "r")}
    P = torch.tensor(x["P"], dtype=torch.float64)
    dout = torch.tensor(x["dout"], dtype=torch.float64)
    Hq, Hkv = t["q"].shape[1], t["k"].shape[1]
    G, E = Hq // Hkv, P.shape[1]
    outs = []
    for b in range(len(x["cq"]) - 1):
        a0, a1, k0, k1 = x["cq"][b], x["cq"][b + 1], x["ck"][b], x["ck"][b + 1]
        Lq, Lk = a1 - a0, k1 - k0
        if Lq == 0:
            continue
        q, r = t["q"][a0:a1], t["r"][a0:a1]
        k = t["k"][k0:k1].repeat_interleave(G, dim=1)
        v = t["v"][k0:k1].repeat_interleave(G, dim=1)
        pos = torch.arange(Lk - Lq, Lk, dtype=torch.int64)
        d = pos[:, None] - torch.arange(Lk)[None, :]                 # [Lq, Lk]
        vis = (d >= 0) & ((d < window) if window > 0 else torch.ones_like(d, dtype=torch.bool))
        R = torch.einsum("thc,ce->hte", r, P)                         # [H, Lq, E]
        inband = vis & (d < E)
        idx = d.clamp(0, E - 1).expand(Hq, -1, -1)
        bias = torch.gather(R, 2, idx) * inband
        s = torch.ones(Lq, dtype=torch.float64)
        if log_scale_base > 0:
            s = torch.clamp(torch.log(pos.double() + 1) / np.log(log_scale_base), min=1.0)
        logit = s[None, :, None] * (ALPHA * torch.einsum("thd,jhd->htj", q, k) + bias)
        logit = logit.masked_fill(~vis, float("-inf"))
        outs.append(torch.einsum("htj,jhd->thd", torch.softmax(logit, -1), v))
    loss = (torch.cat(outs) * dout).sum()
    loss.backward()
    return [t[n].grad.numpy() for n in ("q", "k", "v", "r")]


@pytest.mark.parametrize("kw", [dict(), dict(window=5), dict(log_scale_base=4.0)])
def test_matches_torch_autograd_of_a_dense_formulation(kw):
    x = _inputs(3, [9, 1, 6], [12, 4, 6], Hq=6, Hkv=2, E=5)
    for got, ref, name in zip(_bwd(x, **kw), _dense_torch(x, **kw), "qkvr"):
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-11, err_msg=name)


def test_p_zero_matches_sdpa_backward():
    x = _inputs(4, [8], Hq=4, Hkv=4)
    x["P"][:] = 0.0
    dq, dk, dv, dr = _bwd(x)
    assert not dr.any()
    q, k, v = (torch.tensor(x[n], dtype=torch.float64).transpose(0, 1).requires_grad_()
               for n in ("q", "k", "v"))
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=ALPHA)
    (out.transpose(0, 1) * torch.tensor(x["dout"])).sum().backward()
    np.testing.assert_allclose(dq, q.grad.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, k.grad.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, v.grad.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)


def test_single_visible_key_gives_closed_forms():
    # sequences of one token: out = v, so only dv is non-zero (dv = sum of
    # the group's dout); a window of 1 does the same for every row
    x = _inputs(5, [1, 1, 1], Hq=4, Hkv=2)
    dq, dk, dv, dr = _bwd(x)
    assert not dq.any() and not dk.any() and not dr.any()
    np.testing.assert_allclose(dv, x["dout"].reshape(3, 2, 2, -1).sum(axis=2), atol=1e-14)
    y = _inputs(6, [5], Hq=2, Hkv=1)
    dq, dk, dv, dr = _bwd(y, window=1)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15 and np.abs(dr).max() < 1e-15
    np.testing.assert_allclose(dv[:, 0], y["dout"].sum(axis=1), atol=1e-14)


@pytest.mark.parametrize("kw", [dict(), dict(window=3, log_scale_base=2.0)])
def test_softmax_invariants(kw):
    x = _inputs(7, [6, 9], [8, 9], Hq=4, Hkv=2)
    dq, dk, dv, dr = _bwd(x, **kw)
    for b in range(2):
        k0, k1 = x["ck"][b], x["ck"][b + 1]
        a0, a1 = x["cq"][b], x["cq"][b + 1]
        # shifting every key of the sequence leaves every softmax unchanged
        np.testing.assert_allclose(dk[k0:k1].sum(axis=0), 0.0, atol=1e-12)
        # the weights of each row sum to one
        want = x["dout"][a0:a1].reshape(a1 - a0, 2, 2, -1).sum(axis=(0, 2))
        np.testing.assert_allclose(dv[k0:k1].sum(axis=0), want, atol=1e-12)


def test_key_range_oracle_matches_the_whole_sequence(oracle_mod):
    """The chunked oracle of the full-size test against the oracle run on the
    whole packed batch, on a small windowed workload with the same shape of
    problem (several sequences, GQA, a band): the dk / dv of every sampled
    key range must agree to fp64 rounding."""
    w = W.custom("keyrange", [300, 260], [300, 260], 4, 2, 16, 48, window=70)
    inp = W.make_inputs(w, with_dout=True)
    _, dk, dv, _ = oracle_mod.backward(inp["q"], inp["k"], inp["v"], inp["r"], inp["P"],
                                       inp["dout"], inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                                       alpha=w.alpha, window=w.window)
    for b, j0, m in ((0, 0, 20), (0, 100, 37), (1, 230, 30), (1, 0, 260)):
        rk, rv = PU.oracle_key_range_grads(w, inp, b, j0, m)
        base = sum(w.q_lens[:b])
        assert np.allclose(rk, dk[base + j0:base + j0 + m], rtol=1e-12, atol=1e-12)
        assert np.allclose(rv, dv[base + j0:base + j0 + m], rtol=1e-12, atol=1e-12)
