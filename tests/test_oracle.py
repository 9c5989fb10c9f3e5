"""Pins for the fp64 oracle, each against something other than the oracle itself.

Every pin follows from the definition on the page "SGLang and Miles Add Day-0
Support for Inkling", section "Attention with Relative Positional Embedding"
(rel_logits and logit equations; paragraph "Attention layout" for windows and
the log-scale), plus the mathematics of softmax.  The pins are chosen so that a
plausible slip in the oracle fails at least one of them:

  dropped bias term ............ test_bias_selects_distance, test_geometric_bias_*
  i-j sign / index ............. test_bias_selects_distance, test_geometric_bias_*
  P transposed ([d,c]) ......... test_geometric_bias_multichannel
  E boundary (d<E vs d<=E) ..... test_geometric_bias_*, test_extra_columns_*
  window off-by-one ............ test_window_uniform_closed_form
  alpha / q.k term ............. test_no_bias_matches_sdpa*
  GQA head map ................. test_gqa_head_map_closed_form, test_no_bias_matches_sdpa
  lse base (ln vs log2) ........ closed forms (lse = ln(...))
  log-scale formula ............ test_log_scale_closed_form, test_log_scale_matches_sdpa
  decode alignment ............. test_decode_rows_closed_form, test_decode_equals_prefill_tail
  packing across sequences ..... test_no_bias_matches_sdpa (block-diagonal mask)
"""
import math

import numpy as np
import pytest
import torch

from tests.conftest import ROOT  # noqa: F401

torch.manual_seed(0)


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _run(oracle_mod, q, k, v, r, P, lq, lk=None, **kw):
    lk = lq if lk is None else lk
    kw.setdefault("alpha", 1.0 / math.sqrt(q.shape[-1]))
    return oracle_mod.forward(q, k, v, r, P, _cu(lq), _cu(lk), **kw)


# ---------------------------------------------------------------- special cases

@pytest.mark.parametrize("window", [0, 1, 5, 16])
@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 2), (4, 1)])
def test_no_bias_matches_sdpa(oracle_mod, window, Hq, Hkv):
    """P = 0 reduces to plain causal / windowed GQA softmax attention: compare
    with torch's scaled_dot_product_attention in float64 on a packed batch."""
    rng = np.random.default_rng(1)
    lens = [7, 33, 1, 20]
    T, D, rd, E = sum(lens), 16, 4, 64
    q, k, v = _rand(rng, T, Hq, D), _rand(rng, T, Hkv, D), _rand(rng, T, Hkv, D)
    r, P = _rand(rng, T, Hq, rd), np.zeros((rd, E))
    alpha = 0.37
    out, lse = _run(oracle_mod, q, k, v, r, P, lens, window=window, alpha=alpha)
    # block-diagonal causal (+window) mask over the packed rows
    seg = np.repeat(np.arange(len(lens)), lens)
    pos = np.concatenate([np.arange(n) for n in lens])
    mask = (seg[:, None] == seg[None, :]) & (pos[None, :] <= pos[:, None])
    if window > 0:
        mask &= (pos[:, None] - pos[None, :]) < window
    G = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask), scale=alpha)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)


def test_log_scale_matches_sdpa(oracle_mod):
    """With P = 0 the log-scale multiplies alpha per row: row i equals SDPA with
    scale alpha * max(1, ln(i+1)/ln(base))."""
    rng = np.random.default_rng(2)
    T, D, base, alpha = 40, 16, 8.0, 0.5
    q, k, v = _rand(rng, T, 2, D), _rand(rng, T, 1, D), _rand(rng, T, 1, D)
    out, _ = _run(oracle_mod, q, k, v, _rand(rng, T, 2, 2), np.zeros((2, 8)), [T],
                  alpha=alpha, log_scale_base=base)
    for i in range(T):
        s = max(1.0, math.log(i + 1) / math.log(base))
        qt = torch.from_numpy(q[i:i + 1]).permute(1, 0, 2)[None]
        kt = torch.from_numpy(k[:i + 1]).expand(-1, 2, -1).permute(1, 0, 2)[None]
        vt = torch.from_numpy(v[:i + 1]).expand(-1, 2, -1).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=alpha * s)
        np.testing.assert_allclose(out[i], ref[0, :, 0].numpy(), rtol=0, atol=1e-12)


def test_single_key_returns_v_exactly(oracle_mod):
    """A row that sees one key (position 0, or window 1) returns that v bit-exactly."""
    rng = np.random.default_rng(3)
    T, D = 12, 128
    q, k, v = _rand(rng, T, 2, D), _rand(rng, T, 2, D), _rand(rng, T, 2, D)
    r, P = _rand(rng, T, 2, 4), _rand(rng, 4, 8)
    out, _ = _run(oracle_mod, q, k, v, r, P, [T])
    assert np.array_equal(out[0], v[0])
    out1, _ = _run(oracle_mod, q, k, v, r, P, [T], window=1)
    assert np.array_equal(out1, v)


def test_single_key_lse_is_the_bias(oracle_mod):
    """q = 0, one visible key at distance 0: lse is exactly rel_logits(i, h, 0)."""
    T, D = 6, 16
    z = np.zeros((T, 1, D))
    r = np.ones((T, 1, 1)) * 0.5
    P = np.array([[3.0, -7.0, 11.0]])
    _, lse = _run(oracle_mod, z, z, np.ones((T, 1, D)), r, P, [T], window=1)
    np.testing.assert_array_equal(lse[:, 0], np.full(T, 1.5))


# ---------------------------------------------------------------- closed forms

def test_causal_uniform_closed_form(oracle_mod):
    """q = 0 and P = 0: row i averages v[0..i]; lse = ln(i+1)."""
    rng = np.random.default_rng(4)
    T, D = 50, 16
    z = np.zeros((T, 1, D))
    v = _rand(rng, T, 1, D)
    out, lse = _run(oracle_mod, z, z, v, np.zeros((T, 1, 2)), np.zeros((2, 4)), [T])
    cm = np.cumsum(v[:, 0], axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(out[:, 0], cm, atol=1e-13)
    np.testing.assert_allclose(lse[:, 0], np.log(np.arange(1, T + 1)), atol=1e-13)


@pytest.mark.parametrize("w", [1, 2, 7, 64])
def test_window_uniform_closed_form(oracle_mod, w):
    """q = 0, P = 0, window w: row i averages the last min(w, i+1) values."""
    rng = np.random.default_rng(5)
    T, D = 40, 8
    z = np.zeros((T, 1, D))
    v = _rand(rng, T, 1, D)
    out, lse = _run(oracle_mod, z, z, v, np.zeros((T, 1, 1)), np.zeros((1, 1)), [T], window=w)
    for i in range(T):
        lo = max(0, i - w + 1)
        np.testing.assert_allclose(out[i, 0], v[lo:i + 1, 0].mean(0), atol=1e-13)
        assert abs(lse[i, 0] - math.log(i + 1 - lo)) < 1e-13


def test_gqa_head_map_closed_form(oracle_mod):
    """q = 0, P = 0 with Hq=4, Hkv=2: query head h averages kv head h // 2."""
    rng = np.random.default_rng(6)
    T, D = 9, 8
    v = _rand(rng, T, 2, D)
    out, _ = _run(oracle_mod, np.zeros((T, 4, D)), np.zeros((T, 2, D)), v,
                  np.zeros((T, 4, 1)), np.zeros((1, 1)), [T])
    cm = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None, None]
    for h in range(4):
        np.testing.assert_allclose(out[:, h], cm[:, h // 2], atol=1e-13)


@pytest.mark.parametrize("dstar", [0, 1, 5])
def test_bias_selects_distance(oracle_mod, dstar):
    """q = 0 and a bias of 40 at distance d* only: key j = i - d* gets weight
    e^40 / (e^40 + n - 1) and every other visible key 1 / (e^40 + n - 1)."""
    rng = np.random.default_rng(7)
    T, D, E, beta = 20, 8, 8, 40.0
    z = np.zeros((T, 1, D))
    v = _rand(rng, T, 1, D)
    P = np.zeros((1, E))
    P[0, dstar] = beta
    out, lse = _run(oracle_mod, z, z, v, np.ones((T, 1, 1)), P, [T])
    for i in range(T):
        n = i + 1
        if i >= dstar:
            den = math.exp(beta) + n - 1
            exp_out = (v[:i + 1, 0].sum(0) + (math.exp(beta) - 1) * v[i - dstar, 0]) / den
            exp_lse = math.log(den)
        else:
            exp_out, exp_lse = v[:i + 1, 0].mean(0), math.log(n)
        np.testing.assert_allclose(out[i, 0], exp_out, atol=1e-12)
        assert abs(lse[i, 0] - exp_lse) < 1e-12


def _geometric_lse(i, c, E, w=0):
    """ln sum over visible distances d of exp(-c d) for d < E, exp(0) beyond."""
    n = i + 1 if w <= 0 else min(w, i + 1)
    nb = min(n, E)
    return math.log((1 - math.exp(-c * nb)) / (1 - math.exp(-c)) + (n - nb))


@pytest.mark.parametrize("E,w", [(6, 0), (1, 0), (30, 0), (6, 4), (6, 9)])
def test_geometric_bias_closed_form(oracle_mod, E, w):
    """q = 0, r = 1, P[0, d] = -c d: weights decay geometrically inside the
    extent and are flat beyond it, so lse has a closed form."""
    T, D, c = 24, 4, 0.7
    z = np.zeros((T, 1, D))
    P = -c * np.arange(E, dtype=np.float64)[None, :]
    _, lse = _run(oracle_mod, z, z, np.ones((T, 1, D)), np.ones((T, 1, 1)), P, [T], window=w)
    for i in range(T):
        assert abs(lse[i, 0] - _geometric_lse(i, c, E, w)) < 1e-12


def test_geometric_bias_multichannel(oracle_mod):
    """r picks channel 1 of P ([r_dim, E] with E innermost); channels 0 and 2
    hold noise that must not leak in.  Fails if P is read transposed."""
    rng = np.random.default_rng(8)
    T, D, c, E = 16, 4, 0.3, 10
    P = _rand(rng, 3, E) * 5
    P[1] = -c * np.arange(E)
    r = np.zeros((T, 1, 3))
    r[:, 0, 1] = 1.0
    z = np.zeros((T, 1, D))
    _, lse = _run(oracle_mod, z, z, np.ones((T, 1, D)), r, P, [T])
    for i in range(T):
        assert abs(lse[i, 0] - _geometric_lse(i, c, E)) < 1e-12


def test_log_scale_closed_form(oracle_mod):
    """q = 0, bias beta at distance 0 only, base b: the logit of key i is
    s_i * beta with s_i = max(1, ln(i+1)/ln b); every other logit is 0."""
    rng = np.random.default_rng(9)
    T, D, beta, base = 30, 4, 2.0, 4.0
    z = np.zeros((T, 1, D))
    v = _rand(rng, T, 1, D)
    P = np.zeros((1, 3))
    P[0, 0] = beta
    out, lse = _run(oracle_mod, z, z, v, np.ones((T, 1, 1)), P, [T], log_scale_base=base)
    for i in range(T):
        s = max(1.0, math.log(i + 1) / math.log(base))
        den = math.exp(s * beta) + i
        assert abs(lse[i, 0] - math.log(den)) < 1e-12
        exp_out = (v[:i, 0].sum(0) + math.exp(s * beta) * v[i, 0]) / den
        np.testing.assert_allclose(out[i, 0], exp_out, atol=1e-12)


def test_decode_rows_closed_form(oracle_mod):
    """Bottom-right alignment: 2 query rows against 10 keys sit at positions 8
    and 9, so with q = 0, P = 0 they average v[0..8] and v[0..9]."""
    rng = np.random.default_rng(10)
    D = 8
    v = _rand(rng, 10, 1, D)
    out, lse = _run(oracle_mod, np.zeros((2, 1, D)), np.zeros((10, 1, D)), v,
                    np.zeros((2, 1, 1)), np.zeros((1, 1)), [2], [10])
    np.testing.assert_allclose(out[0, 0], v[:9, 0].mean(0), atol=1e-13)
    np.testing.assert_allclose(out[1, 0], v[:10, 0].mean(0), atol=1e-13)
    np.testing.assert_allclose(lse[:, 0], np.log([9, 10]), atol=1e-13)


# ---------------------------------------------------------------- invariants

def test_extra_columns_beyond_extent_do_not_matter(oracle_mod):
    """Columns of P at distance >= E never enter: appending noise columns while
    keeping E, or appending zeros and raising E, leaves the result unchanged."""
    rng = np.random.default_rng(11)
    T, D, rd, E = 30, 16, 4, 7
    q, k, v = _rand(rng, T, 2, D), _rand(rng, T, 1, D), _rand(rng, T, 1, D)
    r, P = _rand(rng, T, 2, rd), _rand(rng, rd, E)
    o0, l0 = _run(oracle_mod, q, k, v, r, P, [T])
    o2, l2 = _run(oracle_mod, q, k, v, r, np.concatenate([P, np.zeros((rd, 5))], 1), [T])
    np.testing.assert_allclose(o2, o0, atol=1e-14)
    np.testing.assert_allclose(l2, l0, atol=1e-14)
    # noise columns in a wider buffer: pass the first E columns of a wider P
    wide = np.concatenate([P, _rand(rng, rd, 9)], 1)
    o3, l3 = _run(oracle_mod, q, k, v, r, np.ascontiguousarray(wide[:, :E]), [T])
    np.testing.assert_array_equal(o3, o0)
    np.testing.assert_array_equal(l3, l0)


def test_shift_invariance(oracle_mod):
    """With window <= E every visible key is biased; adding a constant c to all
    rel_logits (an extra r channel of 1 and a P row of c) leaves out unchanged
    and moves lse by s_i * c."""
    rng = np.random.default_rng(12)
    T, D, rd, E, w, c, base = 40, 16, 3, 16, 10, 1.75, 4.0
    q, k, v = _rand(rng, T, 2, D), _rand(rng, T, 2, D), _rand(rng, T, 2, D)
    r, P = _rand(rng, T, 2, rd), _rand(rng, rd, E)
    o0, l0 = _run(oracle_mod, q, k, v, r, P, [T], window=w, log_scale_base=base)
    r2 = np.concatenate([r, np.ones((T, 2, 1))], 2)
    P2 = np.concatenate([P, np.full((1, E), c)], 0)
    o1, l1 = _run(oracle_mod, q, k, v, r2, P2, [T], window=w, log_scale_base=base)
    s = np.maximum(1.0, np.log(np.arange(1, T + 1)) / math.log(base))
    np.testing.assert_allclose(o1, o0, atol=1e-12)
    np.testing.assert_allclose(l1 - l0, (s * c)[:, None].repeat(2, 1), atol=1e-12)


def test_decode_equals_prefill_tail(oracle_mod):
    """Decode rows (Lq <= 16 against a longer KV) equal the last rows of a
    prefill over the whole sequence."""
    rng = np.random.default_rng(13)
    T, Lq, D, rd, E = 70, 9, 16, 4, 20
    q, k, v = _rand(rng, T, 4, D), _rand(rng, T, 2, D), _rand(rng, T, 2, D)
    r, P = _rand(rng, T, 4, rd), _rand(rng, rd, E)
    for w, base in [(0, 0.0), (0, 8.0), (12, 0.0)]:
        op, lp = _run(oracle_mod, q, k, v, r, P, [T], window=w, log_scale_base=base)
        od, ld = _run(oracle_mod, q[-Lq:], k, v, r[-Lq:], P, [Lq], [T], window=w,
                      log_scale_base=base)
        np.testing.assert_allclose(od, op[-Lq:], atol=1e-13)
        np.testing.assert_allclose(ld, lp[-Lq:], atol=1e-13)


def test_row_selection_matches_full_run(oracle_mod):
    rng = np.random.default_rng(14)
    lens = [5, 17, 9]
    T, D = sum(lens), 8
    q, k, v = _rand(rng, T, 2, D), _rand(rng, T, 2, D), _rand(rng, T, 2, D)
    r, P = _rand(rng, T, 2, 3), _rand(rng, 3, 6)
    o, l = _run(oracle_mod, q, k, v, r, P, lens)
    rows = [0, 4, 5, 21, 30, 12]
    os_, ls = _run(oracle_mod, q, k, v, r, P, lens, rows=rows)
    np.testing.assert_array_equal(os_, o[rows])
    np.testing.assert_array_equal(ls, l[rows])


def test_bf16_bits_equal_float_path(oracle_mod):
    """bf16 inputs are widened exactly: the bf16-bit path and the float64 path
    on the same (bf16-representable) values agree bit for bit."""
    g = torch.Generator().manual_seed(0)
    T, D = 21, 128
    t = {n: torch.randn(*s, generator=g).to(torch.bfloat16) for n, s in
         dict(q=(T, 4, D), k=(T, 1, D), v=(T, 1, D), r=(T, 4, 32)).items()}
    t["P"] = (torch.randn(32, 64, generator=g) * 0.02).to(torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32)
    ob, lb = oracle_mod.forward(t["q"], t["k"], t["v"], t["r"], t["P"], cu, cu, alpha=0.1)
    of, lf = oracle_mod.forward(*(t[n].double() for n in "q k v r P".split()), cu, cu, alpha=0.1)
    np.testing.assert_array_equal(ob, of)
    np.testing.assert_array_equal(lb, lf)


def test_brute_force_dense_matrix(oracle_mod):
    """Tiny inputs: build the dense T x T logit matrix one element at a time in
    pure Python, mask it, softmax each row with scipy.special; compare."""
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(15)
    T, Hq, Hkv, D, rd, E, alpha, w, base = 11, 2, 1, 4, 2, 4, 0.6, 6, 3.0
    q, k, v = _rand(rng, T, Hq, D), _rand(rng, T, Hkv, D), _rand(rng, T, Hkv, D)
    r, P = _rand(rng, T, Hq, rd), _rand(rng, rd, E)
    out, lse = _run(oracle_mod, q, k, v, r, P, [T], alpha=alpha, window=w, log_scale_base=base)
    for h in range(Hq):
        L = np.full((T, T), -np.inf)
        for i in range(T):
            for j in range(T):
                if j > i or i - j >= w:
                    continue
                dot = sum(q[i, h, e] * k[j, 0, e] for e in range(D))
                b = sum(r[i, h, c] * P[c, i - j] for c in range(rd)) if i - j < E else 0.0
                L[i, j] = max(1.0, math.log(i + 1) / math.log(base)) * (alpha * dot + b)
        np.testing.assert_allclose(lse[:, h], logsumexp(L, axis=1), atol=1e-12)
        np.testing.assert_allclose(out[:, h], softmax(L, axis=1) @ v[:, 0], atol=1e-12)


def test_rejects_bad_arguments(oracle_mod):
    z = np.zeros((4, 2, 8))
    with pytest.raises(ValueError):   # Hq not a multiple of Hkv
        _run(oracle_mod, np.zeros((4, 3, 8)), z, z, np.zeros((4, 3, 1)), np.zeros((1, 1)), [4])
    with pytest.raises(ValueError):   # Lk < Lq
        _run(oracle_mod, z, z[:2], z[:2], np.zeros((4, 2, 1)), np.zeros((1, 1)), [4], [2])
