"""Pins of the prologue oracle (ShortConv + Q/K RMSNorm + KV-cache rows).

Each pin fixes the oracle against something other than its own formula: the
conv's impulse response (tap order and lag direction), identities (zero taps,
unit RMS), invariances the pages imply (causality, per-sequence independence,
a chunk with its conv state equal to the whole sequence) and the cache-row
alignment.
"""
import numpy as np
import pytest

from oracle import prologue as P

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_zero_taps_pass_the_input_through():
    rng = np.random.default_rng(0)
    x = _rand(rng, 7, 5)
    y, st = P.short_conv(x, np.zeros((5, P.W)))
    np.testing.assert_array_equal(y, x)
    np.testing.assert_array_equal(st, x[-3:])


def test_impulse_response_gives_the_taps_in_lag_order():
    # x = delta at t0 in every channel: y[t] = delta[t] + w[:, t - t0] for 0 <= t-t0 < W
    rng = np.random.default_rng(1)
    C, T, t0 = 6, 12, 3
    w = _rand(rng, C, P.W)
    x = np.zeros((T, C))
    x[t0] = 1.0
    y, _ = P.short_conv(x, w)
    expect = np.zeros((T, C))
    expect[t0] = 1.0
    for d in range(P.W):
        expect[t0 + d] += w[:, d]
    np.testing.assert_allclose(y, expect, rtol=0, atol=1e-15)


def test_conv_is_causal_and_linear():
    rng = np.random.default_rng(2)
    C, T = 4, 10
    w = _rand(rng, C, P.W)
    x1, x2 = _rand(rng, T, C), _rand(rng, T, C)
    y1, _ = P.short_conv(x1, w)
    y2, _ = P.short_conv(x2, w)
    y12, _ = P.short_conv(2.0 * x1 - 3.0 * x2, w)
    np.testing.assert_allclose(y12, 2.0 * y1 - 3.0 * y2, atol=1e-12)
    x3 = x1.copy()
    x3[6:] += 5.0                      # change only rows >= 6
    y3, _ = P.short_conv(x3, w)
    np.testing.assert_array_equal(y3[:6], y1[:6])


def test_chunks_with_state_equal_one_pass():
    rng = np.random.default_rng(3)
    C, T = 8, 11
    w = _rand(rng, C, P.W)
    x = _rand(rng, T, C)
    y_all, st_all = P.short_conv(x, w)
    for cut in (1, 2, 3, 5, 10):
        ya, sa = P.short_conv(x[:cut], w)
        yb, sb = P.short_conv(x[cut:], w, sa)
        np.testing.assert_allclose(np.concatenate([ya, yb]), y_all, atol=1e-13)
        np.testing.assert_array_equal(sb, st_all)


def test_rms_norm_gives_unit_rms_and_gamma_scales():
    rng = np.random.default_rng(4)
    x = _rand(rng, 3, 5, 128) * 7.0
    eps = 1e-6
    y = P.rms_norm(x, np.ones(128), eps)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-12)
    g = _rand(rng, 128)
    np.testing.assert_allclose(P.rms_norm(x, g, eps), y * g, rtol=1e-12)
    # a row of zeros stays zero
    np.testing.assert_array_equal(P.rms_norm(np.zeros((1, 128)), g, eps), np.zeros((1, 128)))


def _chunk_inputs(rng, lens, Hq=4, Hkv=2):
    T = sum(lens)
    q = _rand(rng, T, Hq, 128)
    k = _rand(rng, T, Hkv, 128)
    v = _rand(rng, T, Hkv, 128)
    wk = _rand(rng, Hkv * 128, P.W) * 0.3
    wv = _rand(rng, Hkv * 128, P.W) * 0.3
    gq, gk = _rand(rng, 128), _rand(rng, 128)
    return q, k, v, wk, wv, gq, gk


def test_packed_sequences_are_independent_and_rows_bottom_right():
    rng = np.random.default_rng(5)
    lens = [5, 1, 7]
    q, k, v, wk, wv, gq, gk = _chunk_inputs(rng, lens)
    cq = np.cumsum([0] + lens)
    kl = [9, 1, 12]                                    # cache lengths: the chunk is the tail
    ck = np.cumsum([0] + kl)
    out = P.prologue(q, k, v, wk, wv, gq, gk, cq, ck)
    # rows: the last Lq of each sequence's Lk
    expect_rows = np.concatenate([ck[b] + kl[b] - lens[b] + np.arange(lens[b]) for b in range(3)])
    np.testing.assert_array_equal(out["cache_rows"], expect_rows)
    # each sequence alone gives the same rows (no leak across cu_seqlens)
    for b in range(3):
        a, e = cq[b], cq[b + 1]
        one = P.prologue(q[a:e], k[a:e], v[a:e], wk, wv, gq, gk, [0, lens[b]], [0, kl[b]])
        np.testing.assert_allclose(out["k_rows"][a:e], one["k_rows"], atol=1e-13)
        np.testing.assert_allclose(out["v_rows"][a:e], one["v_rows"], atol=1e-13)


def test_prologue_chunking_with_state_equals_whole_sequence():
    rng = np.random.default_rng(6)
    L = 10
    q, k, v, wk, wv, gq, gk = _chunk_inputs(rng, [L])
    whole = P.prologue(q, k, v, wk, wv, gq, gk, [0, L], [0, L])
    cut = 4
    first = P.prologue(q[:cut], k[:cut], v[:cut], wk, wv, gq, gk, [0, cut], [0, cut])
    second = P.prologue(q[cut:], k[cut:], v[cut:], wk, wv, gq, gk, [0, L - cut], [0, L],
                        state_k=first["state_k"], state_v=first["state_v"])
    np.testing.assert_allclose(np.concatenate([first["k_rows"], second["k_rows"]]),
                               whole["k_rows"], atol=1e-12)
    np.testing.assert_allclose(np.concatenate([first["v_rows"], second["v_rows"]]),
                               whole["v_rows"], atol=1e-12)
    np.testing.assert_array_equal(second["cache_rows"], np.arange(cut, L))
    np.testing.assert_array_equal(second["state_k"], whole["state_k"])


def test_v_is_only_convolved_and_q_only_normalised():
    rng = np.random.default_rng(7)
    q, k, v, wk, wv, gq, gk = _chunk_inputs(rng, [6])
    out = P.prologue(q, k, v, np.zeros_like(wk), np.zeros_like(wv), gq, gk, [0, 6], [0, 6])
    np.testing.assert_array_equal(out["v_rows"], v)             # zero taps: v unchanged
    ms = np.mean(k * k, axis=-1, keepdims=True)
    np.testing.assert_allclose(out["k_rows"], k / np.sqrt(ms + 1e-6) * gk, rtol=1e-12)
    msq = np.mean(q * q, axis=-1, keepdims=True)
    np.testing.assert_allclose(out["q_out"], q / np.sqrt(msq + 1e-6) * gq, rtol=1e-12)


def test_empty_chunk_passes_the_state_through():
    rng = np.random.default_rng(8)
    q, k, v, wk, wv, gq, gk = _chunk_inputs(rng, [0, 3])
    sk = _rand(rng, 2, P.W - 1, 2 * 128)
    sv = _rand(rng, 2, P.W - 1, 2 * 128)
    out = P.prologue(q, k, v, wk, wv, gq, gk, [0, 0, 3], [0, 5, 8], state_k=sk, state_v=sv)
    np.testing.assert_array_equal(out["state_k"][0], sk[0])
    np.testing.assert_array_equal(out["state_v"][0], sv[0])
    # the other sequence's state is its last 3 inputs
    np.testing.assert_array_equal(out["state_k"][1], k.reshape(3, -1))
    np.testing.assert_array_equal(out["cache_rows"], [5, 6, 7])
