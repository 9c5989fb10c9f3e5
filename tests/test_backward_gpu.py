"""Backward pass on the GPU (dq, dk, dv, dr; P frozen) against the fp64
backward oracle, through the C ABI.

The GPU backward reads the GPU forward's out / lse, as a training step does.

Tolerance, from the arithmetic: every product term of dq, dk, dv and dr has
exactly one factor rounded to bf16 for the tensor cores, P for dv and dS for
the others, with relative error at most 2^-9. Each result is rounded once more
to bf16, also at most 2^-9. D uses the bf16 out. Sums of such terms stay
within about 2 x 2^-9 of the reference in the Frobenius norm. The tests allow:
- ||gpu - ref|| <= 2^-7 ||ref||;
- max |gpu - ref| <= 2^-6 max |ref|, per tensor.
The observed values are about 2.5e-3 and 5e-3.

Where the exact gradient vanishes, e.g. dq of a row with one visible key, the
GPU value is fp32 cancellation noise, around 1e-7. So both norms are taken
against at least SCALE_FLOOR = 1e-2. That is far above that noise and well
below the O(1) size the gradients have with N(0, 1) inputs.
"""
import numpy as np
import pytest
import torch

from tests.conftest import gpu_available
from relative_position_biased_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]

FRO_TOL = 2.0 ** -7
MAX_TOL = 2.0 ** -6
SCALE_FLOOR = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import relative_position_biased_gb300 as rpb
    rpb.build()
    rpb.load_library()
    import oracle
    oracle.build()


def _kw(w):
    return dict(max_seqlen_q=max(w.q_lens), max_seqlen_k=max(w.k_lens), alpha=w.alpha,
                window=w.window, log_scale_base=w.log_scale_base)


def run_gpu(w, inp):
    import relative_position_biased_gb300 as rpb
    d = {k: v.cuda() for k, v in inp.items()}
    args = (d["q"], d["k"], d["v"], d["r"], d["P"])
    out, lse = rpb.prefill(*args, d["cu_seqlens_q"], d["cu_seqlens_k"], **_kw(w))
    grads = rpb.backward(*args, out, lse, d["dout"], d["cu_seqlens_q"], d["cu_seqlens_k"], **_kw(w))
    torch.cuda.synchronize()
    st = rpb.relattn_get_device_error()
    assert st == rpb.RELATTN_OK, rpb.STATUS_NAMES.get(st, st)
    return [None if g is None else g.float().cpu().double().numpy() for g in grads]


def run_oracle(w, inp):
    import oracle
    return oracle.backward(inp["q"], inp["k"], inp["v"], inp["r"], inp["P"], inp["dout"],
                           inp["cu_seqlens_q"], inp["cu_seqlens_k"], alpha=w.alpha,
                           window=w.window, log_scale_base=w.log_scale_base)


def assert_close(got, ref, name):
    assert got.shape == ref.shape, name
    assert np.isfinite(got).all(), name
    scale = max(np.abs(ref).max(), SCALE_FLOOR)
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), SCALE_FLOOR)
    mx = np.abs(got - ref).max() / scale
    assert fro <= FRO_TOL and mx <= MAX_TOL, (name, fro, mx)


def check(w):
    inp = W.make_inputs(w, with_dout=True)
    got = run_gpu(w, inp)
    ref = run_oracle(w, inp)
    for name, g, r in zip(("dq", "dk", "dv", "dr"), got, ref):
        if r.size == 0:
            assert g is None or g.size == 0
            continue
        assert_close(g, r, name)
    return got, ref, inp


def test_tiny_full():
    check(W.tiny_full())


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 200])
def test_ragged_lengths(T):
    check(W.custom(f"bwd{T}", [T], [T], 4, 2, 32, 64))


def test_packed_chunks_after_a_prefix():
    check(W.custom("bwd_chunks", [50, 100, 1], [80, 100, 40], 4, 2, 32, 64))


@pytest.mark.parametrize("window,E", [(70, 48), (40, 64), (1, 16)])
def test_sliding_window(window, E):
    check(W.custom(f"bwd_w{window}", [300], [300], 4, 1, 32, E, window=window))


def test_log_scale():
    check(W.custom("bwd_log", [180, 90], [180, 90], 4, 2, 16, 64, log_scale_base=16.0))


def test_gqa8_band_beyond_extent():
    # 16 q heads on 2 kv heads, r_dim 64, E 1024, rows past the band
    check(W.custom("bwd_gqa8", [1500], [1500], 16, 2, 64, 1024))


def test_extent_not_a_multiple_of_8():
    check(W.custom("bwd_E100", [260], [260], 4, 2, 24, 100))


def test_without_bias():
    got, _, _ = check(W.custom("bwd_nobias", [130], [130], 4, 2, 0, 0))
    assert got[3] is None


def test_r_without_extent_gives_zero_dr():
    got, _, _ = check(W.custom("bwd_E0", [70], [70], 4, 2, 16, 0))
    assert not got[3].any()


def test_keys_no_query_sees_get_zero_gradients():
    # a 40-row chunk at the end of 400 keys with a window of 50: keys before
    # 400 - 40 - 49 are outside every row's window
    w = W.custom("bwd_winchunk", [40], [400], 4, 2, 32, 64, window=50)
    got, _, _ = check(w)
    first_seen = 400 - 40 - 50 + 1
    assert not got[1][:first_seen].any() and not got[2][:first_seen].any()


def test_empty_chunk_zeroes_the_key_gradients():
    import relative_position_biased_gb300 as rpb
    w = W.custom("bwd_empty", [0, 0], [30, 5], 4, 2, 16, 32)
    d = {k: v.cuda() for k, v in W.make_inputs(w, with_dout=True).items()}
    out = torch.empty_like(d["q"])
    lse = torch.empty(4, 0, dtype=torch.float32, device="cuda")
    dk = torch.full_like(d["k"], 7.0)
    dv = torch.full_like(d["v"], 7.0)
    rpb.backward(d["q"], d["k"], d["v"], d["r"], d["P"], out, lse, d["dout"], d["cu_seqlens_q"],
                 d["cu_seqlens_k"], max_seqlen_q=0, max_seqlen_k=30, alpha=w.alpha, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert not dk.any() and not dv.any()


def test_inconsistent_cu_seqlens_are_reported():
    import relative_position_biased_gb300 as rpb
    w = W.custom("bwd_bad", [8], [8], 4, 2, 16, 32)
    d = {k: v.cuda() for k, v in W.make_inputs(w, with_dout=True).items()}
    out, lse = rpb.prefill(d["q"], d["k"], d["v"], d["r"], d["P"], d["cu_seqlens_q"],
                           d["cu_seqlens_k"], **_kw(w))
    bad_k = torch.tensor([0, 4], dtype=torch.int32, device="cuda")        # Lk 4 < Lq 8
    rpb.backward(d["q"], d["k"], d["v"], d["r"], d["P"], out, lse, d["dout"], d["cu_seqlens_q"],
                 bad_k, max_seqlen_q=8, max_seqlen_k=8, alpha=w.alpha)
    torch.cuda.synchronize()
    assert rpb.relattn_get_device_error() == 6          # RELATTN_ERR_DEVICE_ARGS
    assert rpb.relattn_get_device_error() == rpb.RELATTN_OK


def test_split_reduce_touches_only_rows_it_wrote():
    """GQA 4:1 (dk / dv split over two CTAs per key tile, then the reduce)
    with K / V tensors longer than cu_seqlens_k[batch]: the rows past it keep
    their contents, as on the unsplit path, and the rows inside match the
    oracle."""
    import relative_position_biased_gb300 as rpb
    w = W.custom("bwd_pad", [100, 60], [100, 60], 8, 2, 32, 64)
    inp = W.make_inputs(w, with_dout=True)
    d = {k: v.cuda() for k, v in inp.items()}
    pad = torch.randn(30, 2, 128, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    kp, vp = torch.cat([d["k"], pad]), torch.cat([d["v"], pad])
    args = (d["q"], kp, vp, d["r"], d["P"])
    out, lse = rpb.prefill(*args, d["cu_seqlens_q"], d["cu_seqlens_k"], **_kw(w))
    dk, dv = torch.full_like(kp, 7.0), torch.full_like(vp, 7.0)
    rpb.backward(*args, out, lse, d["dout"], d["cu_seqlens_q"], d["cu_seqlens_k"], dk=dk, dv=dv,
                 **_kw(w))
    torch.cuda.synchronize()
    assert rpb.relattn_get_device_error() == rpb.RELATTN_OK
    assert bool((dk[160:] == 7.0).all()) and bool((dv[160:] == 7.0).all())
    ref = run_oracle(w, inp)
    assert_close(dk[:160].float().cpu().double().numpy(), ref[1], "dk")
    assert_close(dv[:160].float().cpu().double().numpy(), ref[2], "dv")


def test_split_reduce_skips_a_sequence_the_kernels_skipped():
    """GQA 4:1; the second sequence has Lk < Lq: the kernels skip it and
    report it, and the reduce leaves its dk / dv rows as they were."""
    import relative_position_biased_gb300 as rpb
    w = W.custom("bwd_badseq", [100, 60], [100, 60], 8, 2, 32, 64)
    inp = W.make_inputs(w, with_dout=True)
    d = {k: v.cuda() for k, v in inp.items()}
    args = (d["q"], d["k"], d["v"], d["r"], d["P"])
    out, lse = rpb.prefill(*args, d["cu_seqlens_q"], d["cu_seqlens_k"], **_kw(w))
    bad_k = torch.tensor([0, 100, 140], dtype=torch.int32, device="cuda")   # Lk 40 < Lq 60
    dk, dv = torch.full_like(d["k"], 7.0), torch.full_like(d["v"], 7.0)
    rpb.backward(*args, out, lse, d["dout"], d["cu_seqlens_q"], bad_k, dk=dk, dv=dv, **_kw(w))
    torch.cuda.synchronize()
    assert rpb.relattn_get_device_error() == 6          # RELATTN_ERR_DEVICE_ARGS
    assert bool((dk[100:] == 7.0).all()) and bool((dv[100:] == 7.0).all())
    w0 = W.custom("bwd_badseq0", [100], [100], 8, 2, 32, 64)
    sub = {k: inp[k][:100] for k in ("q", "k", "v", "r", "dout")}
    ref = run_oracle(w0, dict(sub, P=inp["P"], cu_seqlens_q=[0, 100], cu_seqlens_k=[0, 100]))
    assert_close(dk[:100].float().cpu().double().numpy(), ref[1], "dk")
    assert_close(dv[:100].float().cpu().double().numpy(), ref[2], "dv")


@pytest.mark.slow
def test_full_size_swa_prefill():
    """4 x 8192 packed, window 4096, E 1024, r_dim 64, Hq 16 / Hkv 2: the
    workload the bench times, with the dq split and the dk / dv split over
    two CTAs per key tile.

    dq and dr of sampled rows against the oracle on that row alone (a
    one-row chunk at the end of its sequence's keys: dq_i and dr_i depend on
    row i only).  dk and dv element by element on sampled key ranges: a
    sequence start (band tiles near the first rows), a range across the
    4096 boundary (band and non-band tiles, the window edge), and a sequence
    end (keys only the last rows see), each against the oracle run on the
    query rows that see those keys.  The softmax identities (the dk of a
    sequence sum to zero per kv head; the dv sum to the group's dout) still
    check every key at once.
    """
    import oracle
    from tests.parity_util import oracle_key_range_grads
    w = W.swa_prefill()
    inp = W.make_inputs(w, with_dout=True)
    dq, dk, dv, dr = run_gpu(w, inp)
    rng = np.random.default_rng(11)
    for t in sorted(rng.choice(sum(w.q_lens), size=6, replace=False).tolist()) + [0, 8191, 8192]:
        b, i = t // 8192, t % 8192
        k0 = b * 8192
        sub = dict(q=inp["q"][t:t + 1], k=inp["k"][k0:k0 + i + 1], v=inp["v"][k0:k0 + i + 1],
                   r=inp["r"][t:t + 1], P=inp["P"], dout=inp["dout"][t:t + 1])
        rq, _, _, rr = oracle.backward(sub["q"], sub["k"], sub["v"], sub["r"], sub["P"], sub["dout"],
                                       [0, 1], [0, i + 1], alpha=w.alpha, window=w.window)
        assert_close(dq[t:t + 1], rq, f"dq row {t}")
        assert_close(dr[t:t + 1], rr, f"dr row {t}")
    for b, j0, m in ((1, 0, 128), (2, 4096 - 64, 128), (3, 8192 - 128, 128)):
        rk, rv = oracle_key_range_grads(w, inp, b, j0, m)
        sl = slice(b * 8192 + j0, b * 8192 + j0 + m)
        assert_close(dk[sl], rk, f"dk keys {b}:{j0}+{m}")
        assert_close(dv[sl], rv, f"dv keys {b}:{j0}+{m}")
    do = inp["dout"].double().numpy()
    for b in range(4):
        sl = slice(b * 8192, (b + 1) * 8192)
        # sum of |terms| sets the rounding scale of each sum
        sk = dk[sl].sum(axis=0)
        assert np.abs(sk).max() <= 2.0 ** -7 * np.abs(dk[sl]).sum(axis=0).max(), "sum of dk"
        want = do[sl].reshape(8192, 2, 8, 128).sum(axis=(0, 2))
        err = np.abs(dv[sl].sum(axis=0) - want).max()
        assert err <= 2.0 ** -7 * np.abs(dv[sl]).sum(axis=0).max(), "sum of dv"


# dq is split: keys that every row of a 128-row query tile sees outside the
# bias band go to the tcgen05 dq kernel, the band's keys to the warp-MMA
# kernel, which adds the first part. These cases give the first kernel long
# runs of keys: with and without a window and a bias, a chunk whose keys start
# well before its queries, a short extent under long rows, many short
# sequences, GQA 8:1 and 6:1 (three heads per dk / dv CTA), an extent beyond
# the sequence and a window below the extent (no keys outside the band).
@pytest.mark.parametrize("name,q_lens,k_lens,Hq,Hkv,r_dim,E,window", [
    ("dq_nobias_long", [700], [700], 4, 2, 0, 0, 0),
    ("dq_nobias_window", [640, 333], [640, 333], 4, 1, 0, 0, 200),
    ("dq_chunk_prefix", [300, 129], [900, 600], 4, 2, 32, 64, 0),
    ("dq_chunk_prefix_nobias", [300, 129], [900, 600], 4, 2, 0, 0, 0),
    ("dq_short_extent", [777], [777], 8, 2, 16, 8, 0),
    ("dq_window_extent", [900], [900], 4, 2, 32, 100, 333),
    ("dq_many_short", [3, 130, 7, 129, 1, 64, 200], [3, 130, 7, 129, 1, 64, 260], 4, 2, 16, 32, 0),
    ("dq_gqa8", [520], [520], 16, 2, 64, 200, 0),
    ("dq_extent_beyond_len", [300], [300], 4, 2, 32, 1024, 0),
    ("dq_window_below_extent", [700], [700], 8, 2, 32, 256, 100),
    ("dq_gqa6", [400], [400], 12, 2, 16, 64, 0),
])
def test_dq_split(name, q_lens, k_lens, Hq, Hkv, r_dim, E, window):
    check(W.custom(name, q_lens, k_lens, Hq, Hkv, r_dim, E, window=window))
