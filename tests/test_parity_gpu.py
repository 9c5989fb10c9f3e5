"""CUDA path vs fp64 oracle, element by element, through the C ABI.

Tolerance: bf16 inputs, fp32 accumulation, bf16 out: max |dout| <= 2e-2 and
max |dlse| <= 1e-3 (natural log) over every checked row and head.
"""
import numpy as np
import pytest
import torch

from tests.conftest import gpu_available
from tests.parity_util import compare, run_gpu, sample_rows
from relative_position_biased_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import relative_position_biased_gb300 as rpb
    rpb.build()
    rpb.load_library()
    import oracle
    oracle.build()


def _check(w, rows=None, **kw):
    inp = W.make_inputs(w)
    return compare(w, inp, run_gpu(w, inp, **kw), rows=rows)


# ------------------------------------------------------------------ prefill

def test_tiny_full_causal():
    _check(W.tiny_full())


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 200, 383])
def test_prefill_ragged_lengths(T):
    _check(W.custom(f"ragged{T}", [T], [T], 4, 2, 32, 64))


def test_prefill_varlen_with_empty_sequences():
    lens = [0, 1, 130, 0, 257, 64]
    _check(W.custom("varlen_empty", lens, lens, 4, 1, 16, 48))


@pytest.mark.parametrize("window", [1, 2, 5, 64, 100, 129, 1000])
def test_prefill_sliding_window(window):
    _check(W.custom(f"win{window}", [300, 77], [300, 77], 4, 2, 32, 40, window=window))


@pytest.mark.parametrize("r_dim,E", [(1, 64), (4, 7), (16, 1), (32, 100), (64, 512), (64, 3),
                                     (8, 1000), (0, 64), (32, 0)])
def test_prefill_bias_shapes(r_dim, E):
    _check(W.custom(f"rd{r_dim}_E{E}", [333], [333], 2, 1, r_dim, E))


def test_prefill_log_scale():
    _check(W.custom("logscale", [400], [400], 4, 2, 32, 64, log_scale_base=16.0))


def test_prefill_log_scale_window():
    _check(W.custom("logscale_win", [400], [400], 4, 2, 32, 64, window=50, log_scale_base=8.0))


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (3, 3), (8, 1), (16, 2)])
def test_prefill_gqa_groupings(Hq, Hkv):
    _check(W.custom(f"gqa{Hq}_{Hkv}", [150], [150], Hq, Hkv, 16, 32))


def test_prefill_large_bias():
    """P with std 1 makes the bias dominate the logit (stress of the gather)."""
    _check(W.custom("bigP", [260], [260], 2, 1, 64, 256, p_std=1.0))


def test_chunked_prefill_bottom_right():
    """Lq < Lk through the prefill kernel: rows sit at the end of the keys."""
    _check(W.custom("chunked", [100, 37], [300, 37 + 200], 4, 2, 32, 64))
    _check(W.custom("chunked_win", [130], [1000], 4, 2, 32, 64, window=256))


# ------------------------------------------------- persistent bias-band launch
# The two-launch prefill (bias band, then the rest) runs its band launch with
# one CTA per SM, each walking several (row tile, sequence, head) items.  The
# test hook caps the CTA count so that small cases take the item-to-item paths
# (stage rings and barrier phases carried over, the next item's q / r rows
# staged during the previous item's epilogue).

@pytest.fixture
def band_ctas():
    """The CTA cap lives in the test build of the library: the test's calls
    run on it while the fixture is active."""
    import relative_position_biased_gb300 as rpb

    def set_cap(n):
        assert rpb.relattn_test_band_ctas(n) == 0

    with rpb.test_library():
        try:
            yield set_cap
        finally:
            rpb.relattn_test_band_ctas(0)


@pytest.mark.parametrize("ctas", [1, 3])
def test_band_ctas_walk_many_items(band_ctas, ctas):
    """Items with different band lengths (short, empty and ragged sequences) in one CTA."""
    band_ctas(ctas)
    lens = [333, 77, 520, 1, 129, 0, 256]
    _check(W.custom(f"persist{ctas}", lens, lens, 4, 2, 32, 104))


def test_band_ctas_rows_staged_by_softmax(band_ctas):
    """r_dim 40 (not a multiple of 16): the softmax warps stage the q / r rows."""
    band_ctas(2)
    _check(W.custom("persist_rd40", [300, 200], [300, 200], 4, 2, 40, 200, window=250))


def test_band_ctas_log_scale_chunked(band_ctas):
    band_ctas(2)
    _check(W.custom("persist_ls", [130, 260], [400, 300], 4, 2, 64, 128, log_scale_base=16.0))


@pytest.mark.parametrize("ctas", [0, 2])
def test_band_many_sequences(band_ctas, ctas):
    """More sequences than the per-CTA copy of the sequence offsets holds (64)."""
    band_ctas(ctas)
    lens = np.random.default_rng(7).integers(1, 150, size=70).tolist()
    _check(W.custom(f"many_seqs{ctas}", lens, lens, 2, 1, 16, 64))


@pytest.mark.parametrize("alpha", [-0.0883883, 0.0, 0.5])
def test_prefill_alpha(alpha):
    """alpha < 0 (the score sign is folded into q; one-launch path), alpha = 0
    (the logits are the bias alone) and a large alpha (steep softmax, O rescales)."""
    _check(W.custom(f"alpha{alpha}", [300, 130], [300, 130], 4, 2, 32, 200, alpha=alpha))


def test_single_key_rows_exact():
    """window = 1: every row sees only itself, so out is v exactly."""
    w = W.custom("win1", [200], [200], 4, 2, 32, 64, window=1)
    inp = W.make_inputs(w)
    out, _ = run_gpu(w, inp)
    v = inp["v"].float().numpy().repeat(2, axis=1)
    assert np.array_equal(out, v)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("splits", [1, 2, 3, 0])
@pytest.mark.parametrize("Lq", [1, 2, 9, 16])
def test_decode_splits(Lq, splits):
    ks = [700, 1500, 64 + Lq, Lq]
    _check(W.custom(f"dec{Lq}", [Lq] * 4, ks, 16, 2, 32, 256), decode=True, num_splits=splits)


# Few-row decode bias sources: in the kernel on the tensor cores (r_dim a
# multiple of 8 up to 64, rel_extent a multiple of 8 up to 1024: one to eight
# blocks of 128 distances, full and partial), else computed by a kernel
# before the decode (E = 1, r_dim 20, E = 1032 and 1500: past the eight
# blocks).  One token per sequence (one distance per item) and two (a
# distance per token), full and windowed keys.
@pytest.mark.parametrize("rd,E", [(8, 64), (16, 136), (24, 640), (40, 120), (64, 1024),
                                  (8, 1), (20, 700), (64, 1032), (64, 1500)])
@pytest.mark.parametrize("Lq,window", [(1, 0), (2, 0), (1, 900)])
def test_decode_bias_sources(rd, E, Lq, window):
    ks = [2500, 1300, 129, 600 + Lq, Lq]
    _check(W.custom(f"dec_bias{rd}_{E}", [Lq] * len(ks), ks, 16, 2, rd, E, window=window), decode=True,
           num_splits=2)


# The stream-K walk of the few-row decode (several splits, at most 64
# sequences): CTA c takes an equal range of the units' tiles laid end to end.
# Cases: sequences without query rows between others (units of no rows), a
# unit far longer than the others (it meets the most ranges, up to the split
# count), CTA counts that put range boundaries on and off unit boundaries,
# many splits over few tiles (the range size held at its lower bound), the
# window, and two tokens per sequence.
@pytest.mark.parametrize("ctas,splits", [(0, 2), (0, 8), (5, 3), (7, 6), (2, 16)])
def test_decode_stream_k_ranges(band_ctas, ctas, splits):
    band_ctas(ctas)
    q = [1, 0, 1, 1, 0, 1, 1, 1]
    ks = [1, 5, 9000, 130, 777, 2048, 257, 3333]
    _check(W.custom(f"sk{ctas}_{splits}", q, ks, 16, 2, 64, 1024), decode=True, num_splits=splits)


@pytest.mark.parametrize("splits", [3, 5])
def test_decode_stream_k_window_two_tokens(band_ctas, splits):
    band_ctas(11)
    ks = [4100, 260, 6000, 2, 1500]
    _check(W.custom(f"skw{splits}", [2] * len(ks), ks, 16, 2, 32, 512, window=1100), decode=True,
           num_splits=splits)


@pytest.mark.parametrize("window", [1, 5, 300])
def test_decode_window(window):
    ks = [700, 1500, 300]
    _check(W.custom(f"decw{window}", [9] * 3, ks, 8, 2, 32, 128, window=window), decode=True)


@pytest.mark.parametrize("alpha", [-0.0883883, 0.0, 0.5])
def test_decode_alpha(alpha):
    _check(W.custom(f"dalpha{alpha}", [9, 1], [3000, 800], 16, 2, 32, 256, alpha=alpha), decode=True)


def test_decode_log_scale_and_gqa1():
    _check(W.custom("dec_ls", [16, 3], [2000, 40], 4, 4, 16, 100, log_scale_base=32.0),
           decode=True)


def test_decode_group16_row_blocks():
    """Hq/Hkv = 16 with 16 query rows: 256 rows span two 128-row blocks."""
    _check(W.custom("dec_g16", [16], [900], 16, 1, 32, 64), decode=True)


def test_decode_matches_prefill_tail():
    """Decode rows equal the last rows of a prefill over the same sequence."""
    import relative_position_biased_gb300 as rpb
    T, Lq = 1000, 9
    w = W.custom("tail", [T], [T], 8, 2, 32, 200, log_scale_base=64.0)
    inp = W.make_inputs(w)
    pre_out, pre_lse = run_gpu(w, inp, decode=False)
    dec_inp = dict(inp)
    dec_inp["q"], dec_inp["r"] = inp["q"][-Lq:].contiguous(), inp["r"][-Lq:].contiguous()
    dec_inp["cu_seqlens_q"] = torch.tensor([0, Lq], dtype=torch.int32)
    wd = W.custom("tail_dec", [Lq], [T], 8, 2, 32, 200, log_scale_base=64.0)
    dec_out, dec_lse = run_gpu(wd, dec_inp, decode=True, num_splits=4)
    assert np.max(np.abs(dec_out - pre_out[-Lq:])) <= 2e-2
    assert np.max(np.abs(dec_lse - pre_lse[:, -Lq:])) <= 1e-3
    assert rpb.relattn_get_device_error() == 0


# ------------------------------------------------------------------ full-size workloads

# Decode CTAs walk (sequence, split, kv head, row block) items too, the
# longest first: full chunks, then partial chunks by size, then the rest,
# dealt round by round with every other full round reversed. The cap makes
# each CTA take many items, so these cases cover:
# - empty and one-key splits;
# - a partial last round;
# - two row blocks;
# - windows;
# - more sequences than the work-order tables hold, which takes the plain order.

@pytest.mark.parametrize("ctas", [1, 3, 7])
@pytest.mark.parametrize("splits", [0, 5])
def test_decode_ctas_walk_many_items(band_ctas, ctas, splits):
    band_ctas(ctas)
    ks = [1, 4000, 130, 900, 2, 2600, 129, 1500]
    _check(W.custom(f"dec_persist{ctas}", [1] * len(ks), ks, 16, 2, 32, 256), decode=True,
           num_splits=splits)


def test_decode_ctas_mtp_rows_window(band_ctas):
    band_ctas(4)
    ks = [3000, 40, 1200, 2048]
    _check(W.custom("dec_persist_w", [9] * len(ks), ks, 8, 2, 32, 128, window=700), decode=True,
           num_splits=3)


def test_decode_ctas_row_blocks(band_ctas):
    band_ctas(2)
    _check(W.custom("dec_persist_g16", [16, 16], [900, 300], 16, 1, 32, 64), decode=True, num_splits=2)


@pytest.mark.parametrize("ctas", [0, 5])
def test_decode_many_sequences(band_ctas, ctas):
    """70 sequences: more than the work-order tables hold (plain order)."""
    band_ctas(ctas)
    ks = (np.random.default_rng(11).integers(1, 700, size=70) + 1).tolist()
    _check(W.custom(f"dec_many{ctas}", [1] * 70, ks, 4, 1, 16, 64), decode=True, num_splits=2)


def test_workload_tiny():
    _check(W.tiny_full())


def test_workload_swa_prefill_sampled():
    w = W.swa_prefill()
    _check(w, rows=sample_rows(w))


def test_workload_full_prefill_logscale_sampled():
    w = W.full_prefill_logscale()
    _check(w, rows=sample_rows(w, n_random=32))


def test_workload_decode_batched():
    _check(W.decode_batched())


def test_workload_decode_batched_window():
    _check(W.decode_batched(window=4096))


def test_workload_decode_mtp_long():
    _check(W.decode_mtp_long())


# ------------------------------------------------------------------ device-side checks

def test_inconsistent_seqlens_reported_not_faulted():
    """Lk < Lq for one sequence: that sequence is skipped and the device error
    word reports it; the others still compute."""
    import relative_position_biased_gb300 as rpb
    w = W.custom("bad", [50, 20], [50, 20], 2, 1, 16, 32)
    inp = W.make_inputs(w)
    dev = {k: v.cuda() for k, v in inp.items()}
    cu_k = torch.tensor([0, 50, 60], dtype=torch.int32, device="cuda")  # 2nd: Lk=10 < Lq=20
    rpb.prefill(dev["q"], dev["k"], dev["v"], dev["r"], dev["P"], dev["cu_seqlens_q"], cu_k,
                max_seqlen_q=50, max_seqlen_k=50, alpha=w.alpha)
    torch.cuda.synchronize()
    assert rpb.relattn_get_device_error() == 6
    assert rpb.relattn_get_device_error() == 0   # reading clears it
