"""Decode against a paged KV cache (relattn_decode_paged) on the GPU.

Each case scatters the contiguous K / V rows of a seeded workload into a
shuffled page pool. The tail of each sequence's last page, and some spare
pages, hold 1e4, so a key read by mistake would show. Three checks follow:
- paged out / lse equal the contiguous relattn_decode bit for bit (same split
  plan, same tiles, same arithmetic);
- both match the fp64 oracle within the forward's tolerance;
- a page number outside the pool is reported and reads as zero.
"""
import numpy as np
import pytest
import torch

from tests.conftest import gpu_available
from tests.parity_util import compare
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


def _kw(w):
    return dict(max_seqlen_q=max(w.q_lens), max_seqlen_k=max(w.k_lens), alpha=w.alpha,
                window=w.window, log_scale_base=w.log_scale_base)


def run_both(w, page_size, seed=0):
    import relative_position_biased_gb300 as rpb
    inp = W.make_inputs(w)
    kp, vp, table = W.page_kv(inp["k"], inp["v"], w.k_lens, page_size, seed=seed)
    d = {k: v.cuda() for k, v in inp.items()}
    out_c, lse_c = rpb.decode(d["q"], d["k"], d["v"], d["r"], d["P"], d["cu_seqlens_q"],
                              d["cu_seqlens_k"], **_kw(w))
    out_p, lse_p = rpb.decode_paged(d["q"], kp.cuda(), vp.cuda(), d["r"], d["P"],
                                    d["cu_seqlens_q"], d["cu_seqlens_k"], table.cuda(),
                                    page_size=page_size, **_kw(w))
    torch.cuda.synchronize()
    st = rpb.relattn_get_device_error()
    assert st == rpb.RELATTN_OK, rpb.STATUS_NAMES.get(st, st)
    return inp, (out_c, lse_c), (out_p, lse_p)


def check(w, page_size):
    inp, (oc, lc), (op, lp) = run_both(w, page_size)
    assert torch.equal(op, oc) and torch.equal(lp, lc), "paged differs from contiguous"
    compare(w, inp, (op.float().cpu().numpy(), lp.cpu().numpy()))


@pytest.mark.parametrize("page_size", [128, 256, 1024])
def test_batched_decode(page_size):
    w = W.custom("paged_b16", [1] * 16, [int(x) for x in np.random.default_rng(1).integers(1, 3000, 16)],
                 16, 2, 64, 1024, log_scale_base=65536.0)
    check(w, page_size)


def test_mtp_rows_with_short_and_long_sequences():
    check(W.custom("paged_mtp", [9, 9, 3], [9, 5000, 130], 16, 2, 64, 256), 128)


def test_sliding_window_decode():
    check(W.custom("paged_win", [1, 4], [6000, 3000], 16, 2, 64, 1024, window=1024), 256)


def test_gqa4_no_bias():
    check(W.custom("paged_nobias", [1, 2], [700, 129], 8, 2, 0, 0), 128)


@pytest.mark.slow
def test_long_context_mtp_verify():
    # the 9-row MTP verify against 1,048,576 keys, through 128-key pages
    w = W.decode_mtp_long()
    inp, (oc, lc), (op, lp) = run_both(w, 128)
    assert torch.equal(op, oc) and torch.equal(lp, lc)


def test_page_outside_the_pool_is_reported():
    import relative_position_biased_gb300 as rpb
    w = W.custom("paged_bad", [1], [300], 4, 1, 32, 64)
    inp = W.make_inputs(w)
    kp, vp, table = W.page_kv(inp["k"], inp["v"], w.k_lens, 128)
    table[0, 1] = 10_000                      # past the pool: its keys read as zero
    d = {k: v.cuda() for k, v in inp.items()}
    out, lse = rpb.decode_paged(d["q"], kp.cuda(), vp.cuda(), d["r"], d["P"], d["cu_seqlens_q"],
                                d["cu_seqlens_k"], table.cuda(), page_size=128, **_kw(w))
    torch.cuda.synchronize()
    assert rpb.relattn_get_device_error() == 6          # RELATTN_ERR_DEVICE_ARGS
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
