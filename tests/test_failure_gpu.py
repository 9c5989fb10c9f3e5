"""Failure path of the tensor-core kernels, without faulting the GPU.

A test hook makes a TMA producer leave one tile or step unloaded, so the
waits behind it (bounded by a clock limit, about a second) run out.  The
CTA must give up cleanly: drain its own copies and MMAs, free its tensor
memory and exit; the host then reads RELATTN_ERR_TIMEOUT from the device
error word, with the first wait site that gave up in bits 8+, and the
context stays usable for the next, normal call.

The hooks exist only in the test build of the library (librelattn_test.so);
every test here runs its calls on that build, and the product library is
checked to have none of them.
"""
import pytest
import torch

import relative_position_biased_gb300 as rpb
from relative_position_biased_gb300 import workloads as W

from tests.parity_util import compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _test_build():
    rpb.build()
    with rpb.test_library():
        yield


def test_product_library_has_no_hooks():
    prod = rpb.load_library(rpb.LIB_PATH)
    for name in rpb.TEST_HOOKS:
        assert not hasattr(prod, name), name


def test_bounded_wait_gives_up_and_context_recovers(oracle_mod):
    # 384 tokens, no bias: the tensor-core path; the CTAs of the last two
    # query tiles visit 2 and 3 key tiles, so key tile 1 is on their path
    w = W.custom("fail_t384", [384], [384], 2, 1, 0, 64)
    inp = W.make_inputs(w)
    dev = {k: v.cuda() for k, v in inp.items()}
    args = [dev[k] for k in ("q", "k", "v", "r", "P", "cu_seqlens_q", "cu_seqlens_k")]
    kw = dict(max_seqlen_q=384, max_seqlen_k=384, alpha=w.alpha, window=0, log_scale_base=0.0)
    assert rpb.relattn_get_device_error() == rpb.RELATTN_OK   # start clean
    assert rpb.relattn_test_skip_k_tile(1) == rpb.RELATTN_OK
    try:
        rpb.prefill(*args, **kw)          # the launch itself succeeds
        torch.cuda.synchronize()          # and the CTAs finish (no hang)
        st = rpb.relattn_get_device_error()
        word = rpb.relattn_last_device_error_word()
    finally:
        rpb.relattn_test_skip_k_tile(-1)
    assert st == rpb.RELATTN_ERR_TIMEOUT, (rpb.STATUS_NAMES.get(st, st), hex(word))
    assert word & 2 and (word >> 8) > 0
    # the same call, hook off: correct results on the same context
    compare(w, inp, run_gpu(w, inp))


def test_skip_hook_rejects_bad_tile():
    assert rpb.relattn_test_skip_k_tile(-2) != rpb.RELATTN_OK
    assert rpb.relattn_test_skip_k_tile(-1) == rpb.RELATTN_OK


def test_prologue_wait_gives_up_and_context_recovers():
    """The staged prologue kernel: its producer leaves token tile 3 without
    copies, so the consumer warps' bounded waits on that stage run out; the
    CTA drains and exits, RELATTN_ERR_TIMEOUT is read back, and the next
    call on the same context is correct."""
    from tests.test_prologue_gpu import check, _w
    w = _w([100, 100])                   # 25 tiles of 8 tokens (Hq 16, Hkv 2)
    inp = W.make_prologue_inputs(w)
    d = {k: v.cuda() for k, v in inp.items()}
    kc = torch.zeros(200, 2, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    assert rpb.relattn_get_device_error() == rpb.RELATTN_OK   # start clean
    assert rpb.relattn_test_prologue_skip_tile(3) == rpb.RELATTN_OK
    try:
        rpb.prologue(d["q"], d["k"], d["v"], d["conv_k"], d["conv_v"], d["norm_q"], d["norm_k"],
                     d["cu_seqlens_q"], d["cu_seqlens_k"], kc, vc)
        torch.cuda.synchronize()          # the CTAs finish (no hang)
        st = rpb.relattn_get_device_error()
        word = rpb.relattn_last_device_error_word()
    finally:
        rpb.relattn_test_prologue_skip_tile(-1)
    assert st == rpb.RELATTN_ERR_TIMEOUT, (rpb.STATUS_NAMES.get(st, st), hex(word))
    assert word & 2 and (word >> 8) > 0
    check(w)                              # hook off: correct on the same context


def test_prologue_skip_hook_rejects_bad_tile():
    assert rpb.relattn_test_prologue_skip_tile(-2) != rpb.RELATTN_OK
    assert rpb.relattn_test_prologue_skip_tile(-1) == rpb.RELATTN_OK


# wait sites of the two tcgen05 backward kernels (the ids their bounded waits
# record): the dk / dv kernel 1-10, the dq kernel outside the band 11-16
BWD_SITES = {0: range(1, 11), 1: range(11, 17)}


@pytest.mark.parametrize("kernel", [0, 1])
def test_backward_skip_hook_times_out_and_recovers(kernel):
    """One tcgen05 backward kernel's producer (kernel 0: dk / dv, 1: dq)
    leaves its step 0 without copies: the waits behind it run out, every CTA
    of that kernel drains and frees its tensor memory, the status is
    RELATTN_ERR_TIMEOUT with a wait site of that kernel (the other kernel
    runs normally), and the next call on the same context is correct.  The
    shape keeps each kernel to one wave of CTAs."""
    from tests.test_backward_gpu import check as check_bwd, run_gpu as bwd_gpu
    w = W.custom("bwd_skip", [300], [300], 4, 2, 32, 64)
    inp = W.make_inputs(w, with_dout=True)
    assert rpb.relattn_test_backward_skip_step(kernel, 0) == rpb.RELATTN_OK
    try:
        with pytest.raises(AssertionError, match="RELATTN_ERR_TIMEOUT"):
            bwd_gpu(w, inp)               # synchronises, then reads the status
        word = rpb.relattn_last_device_error_word()
    finally:
        rpb.relattn_test_backward_skip_step(kernel, -1)
    assert word & 2 and (word >> 8) in BWD_SITES[kernel], hex(word)
    check_bwd(w)                          # hook off: correct on the same context


def test_backward_skip_hook_rejects_bad_arguments():
    assert rpb.relattn_test_backward_skip_step(0, -2) != rpb.RELATTN_OK
    assert rpb.relattn_test_backward_skip_step(2, 0) != rpb.RELATTN_OK
    assert rpb.relattn_test_backward_skip_step(-1, 0) != rpb.RELATTN_OK
    assert rpb.relattn_test_backward_skip_step(0, -1) == rpb.RELATTN_OK
    assert rpb.relattn_test_backward_skip_step(1, -1) == rpb.RELATTN_OK
