"""The pieces chained as one attention layer on the GPU, each step through its
C-ABI entry:
1. the prologue (ShortConv of k / v, RMSNorm of q / k, cache write);
2. the prefill over the cache;
3. the backward from the saved out / lse.

The same chain runs through the oracles, and each stage's GPU output is
compared with the oracle fed by the GPU's previous stage. Each step is then
checked on exactly its own inputs, at the step's own tolerance.

A second case runs the chain as two chunks. The first chunk leaves the conv
state and the cache rows; the second continues from them, its attention
reading both chunks' cache rows. Its prologue outputs must equal a single
pass over the whole sequence bit for bit. Its prefill rows must equal the
single pass's last rows within the forward's tolerance, since the prefill
tiles rows from the chunk's start.
"""
import numpy as np
import pytest
import torch

from tests.conftest import gpu_available
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


def _layer_inputs(lens, Hq=8, Hkv=2, r_dim=32, E=96, seed=3):
    w = W.custom("layer", lens, lens, Hq, Hkv, r_dim, E, seed=seed)
    att = W.make_inputs(w, with_dout=True)        # r, P, dout (q / k / v come from the prologue)
    pro = W.make_prologue_inputs(w)
    return w, att, pro


def _prologue_gpu(pro, lens, k_lens=None, state=None, kc=None, vc=None, state_out=None):
    import relative_position_biased_gb300 as rpb
    k_lens = lens if k_lens is None else k_lens
    d = {k: v.cuda() for k, v in pro.items()}
    cu_k = W.cu_seqlens(k_lens).cuda()
    Hkv = d["k"].shape[1]
    if kc is None:
        kc = torch.zeros(sum(k_lens), Hkv, 128, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
    q = rpb.prologue(d["q"], d["k"], d["v"], d["conv_k"], d["conv_v"], d["norm_q"], d["norm_k"],
                     W.cu_seqlens(lens).cuda(), cu_k, kc, vc, conv_state_in=state,
                     conv_state_out=state_out)
    return q, kc, vc


def test_prologue_prefill_backward_chain():
    import oracle
    import relative_position_biased_gb300 as rpb
    from oracle import prologue as OP
    from tests.parity_util import OUT_TOL, LSE_TOL
    from tests.test_backward_gpu import assert_close

    lens = [300, 77]
    w, att, pro = _layer_inputs(lens)
    cu = W.cu_seqlens(lens)
    # 1. prologue
    q, kc, vc = _prologue_gpu(pro, lens)
    ref = OP.prologue(pro["q"], pro["k"], pro["v"], pro["conv_k"], pro["conv_v"], pro["norm_q"],
                      pro["norm_k"], cu, cu)
    for got, exp in ((q, ref["q_out"]), (kc, ref["k_rows"]), (vc, ref["v_rows"])):
        g = got.float().cpu().double().numpy()
        assert np.all(np.abs(g - exp) <= 2.0 ** -8 * np.abs(exp) + 1e-5)
    # 2. prefill over the GPU's prologue outputs
    r, P, dout = att["r"].cuda(), att["P"].cuda(), att["dout"].cuda()
    kw = dict(max_seqlen_q=max(lens), max_seqlen_k=max(lens), alpha=w.alpha)
    out, lse = rpb.prefill(q, kc, vc, r, P, cu.cuda(), cu.cuda(), **kw)
    ro, rl = oracle.forward(q.cpu(), kc.cpu(), vc.cpu(), att["r"], att["P"], cu, cu, alpha=w.alpha)
    assert np.abs(out.float().cpu().numpy() - ro).max() <= OUT_TOL
    assert np.abs(lse.cpu().numpy().T - rl).max() <= LSE_TOL
    # 3. backward from the saved out / lse
    grads = rpb.backward(q, kc, vc, r, P, out, lse, dout, cu.cuda(), cu.cuda(), **kw)
    torch.cuda.synchronize()
    assert rpb.relattn_get_device_error() == rpb.RELATTN_OK
    refs = oracle.backward(q.cpu(), kc.cpu(), vc.cpu(), att["r"], att["P"], att["dout"], cu, cu,
                           alpha=w.alpha)
    for name, g, rr in zip(("dq", "dk", "dv", "dr"), grads, refs):
        assert_close(g.float().cpu().double().numpy(), rr, name)


def test_two_chunks_equal_one_pass():
    """Chunk 1 (rows 0..c) then chunk 2 (rows c..L) of one sequence: the conv
    state and the cache carry over; the cache and q equal a single pass bit
    for bit, and chunk 2's prefill rows match the single pass's."""
    import relative_position_biased_gb300 as rpb
    L, c = 400, 150
    w, att, pro = _layer_inputs([L], Hq=4, Hkv=1)
    r, P = att["r"].cuda(), att["P"].cuda()
    # one pass
    q1, kc1, vc1 = _prologue_gpu(pro, [L])
    o1, l1 = rpb.prefill(q1, kc1, vc1, r, P, W.cu_seqlens([L]).cuda(), W.cu_seqlens([L]).cuda(),
                         max_seqlen_q=L, max_seqlen_k=L, alpha=w.alpha)
    # two chunks into one cache of L rows
    first = {k: (v[:c] if k in ("q", "k", "v") else v) for k, v in pro.items()}
    second = {k: (v[c:] if k in ("q", "k", "v") else v) for k, v in pro.items()}
    st = tuple(torch.empty(1, 3, 128, dtype=torch.bfloat16, device="cuda") for _ in range(2))
    kc = torch.zeros(L, 1, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    qa, _, _ = _prologue_gpu(first, [c], [c], kc=kc[:c], vc=vc[:c], state_out=st)
    qb, _, _ = _prologue_gpu(second, [L - c], [L], state=(st[0].clone(), st[1].clone()), kc=kc, vc=vc)
    torch.cuda.synchronize()
    assert torch.equal(kc, kc1) and torch.equal(vc, vc1)
    assert torch.equal(torch.cat([qa, qb]), q1)
    o2, l2 = rpb.prefill(qb, kc, vc, r[c:], P, W.cu_seqlens([L - c]).cuda(),
                         W.cu_seqlens([L]).cuda(), max_seqlen_q=L - c, max_seqlen_k=L, alpha=w.alpha)
    torch.cuda.synchronize()
    # the chunk's rows against the single pass: same inputs, but the prefill
    # tiles the rows differently (its 128-row tiles start at the chunk), so
    # compare to the oracle's tolerance rather than bit for bit
    assert (o2.float() - o1[c:].float()).abs().max().item() <= 2e-2
    assert (l2 - l1[:, c:]).abs().max().item() <= 1e-3
