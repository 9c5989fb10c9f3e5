"""MXFP8 K / V on the GPU (page "SGLang and Miles Add Day-0 Support for
Inkling", section "Relative Logits Optimization", paragraph "MXFP8 Support"):

- relattn_quantize_mxfp8 gives the oracle's codes and scales bit for bit
  (byte outputs), on blocks spanning the exponent range, all-zero blocks,
  values that round to (signed) zero and values past the saturation point;
- relattn_decode_mxfp8 on codes made by the oracle matches the oracle's MXFP8
  decode (q rounded through MXFP8, K and V dequantised, fp64 forward) within
  the forward's tolerance, over GQA widths, several tokens per item, windows,
  log-scale, no bias, forced split counts, and the full batched decode
  workload (64 sequences, KV lengths 1K-32K, with and without a window) on
  sampled sequences;
- shapes the kernel does not take are refused with RELATTN_ERR_UNSUPPORTED.
"""
import numpy as np
import pytest
import torch

from tests.conftest import gpu_available
from tests.parity_util import LSE_TOL, OUT_TOL
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


def _np_f(t):
    return t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()


def test_quantize_bit_exact():
    import relative_position_biased_gb300 as rpb
    from oracle import mxfp8 as M
    gen = torch.Generator().manual_seed(11)
    x = torch.randn(2048, 128, generator=gen)
    x *= torch.exp2(torch.randint(-40, 40, (2048, 1), generator=gen).float())
    x[0] = 0.0                                         # all-zero blocks
    x[1, :32] = 1.9                                    # saturates (486.4 units of 2^-8)
    x[1, 32:64] = torch.linspace(-448, 448, 32) * 2.0 ** -5
    x[2, :] = -1e-30                                   # tiny: e clamps, codes round to -0
    x[2, 0] = 1.0
    x[3, :] = torch.tensor([272.0, 304.0, -272.0, 1.0] * 32) * 2.0 ** -8   # ties at amax 2^0
    x[3, 3::4] = 1.0
    xb = x.to(torch.bfloat16)
    codes, scales = rpb.quantize_mxfp8(xb.cuda())
    torch.cuda.synchronize()
    c_o, s_o = M.quantize(xb.float().numpy())
    c_g, s_g = codes.cpu().numpy(), scales.cpu().numpy()
    assert np.array_equal(s_g, s_o), np.argwhere(s_g != s_o)[:5]
    assert np.array_equal(c_g, c_o), np.argwhere(c_g != c_o)[:5]


def test_quantize_kv_shape_and_refusals():
    import relative_position_biased_gb300 as rpb
    from oracle import mxfp8 as M
    k = torch.randn(300, 2, 128, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    codes, scales = rpb.quantize_mxfp8(k.cuda())
    assert tuple(scales.shape) == (300, 2, 4)
    c_o, s_o = M.quantize(k.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), c_o) and np.array_equal(scales.cpu().numpy(), s_o)
    # misaligned input is refused before any launch
    buf = torch.zeros(64 * 32 + 8, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(64 * 32, dtype=torch.uint8, device="cuda")
    sc = torch.empty(64, dtype=torch.uint8, device="cuda")
    st = rpb.relattn_quantize_mxfp8(buf.data_ptr() + 2, 64, out.data_ptr(), sc.data_ptr(), 0)
    assert st == rpb.RELATTN_ERR_INVALID_ARG


def _mx_case(w):
    """Seeded bf16 inputs of w with K / V quantised by the oracle."""
    from oracle import mxfp8 as M
    inp = W.make_inputs(w)
    k8, ks = M.quantize(_np_f(inp["k"]))
    v8, vs = M.quantize(_np_f(inp["v"]))
    return inp, (k8, ks, v8, vs)


def _run_mx(w, inp, kv, num_splits=0):
    import relative_position_biased_gb300 as rpb
    d = {k: v.cuda() for k, v in inp.items()}
    k8, ks, v8, vs = (a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a)).cuda()
                      for a in kv)
    out, lse = rpb.decode_mxfp8(d["q"], k8, v8, ks, vs, d["r"], d["P"], d["cu_seqlens_q"],
                                d["cu_seqlens_k"], max_seqlen_q=max(w.q_lens), max_seqlen_k=max(w.k_lens),
                                alpha=w.alpha, window=w.window, log_scale_base=w.log_scale_base,
                                num_splits=num_splits)
    torch.cuda.synchronize()
    st = rpb.relattn_get_device_error()
    assert st == rpb.RELATTN_OK, rpb.STATUS_NAMES.get(st, st)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _compare(w, inp, kv, gpu, seqs=None):
    """Oracle MXFP8 decode of the whole workload, or of the sequences `seqs`
    one at a time (each with only its own keys), against the GPU rows."""
    from oracle import mxfp8 as M
    out_g, lse_g = gpu
    cq = inp["cu_seqlens_q"].numpy()
    ck = inp["cu_seqlens_k"].numpy()
    k8, ks, v8, vs = kv
    kw = dict(alpha=w.alpha, window=w.window, log_scale_base=w.log_scale_base)
    worst = (0.0, 0.0)
    for b in (range(len(w.q_lens)) if seqs is None else seqs):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        o, l = M.decode_reference(inp["q"][q0:q1], k8[k0:k1], ks[k0:k1], v8[k0:k1], vs[k0:k1],
                                  inp["r"][q0:q1], inp["P"], np.array([0, q1 - q0], np.int32),
                                  np.array([0, k1 - k0], np.int32), **kw)
        d_out = float(np.max(np.abs(out_g[q0:q1] - o))) if o.size else 0.0
        d_lse = float(np.max(np.abs(lse_g[:, q0:q1].T - l))) if l.size else 0.0
        assert np.all(np.isfinite(out_g[q0:q1])), (w.name, b)
        assert d_out <= OUT_TOL, f"{w.name} seq {b}: max |dout| = {d_out:.3e}"
        assert d_lse <= LSE_TOL, f"{w.name} seq {b}: max |dlse| = {d_lse:.3e}"
        worst = (max(worst[0], d_out), max(worst[1], d_lse))
    return worst


CASES = [
    # name, q_lens, k_lens, Hq, Hkv, r_dim, E, extra
    ("b6_gqa8", [1] * 6, [1, 130, 1000, 2500, 4097, 300], 16, 2, 64, 1024, {}),
    ("b4_gqa16", [1] * 4, [129, 2000, 777, 3000], 16, 1, 64, 1024, {}),
    ("b3_tok2_gqa8", [2] * 3, [2, 1500, 2049], 16, 2, 32, 256, {}),
    ("b5_window", [1] * 5, [64, 900, 1800, 2600, 3333], 16, 2, 64, 1024, {"window": 700}),
    ("b4_logscale", [1] * 4, [500, 1500, 2500, 3500], 8, 1, 16, 512, {"log_scale_base": 1024.0}),
    ("b4_nobias", [1] * 4, [300, 1200, 2200, 128], 16, 2, 0, 0, {}),
    ("b2_odd_rdim_E", [1] * 2, [700, 1900], 16, 2, 20, 300, {}),
]


@pytest.mark.parametrize("name,q_lens,k_lens,Hq,Hkv,rd,E,extra", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("num_splits", [0, 1, 5])
def test_decode_mxfp8_parity(name, q_lens, k_lens, Hq, Hkv, rd, E, extra, num_splits):
    w = W.custom(name, q_lens, k_lens, Hq, Hkv, rd, E, **extra)
    inp, kv = _mx_case(w)
    _compare(w, inp, kv, _run_mx(w, inp, kv, num_splits))


@pytest.mark.parametrize("window", [0, 4096])
def test_decode_mxfp8_full_batched(window):
    """64 sequences, KV 1K-32K (the batched decode workload), checked on 8
    sequences: the shortest, the longest and six seeded ones.  Their K / V
    codes are the oracle's; the other sequences' codes (not checked) come from
    relattn_quantize_mxfp8 (bit-exact with the oracle, tested above)."""
    import relative_position_biased_gb300 as rpb
    from oracle import mxfp8 as M
    w = W.decode_batched(window=window)
    inp = W.make_inputs(w)
    lens = np.array(w.k_lens)
    seqs = sorted({int(lens.argmin()), int(lens.argmax())} |
                  set(int(x) for x in np.random.default_rng(3).choice(len(lens), 6, replace=False)))
    k8, ks = rpb.quantize_mxfp8(inp["k"].cuda())
    v8, vs = rpb.quantize_mxfp8(inp["v"].cuda())
    ck = inp["cu_seqlens_k"].numpy()
    kv_o = [np.zeros(tuple(k8.shape), np.uint8), np.zeros(tuple(ks.shape), np.uint8),
            np.zeros(tuple(v8.shape), np.uint8), np.zeros(tuple(vs.shape), np.uint8)]
    for b in seqs:
        k0, k1 = ck[b], ck[b + 1]
        kc, kss = M.quantize(_np_f(inp["k"][k0:k1]))
        vc, vss = M.quantize(_np_f(inp["v"][k0:k1]))
        for dst_g, dst_o, src in ((k8, kv_o[0], kc), (ks, kv_o[1], kss), (v8, kv_o[2], vc), (vs, kv_o[3], vss)):
            dst_o[k0:k1] = src
            dst_g[k0:k1] = torch.from_numpy(src).cuda()
    gpu = _run_mx(w, inp, (k8, ks, v8, vs))
    _compare(w, inp, kv_o, gpu, seqs)


def test_decode_mxfp8_refuses_wide_items():
    import relative_position_biased_gb300 as rpb
    w = W.custom("mtp_wide", [9], [4000], 16, 2, 64, 1024)    # 9 tokens x 8 heads = 72 rows
    inp, kv = _mx_case(w)
    with pytest.raises(rpb.RelattnError) as e:
        _run_mx(w, inp, kv)
    assert e.value.status == rpb.RELATTN_ERR_UNSUPPORTED
