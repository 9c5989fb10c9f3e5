"""The standalone LSE combine (relattn_combine) on the GPU against an fp64
merge written here from its definition.

A split s of a row's keys leaves a partial (o_s, lse_s): the softmax-weighted
mean of its values and the logsumexp of its logits.  Softmax over the union
of disjoint key sets is then
    lse = ln sum_s exp(lse_s),    out = sum_s exp(lse_s - lse) * o_s,
with empty splits (lse_s = -inf) contributing nothing (page "vLLM Day-0
support for TML Inkling", paragraph on FA4 with sheared bias: split-KV with
num_splits).  A row with no non-empty split has lse = -inf and out = 0.

The cases cover every row layout of the kernel (1, 2, 4 and 8 warps per row,
chosen by the split count), a row count that leaves the last CTA partly
empty, NaN in the o_s of empty splits, and all-empty rows.

Tolerance: out is rounded once to bf16 (relative 2^-9 of |out|) after an
fp32 weighted sum of at most a few hundred terms; lse is fp32.  The test
allows |out - ref| <= 2^-8 max(1, |ref|) and |lse - ref| <= 1e-5 max(1, |ref|).
"""
import numpy as np
import pytest
import torch

from tests.conftest import gpu_available

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import relative_position_biased_gb300 as rpb
    rpb.build()
    rpb.load_library()


def merge_fp64(o_part, lse_part):
    """o_part [S, rows, 128], lse_part [S, rows] (fp64) -> (out [rows, 128], lse [rows])."""
    S, rows = lse_part.shape
    out = np.zeros((rows, o_part.shape[2]))
    lse = np.full(rows, -np.inf)
    for n in range(rows):
        live = [s for s in range(S) if np.isfinite(lse_part[s, n])]
        if not live:
            continue
        m = max(lse_part[s, n] for s in live)
        z = sum(np.exp(lse_part[s, n] - m) for s in live)
        lse[n] = m + np.log(z)
        for s in live:
            out[n] += np.exp(lse_part[s, n] - lse[n]) * o_part[s, n]
    return out, lse


def draw(S, total_q, Hq, seed, empty_frac=0.2, empty_rows=()):
    g = torch.Generator().manual_seed(seed)
    rows = total_q * Hq
    o = torch.randn(S, rows, 128, generator=g, dtype=torch.float32)
    lse = 3.0 * torch.randn(S, rows, generator=g, dtype=torch.float32)
    empty = torch.rand(S, rows, generator=g) < empty_frac
    for n in empty_rows:
        empty[:, n] = True
    lse[empty] = -float("inf")
    o[empty] = float("nan")        # whatever an empty split's o_s holds is ignored
    return o, lse


@pytest.mark.parametrize("S", [1, 3, 4, 15, 16, 63, 64, 200])
def test_combine_matches_fp64_merge(S):
    import relative_position_biased_gb300 as rpb
    total_q, Hq = 7, 3                 # 21 rows: the last CTA is partly empty
    o, lse = draw(S, total_q, Hq, seed=100 + S, empty_rows=(5,) if S > 1 else ())
    out = torch.empty(total_q, Hq, 128, dtype=torch.bfloat16, device="cuda")
    lse_out = torch.empty(Hq, total_q, dtype=torch.float32, device="cuda")
    o_d, lse_d = o.cuda(), lse.cuda()
    st = rpb.relattn_combine(o_d.data_ptr(), lse_d.data_ptr(), S, total_q, Hq, out.data_ptr(),
                             lse_out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == rpb.RELATTN_OK
    torch.cuda.synchronize()
    ref_out, ref_lse = merge_fp64(o.double().numpy(), lse.double().numpy())
    got_out = out.float().cpu().double().numpy().reshape(total_q * Hq, 128)
    # lse is [Hq, total_q]; row n = t * Hq + h
    got_lse = lse_out.cpu().double().numpy().T.reshape(-1)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), fin)
    assert np.all(got_lse[~fin] == -np.inf)
    assert np.all(got_out[~fin] == 0.0)
    assert np.all(np.abs(got_lse[fin] - ref_lse[fin]) <= 1e-5 * np.maximum(1.0, np.abs(ref_lse[fin])))
    assert np.isfinite(got_out).all()
    assert np.all(np.abs(got_out - ref_out) <= 2.0 ** -8 * np.maximum(1.0, np.abs(ref_out)))


def test_combine_of_one_split_is_the_partial():
    """With a single split the merge is the identity (up to the bf16 cast)."""
    import relative_position_biased_gb300 as rpb
    o, lse = draw(1, 5, 4, seed=7, empty_frac=0.0)
    out = torch.empty(5, 4, 128, dtype=torch.bfloat16, device="cuda")
    lse_out = torch.empty(4, 5, dtype=torch.float32, device="cuda")
    o_d, lse_d = o.cuda(), lse.cuda()
    assert rpb.relattn_combine(o_d.data_ptr(), lse_d.data_ptr(), 1, 5, 4, out.data_ptr(),
                               lse_out.data_ptr(), 0) == rpb.RELATTN_OK
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), o[0].reshape(5, 4, 128).to(torch.bfloat16))
    assert torch.allclose(lse_out.cpu().T.reshape(-1), lse[0], rtol=0, atol=1e-6)
