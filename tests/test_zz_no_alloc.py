"""relattn_decode_noalloc: the decode variant for callers that cannot allocate
device memory where they run attention (engines whose pools already own all
free memory, plugin hosts without a workspace hook, paths that cannot take
cudaMalloc's implicit synchronisation).  Its split partials live in a fixed
scratch array inside the library.  This file is collected last on purpose, so
that a failure here comes after every other test has run.
"""
import numpy as np
import pytest
import torch

from tests.conftest import gpu_available
from relative_position_biased_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]

OUT_TOL, LSE_TOL = 2e-2, 1e-3


@pytest.fixture(scope="module")
def rpb():
    import relative_position_biased_gb300 as m
    m.build()
    m.load_library()
    return m


def _case(seed, window=0):
    w = W.custom(f"noalloc{seed}", [9, 1, 4], [3000, 700, 1500], 16, 2, 64, 512,
                 window=window, log_scale_base=64.0 if window <= 0 else 0.0, seed=seed)
    inp = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    return w, inp


def _params(rpb, w, inp, out, lse, num_splits):
    return rpb.make_params(inp["q"], inp["k"], inp["v"], inp["r"], inp["P"],
                           inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                           max_seqlen_q=max(w.q_lens), max_seqlen_k=max(w.k_lens),
                           alpha=w.alpha, window=w.window, log_scale_base=w.log_scale_base,
                           out=out, lse=lse, num_splits=num_splits)


def test_noalloc_decode_matches_workspace_decode_twice(rpb):
    """Two calls in a row (different inputs) through the C ABI: each equals the
    workspace-taking relattn_decode on the same inputs."""
    stream = torch.cuda.current_stream().cuda_stream
    for seed, window, splits in [(11, 0, 0), (12, 600, 5)]:
        w, inp = _case(seed, window)
        ref_out, ref_lse = rpb.decode(inp["q"], inp["k"], inp["v"], inp["r"], inp["P"],
                                      inp["cu_seqlens_q"], inp["cu_seqlens_k"],
                                      max_seqlen_q=max(w.q_lens), max_seqlen_k=max(w.k_lens),
                                      alpha=w.alpha, window=w.window,
                                      log_scale_base=w.log_scale_base, num_splits=splits)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        prm = _params(rpb, w, inp, out, lse, splits)
        st, n_splits = rpb.relattn_decode_num_splits(prm)
        assert st == 0 and n_splits > 1, "the case must exercise the scratch (split partials)"
        assert rpb.relattn_decode_noalloc(prm, stream) == 0
        torch.cuda.synchronize()
        assert rpb.relattn_get_device_error() == 0
        d_out = (out.float() - ref_out.float()).abs().max().item()
        d_lse = (lse - ref_lse).abs().max().item()
        assert np.isfinite(d_out) and d_out <= OUT_TOL, d_out
        assert np.isfinite(d_lse) and d_lse <= LSE_TOL, d_lse


def test_noalloc_rejects_partials_beyond_the_scratch(rpb):
    """Split partials larger than the fixed scratch: a clear error, no launch.
    64 sequences x 16 query rows x 16 heads make one split's partials 8.5 MB,
    so four splits exceed the 32 MiB scratch."""
    w = W.custom("noalloc_big", [16] * 64, [640] * 64, 16, 2, 64, 512, seed=14)
    inp = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    out = torch.zeros_like(inp["q"])
    lse = torch.zeros(inp["q"].shape[1], inp["q"].shape[0], device="cuda")
    prm = _params(rpb, w, inp, out, lse, 5)
    st, n_splits = rpb.relattn_decode_num_splits(prm)
    assert st == 0 and n_splits >= 4
    st, need = rpb.relattn_decode_workspace_size(prm)
    assert st == 0 and need > rpb.NOALLOC_SCRATCH_BYTES
    assert rpb.relattn_decode_noalloc(prm, 0) == 5   # RELATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
