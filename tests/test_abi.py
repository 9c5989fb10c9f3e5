"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every symbol the header declares, and rejects bad arguments before
touching the device."""
import os
import re

import pytest
import torch

import relative_position_biased_gb300 as rpb
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    rpb.build()
    return rpb.load_library()


_DECL = re.compile(r"^\s*(?:const\s+)?\w+\s*\*?\s*(relattn_\w+)\s*\(", re.M)


def _header_sections():
    """(product declarations, test-build declarations) of include/relattn.h:
    the test hooks are the ones inside #ifdef RELATTN_TEST_HOOKS."""
    text = open(os.path.join(ROOT, "include", "relattn.h")).read()
    m = re.search(r"#ifdef RELATTN_TEST_HOOKS(.*?)#endif", text, re.S)
    test = set(_DECL.findall(m.group(1))) if m else set()
    prod = set(_DECL.findall(text)) - test
    return sorted(prod), sorted(test)


def _declared_functions():
    return _header_sections()[0]


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("relattn_prefill", "relattn_decode", "relattn_combine"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    prod, test = _header_sections()
    for name in prod:
        assert hasattr(lib, name), name
    assert set(prod) == set(rpb.EXPORTED)
    assert set(test) == set(rpb.TEST_HOOKS) and test


def test_test_hooks_live_in_the_test_build_only(lib):
    """The product library exports no relattn_test_* entry point; the test
    build exports every product entry point plus the hooks."""
    prod, test = _header_sections()
    for name in test:
        assert not hasattr(lib, name), name
    tlib = rpb.load_test_library()
    for name in prod + test:
        assert hasattr(tlib, name), name


def test_struct_layout_matches_header(lib):
    # 7 pointers, 11 int32, 2 floats, then out/lse/workspace, size_t, int32
    off = {f[0]: getattr(rpb.RelattnParams, f[0]).offset for f in rpb.RelattnParams._fields_}
    assert off["batch"] == 56 and off["alpha"] == 100 and off["out"] == 112
    assert off["workspace_bytes"] == 136 and off["num_splits"] == 144


def test_status_strings(lib):
    for code, name in rpb.STATUS_NAMES.items():
        assert rpb.relattn_status_string(code) == name
    assert "sm_103a" in rpb.relattn_version()


def _params(**over):
    base = dict(q=256, k=256, v=256, r=256, P=256, cu_seqlens_q=256, cu_seqlens_k=256, batch=1,
                total_q=8, total_k=8, max_seqlen_q=8, max_seqlen_k=8, num_heads_q=4,
                num_heads_kv=2, head_dim=128, r_dim=32, rel_extent=64, window=0,
                alpha=0.088, log_scale_base=0.0, out=256, lse=256, workspace=None,
                workspace_bytes=0, num_splits=0)
    base.update(over)
    return rpb.RelattnParams(**base)


@pytest.mark.parametrize("over,expect", [
    (dict(head_dim=64), 2),
    (dict(num_heads_q=3), 1),
    (dict(num_heads_kv=0), 1),
    (dict(r_dim=65), 2),
    (dict(r_dim=-1), 1),
    (dict(rel_extent=-1), 1),
    (dict(log_scale_base=0.5), 1),
    (dict(log_scale_base=1.0), 1),
    (dict(alpha=float("nan")), 1),
    (dict(q=None), 1),
    (dict(lse=None), 1),
    (dict(cu_seqlens_k=None), 1),
    (dict(P=None), 1),
    (dict(q=264), 1),            # not 16-byte aligned
    (dict(out=258), 1),
    (dict(max_seqlen_k=4), 1),   # below max_seqlen_q
    (dict(batch=-1), 1),
])
def test_prefill_rejects_bad_arguments(lib, over, expect):
    assert rpb.relattn_prefill(_params(**over)) == expect


def test_decode_rejects_too_many_rows(lib):
    assert rpb.relattn_decode(_params(max_seqlen_q=17, max_seqlen_k=100)) == 2


def test_empty_batch_is_a_no_op(lib):
    assert rpb.relattn_prefill(_params(batch=0, total_q=0)) == 0
    assert rpb.relattn_decode(_params(total_q=0)) == 0


def test_combine_rejects_bad_arguments(lib):
    assert rpb.relattn_combine(0, 0, 0, 1, 1, 0, 0) == 1
    assert rpb.relattn_combine(256, 256, 2, 4, 0, 256, 256) == 1
    assert rpb.relattn_combine(264, 256, 2, 4, 2, 256, 256) == 1


@pytest.mark.parametrize("kv_over,expect", [
    (dict(page_size=64), 2),                  # not a multiple of 128
    (dict(page_size=0), 2),
    (dict(num_pages=0), 1),
    (dict(max_pages_per_seq=0), 1),
    (dict(block_table=None), 1),
    (dict(block_table=(7 << 22) + 2), 1),     # not 4-byte aligned
    (dict(max_pages_per_seq=1, page_size=128), 1),   # 1 x 128 < max_seqlen_k 200
])
def test_decode_paged_rejects_bad_arguments(lib, kv_over, expect):
    kv = dict(block_table=7 << 22, max_pages_per_seq=2, page_size=128, num_pages=4)
    kv.update(kv_over)
    prm = _params(total_q=1, max_seqlen_q=1, max_seqlen_k=200, total_k=200)
    assert rpb.relattn_decode_paged(prm, rpb.RelattnPagedKV(**kv)) == expect


def _bwd_params(fwd=None, **over):
    base = dict(dout=1 << 22, dq=2 << 22, dk=3 << 22, dv=4 << 22, dr=5 << 22,
                workspace=6 << 22, workspace_bytes=1 << 24)
    base.update(over)
    return rpb.RelattnBwdParams(fwd=fwd if fwd is not None else _params(), **base)


def test_backward_struct_layout_matches_header(lib):
    off = {f[0]: getattr(rpb.RelattnBwdParams, f[0]).offset for f in rpb.RelattnBwdParams._fields_}
    assert off["dout"] == rpb.ctypes.sizeof(rpb.RelattnParams) == 152
    assert off["workspace_bytes"] == 200 and rpb.ctypes.sizeof(rpb.RelattnBwdParams) == 208


def test_backward_workspace_size(lib):
    # D: 4 heads x 8 rows x 4 bytes rounded up to 256; R: 8 rows x 4 heads x 64
    # distances x 4 bytes; the partial dq: 8 rows x 4 heads x 128 x 4 bytes
    st, n = rpb.relattn_backward_workspace_size(_bwd_params())
    assert st == 0 and n == 256 + 8 * 4 * 64 * 4 + 8 * 4 * 128 * 4
    st, n = rpb.relattn_backward_workspace_size(_bwd_params(fwd=_params(total_q=1000)))
    assert st == 0 and n == 16128 + 1000 * 4 * 64 * 4 + 1000 * 4 * 128 * 4
    # E = 61 is padded to 64 per row; no bias: D alone
    st, n = rpb.relattn_backward_workspace_size(_bwd_params(fwd=_params(rel_extent=61)))
    assert st == 0 and n == 256 + 8 * 4 * 64 * 4 + 8 * 4 * 128 * 4
    st, n = rpb.relattn_backward_workspace_size(_bwd_params(fwd=_params(r_dim=0)))
    assert st == 0 and n == 256
    # a GQA group of 4: two fp32 halves of dk and dv, total_k x Hkv x 128 each
    st, n = rpb.relattn_backward_workspace_size(_bwd_params(fwd=_params(num_heads_q=8, num_heads_kv=2)))
    tk = _params().total_k
    assert st == 0 and n == 256 + 8 * 8 * 64 * 4 + 8 * 8 * 128 * 4 + 4 * tk * 2 * 128 * 4


@pytest.mark.parametrize("over,fwd_over,expect", [
    (dict(dq=None), {}, 1),
    (dict(dk=None), {}, 1),
    (dict(dout=(1 << 22) + 8), {}, 1),      # not 16-byte aligned
    (dict(dr=None), {}, 1),                 # r_dim 32 needs dr
    (dict(workspace=None), {}, 5),
    (dict(workspace_bytes=64), {}, 5),
    (dict(workspace_bytes=1000), {}, 5),    # D fits, R does not
    (dict(), dict(r_dim=12), 2),            # r_dim not a multiple of 8
    (dict(), dict(head_dim=64), 2),
    (dict(), dict(lse=256 + 4), 1),         # lse not 16-byte aligned
])
def test_backward_rejects_bad_arguments(lib, over, fwd_over, expect):
    assert rpb.relattn_backward(_bwd_params(fwd=_params(**fwd_over), **over)) == expect


def test_backward_empty_batch_is_a_no_op(lib):
    assert rpb.relattn_backward(_bwd_params(fwd=_params(batch=0, total_q=0), dq=None)) == 0


def _prologue_params(**over):
    # fake, well separated addresses: every check fails before the device is touched
    names = ("q", "k", "v", "conv_k", "conv_v", "norm_q", "norm_k", "cu_seqlens_q",
             "cu_seqlens_k", "q_out", "k_cache", "v_cache")
    base = {n: (i + 1) << 20 for i, n in enumerate(names)}
    base.update(eps=1e-6, batch=1, total_q=8, total_k=16, num_heads_q=4, num_heads_kv=2,
                head_dim=128)
    base.update(over)
    return rpb.RelattnPrologueParams(**base)


def test_prologue_struct_layout_matches_header(lib):
    off = {f[0]: getattr(rpb.RelattnPrologueParams, f[0]).offset
           for f in rpb.RelattnPrologueParams._fields_}
    # 7 pointers, a float, 2 pointers, 6 int32, then 7 pointers
    assert off["eps"] == 56 and off["cu_seqlens_q"] == 64 and off["batch"] == 80
    assert off["q_out"] == 104 and off["conv_state_out_v"] == 152
    assert rpb.ctypes.sizeof(rpb.RelattnPrologueParams) == 160


@pytest.mark.parametrize("over,expect", [
    (dict(head_dim=64), 2),
    (dict(num_heads_q=3), 1),
    (dict(num_heads_kv=0), 1),
    (dict(total_q=-1), 1),
    (dict(eps=0.0), 1),
    (dict(eps=float("inf")), 1),
    (dict(q=None), 1),
    (dict(k_cache=None), 1),
    (dict(norm_k=None), 1),
    (dict(cu_seqlens_k=None), 1),
    (dict(q=(1 << 20) + 8), 1),                    # not 16-byte aligned
    (dict(v_cache=(12 << 20) + 8), 1),
    (dict(conv_v=(5 << 20) + 8), 1),
    (dict(conv_state_out_k=(20 << 20) + 8), 1),
    (dict(q_out=(1 << 20) + 256), 1),              # q_out partly overlaps q
    (dict(k_cache=(2 << 20) + 512), 1),            # cache overlaps k
    (dict(conv_state_in_k=30 << 20, conv_state_out_v=(30 << 20) + 512), 1),
])
def test_prologue_rejects_bad_arguments(lib, over, expect):
    assert rpb.relattn_prologue(_prologue_params(**over)) == expect


def test_prologue_empty_batch_is_a_no_op(lib):
    assert rpb.relattn_prologue(_prologue_params(batch=0, q=None)) == 0


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        rpb._open(str(tmp_path / "librelattn.so"))


def test_workload_generator_is_deterministic():
    from relative_position_biased_gb300 import workloads as W
    w = W.custom("det", [10, 3], [10, 3], 2, 1, 4, 8, seed=3)
    a, b = W.make_inputs(w), W.make_inputs(w)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert a["q"].dtype == torch.bfloat16 and a["cu_seqlens_q"].tolist() == [0, 10, 13]
