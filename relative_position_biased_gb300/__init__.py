"""GB300 relative-attention forward (Inkling-style relative position bias).

A thin ctypes binding over ``librelattn.so`` (C ABI in ``include/relattn.h``).
Functions named ``relattn_*`` mirror the C entry points one to one and only
marshal arguments; ``prefill`` / ``decode`` are conveniences that also allocate
``out`` / ``lse`` / workspace with torch (device memory is torch's job) before
calling the same entry points.  Every step of the computation runs in the CUDA
kernels; if the library is missing these functions raise -- there is no
fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional, Tuple

from . import workloads  # noqa: F401  (seeded input generators)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librelattn.so")
# the same kernels with the relattn_test_* hooks (built beside the product library)
TEST_LIB_PATH = os.path.join(_HERE, "librelattn_test.so")

RELATTN_OK = 0
RELATTN_ERR_INVALID_ARG = 1
RELATTN_ERR_UNSUPPORTED = 2
RELATTN_ERR_TIMEOUT = 4
STATUS_NAMES = {
    0: "RELATTN_OK", 1: "RELATTN_ERR_INVALID_ARG", 2: "RELATTN_ERR_UNSUPPORTED",
    3: "RELATTN_ERR_CUDA", 4: "RELATTN_ERR_TIMEOUT", 5: "RELATTN_ERR_WORKSPACE",
    6: "RELATTN_ERR_DEVICE_ARGS",
}
EXPORTED = (
    "relattn_prefill", "relattn_decode", "relattn_decode_workspace_size",
    "relattn_decode_num_splits", "relattn_combine", "relattn_get_device_error",
    "relattn_status_string", "relattn_version", "relattn_decode_noalloc",
    "relattn_last_device_error_word",
    "relattn_prologue", "relattn_backward", "relattn_backward_workspace_size",
    "relattn_decode_paged", "relattn_decode_mxfp8", "relattn_quantize_mxfp8",
    "relattn_prologue_mxfp8",
)
# exported by the test build only
TEST_HOOKS = (
    "relattn_test_skip_k_tile", "relattn_test_band_ctas", "relattn_test_prologue_skip_tile",
    "relattn_test_backward_skip_step",
)
NOALLOC_SCRATCH_BYTES = 32 << 20   # RELATTN_NOALLOC_SCRATCH_BYTES


class RelattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class RelattnParams(ctypes.Structure):
    """Mirror of ``relattn_params`` (field order and types must match the header)."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("r", ctypes.c_void_p), ("P", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("batch", ctypes.c_int32), ("total_q", ctypes.c_int32), ("total_k", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32), ("max_seqlen_k", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("r_dim", ctypes.c_int32), ("rel_extent", ctypes.c_int32),
        ("window", ctypes.c_int32), ("alpha", ctypes.c_float), ("log_scale_base", ctypes.c_float),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("num_splits", ctypes.c_int32),
    ]


class RelattnPagedKV(ctypes.Structure):
    """Mirror of ``relattn_paged_kv``."""
    _fields_ = [("block_table", ctypes.c_void_p), ("max_pages_per_seq", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


class RelattnKvMxfp8(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


class RelattnBwdParams(ctypes.Structure):
    """Mirror of ``relattn_bwd_params`` (field order and types must match the header)."""
    _fields_ = [
        ("fwd", RelattnParams), ("dout", ctypes.c_void_p), ("dq", ctypes.c_void_p),
        ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p), ("dr", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class RelattnPrologueParams(ctypes.Structure):
    """Mirror of ``relattn_prologue_params`` (field order and types must match the header)."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("conv_k", ctypes.c_void_p), ("conv_v", ctypes.c_void_p),
        ("norm_q", ctypes.c_void_p), ("norm_k", ctypes.c_void_p), ("eps", ctypes.c_float),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("batch", ctypes.c_int32), ("total_q", ctypes.c_int32), ("total_k", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("q_out", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("conv_state_in_k", ctypes.c_void_p), ("conv_state_in_v", ctypes.c_void_p),
        ("conv_state_out_k", ctypes.c_void_p), ("conv_state_out_v", ctypes.c_void_p),
    ]


_lock = threading.RLock()
_lib = None
_libs = {}    # path -> configured handle


def build(force: bool = False) -> str:
    from .buildlib import build as _build
    return _build(force=force)


def _open(path: str):
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with relative_position_biased_gb300.build()")
    return ctypes.CDLL(path)


def load_library(path: Optional[str] = None):
    """Load ``librelattn.so`` (raises if it has not been built).  Inside
    ``test_library()`` this is the test build instead."""
    global _lib
    with _lock:
        if path is not None:
            return _configure(path)
        if _lib is None:
            _lib = _configure(LIB_PATH)
        return _lib


def load_test_library():
    """Load ``librelattn_test.so``: the same kernels plus the relattn_test_* hooks."""
    with _lock:
        lib = _configure(TEST_LIB_PATH)
        for name in TEST_HOOKS:
            getattr(lib, name).restype = ctypes.c_int
        lib.relattn_test_skip_k_tile.argtypes = [ctypes.c_int32]
        lib.relattn_test_prologue_skip_tile.argtypes = [ctypes.c_int32]
        lib.relattn_test_backward_skip_step.argtypes = [ctypes.c_int32, ctypes.c_int32]
        lib.relattn_test_band_ctas.argtypes = [ctypes.c_int32]
        return lib


@contextlib.contextmanager
def test_library():
    """Route every call of this module to the test build for the duration of
    the block (tests that set a hook run their calls inside one).  The device
    error word and the hooks belong to the test build's own copy."""
    global _lib
    with _lock:
        prev = load_library()
        _lib = load_test_library()
    try:
        yield _lib
    finally:
        with _lock:
            _lib = prev


def _configure(path: str):
    with _lock:
        if path in _libs:
            return _libs[path]
        lib = _open(path)
        P, vp = ctypes.POINTER(RelattnParams), ctypes.c_void_p
        for name in ("relattn_prefill", "relattn_decode", "relattn_decode_noalloc"):
            f = getattr(lib, name)
            f.argtypes, f.restype = [P, vp], ctypes.c_int
        lib.relattn_decode_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        lib.relattn_decode_workspace_size.restype = ctypes.c_int
        lib.relattn_decode_num_splits.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
        lib.relattn_decode_num_splits.restype = ctypes.c_int
        lib.relattn_combine.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        vp, vp, vp]
        lib.relattn_combine.restype = ctypes.c_int
        lib.relattn_get_device_error.argtypes = [vp]
        lib.relattn_get_device_error.restype = ctypes.c_int
        lib.relattn_status_string.argtypes = [ctypes.c_int]
        lib.relattn_status_string.restype = ctypes.c_char_p
        lib.relattn_last_device_error_word.argtypes = []
        lib.relattn_last_device_error_word.restype = ctypes.c_int32
        lib.relattn_decode_paged.argtypes = [P, ctypes.POINTER(RelattnPagedKV), vp]
        lib.relattn_decode_paged.restype = ctypes.c_int
        lib.relattn_decode_mxfp8.argtypes = [P, ctypes.POINTER(RelattnKvMxfp8), vp]
        lib.relattn_decode_mxfp8.restype = ctypes.c_int
        lib.relattn_quantize_mxfp8.argtypes = [vp, ctypes.c_int64, vp, vp, vp]
        lib.relattn_quantize_mxfp8.restype = ctypes.c_int
        BP = ctypes.POINTER(RelattnBwdParams)
        lib.relattn_backward.argtypes = [BP, vp]
        lib.relattn_backward.restype = ctypes.c_int
        lib.relattn_backward_workspace_size.argtypes = [BP, ctypes.POINTER(ctypes.c_size_t)]
        lib.relattn_backward_workspace_size.restype = ctypes.c_int
        lib.relattn_prologue.argtypes = [ctypes.POINTER(RelattnPrologueParams), vp]
        lib.relattn_prologue.restype = ctypes.c_int
        lib.relattn_prologue_mxfp8.argtypes = [ctypes.POINTER(RelattnPrologueParams),
                                               ctypes.POINTER(RelattnKvMxfp8), vp]
        lib.relattn_prologue_mxfp8.restype = ctypes.c_int
        lib.relattn_version.argtypes = []
        lib.relattn_version.restype = ctypes.c_char_p
        _libs[path] = lib
        return lib


def _check(status: int, where: str) -> None:
    if status != RELATTN_OK:
        raise RelattnError(status, where)


# ------------------------------------------------------------------ C mirrors

def relattn_prefill(params: RelattnParams, stream: int = 0) -> int:
    return load_library().relattn_prefill(ctypes.byref(params), ctypes.c_void_p(stream))


def relattn_decode(params: RelattnParams, stream: int = 0) -> int:
    return load_library().relattn_decode(ctypes.byref(params), ctypes.c_void_p(stream))


def relattn_decode_noalloc(params: RelattnParams, stream: int = 0) -> int:
    """Decode with the library's fixed scratch array; params.workspace is ignored."""
    return load_library().relattn_decode_noalloc(ctypes.byref(params), ctypes.c_void_p(stream))


def relattn_decode_workspace_size(params: RelattnParams) -> Tuple[int, int]:
    n = ctypes.c_size_t(0)
    st = load_library().relattn_decode_workspace_size(ctypes.byref(params), ctypes.byref(n))
    return st, int(n.value)


def relattn_decode_num_splits(params: RelattnParams) -> Tuple[int, int]:
    n = ctypes.c_int32(0)
    st = load_library().relattn_decode_num_splits(ctypes.byref(params), ctypes.byref(n))
    return st, int(n.value)


def relattn_combine(o_part: int, lse_part: int, num_splits: int, total_q: int, num_heads: int,
                    out: int, lse: int, stream: int = 0) -> int:
    return load_library().relattn_combine(o_part, lse_part, num_splits, total_q, num_heads,
                                          out, lse, ctypes.c_void_p(stream))


def relattn_get_device_error(stream: int = 0) -> int:
    return load_library().relattn_get_device_error(ctypes.c_void_p(stream))


def relattn_last_device_error_word() -> int:
    return int(load_library().relattn_last_device_error_word())


def relattn_test_skip_k_tile(tile: int) -> int:
    """Test build: later tensor-core launches never load key tile ``tile`` (-1: off)."""
    return int(load_test_library().relattn_test_skip_k_tile(int(tile)))


def relattn_test_prologue_skip_tile(tile: int) -> int:
    """Test build: the staged prologue never copies token tile ``tile`` (-1: off)."""
    return int(load_test_library().relattn_test_prologue_skip_tile(int(tile)))


def relattn_test_backward_skip_step(kernel: int, step: int) -> int:
    """Test build: the tcgen05 backward producer of ``kernel`` (0: dk / dv, 1:
    dq) never loads its step ``step`` (-1: off)."""
    return int(load_test_library().relattn_test_backward_skip_step(int(kernel), int(step)))


def relattn_test_band_ctas(n: int) -> int:
    """Test build: at most ``n`` CTAs for the persistent / walking launches (0: one per SM)."""
    return int(load_test_library().relattn_test_band_ctas(int(n)))


def relattn_status_string(status: int) -> str:
    return load_library().relattn_status_string(status).decode()


def relattn_decode_paged(params: RelattnParams, kv: RelattnPagedKV, stream: int = 0) -> int:
    return load_library().relattn_decode_paged(ctypes.byref(params), ctypes.byref(kv),
                                               ctypes.c_void_p(stream))


def relattn_backward(params: RelattnBwdParams, stream: int = 0) -> int:
    return load_library().relattn_backward(ctypes.byref(params), ctypes.c_void_p(stream))


def relattn_backward_workspace_size(params: RelattnBwdParams) -> Tuple[int, int]:
    n = ctypes.c_size_t(0)
    st = load_library().relattn_backward_workspace_size(ctypes.byref(params), ctypes.byref(n))
    return st, int(n.value)


def relattn_prologue(params: RelattnPrologueParams, stream: int = 0) -> int:
    return load_library().relattn_prologue(ctypes.byref(params), ctypes.c_void_p(stream))


def relattn_version() -> str:
    return load_library().relattn_version().decode()


# ------------------------------------------------------------------ torch conveniences

def make_params(q, k, v, r, P, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q: int,
                max_seqlen_k: int, alpha: float, window: int = 0, log_scale_base: float = 0.0,
                out=None, lse=None, workspace=None, num_splits: int = 0,
                total_q: Optional[int] = None, total_k: Optional[int] = None) -> RelattnParams:
    """Fill a RelattnParams from torch tensors (pointers and sizes only)."""
    def ptr(t):
        return None if t is None else t.data_ptr()
    r_dim = int(r.shape[-1]) if r is not None and r.dim() == 3 else 0
    E = int(P.shape[-1]) if P is not None and P.dim() == 2 else 0
    return RelattnParams(
        q=ptr(q), k=ptr(k), v=ptr(v), r=ptr(r), P=ptr(P),
        cu_seqlens_q=ptr(cu_seqlens_q), cu_seqlens_k=ptr(cu_seqlens_k),
        batch=int(cu_seqlens_q.numel()) - 1,
        total_q=int(q.shape[0]) if total_q is None else int(total_q),
        total_k=int(k.shape[0]) if total_k is None else int(total_k),
        max_seqlen_q=int(max_seqlen_q), max_seqlen_k=int(max_seqlen_k),
        num_heads_q=int(q.shape[1]), num_heads_kv=int(k.shape[1]), head_dim=int(q.shape[2]),
        r_dim=r_dim, rel_extent=E, window=int(window), alpha=float(alpha),
        log_scale_base=float(log_scale_base), out=ptr(out), lse=ptr(lse),
        workspace=ptr(workspace),
        workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
        num_splits=int(num_splits))


def _current_stream() -> int:
    import torch
    return torch.cuda.current_stream().cuda_stream


def _outputs(q, out, lse):
    import torch
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
    return out, lse


def prefill(q, k, v, r, P, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q: int, max_seqlen_k: int,
            alpha: float, window: int = 0, log_scale_base: float = 0.0, out=None, lse=None,
            stream: Optional[int] = None):
    """Relative-attention prefill on device tensors; returns (out, lse[Hq, Tq])."""
    out, lse = _outputs(q, out, lse)
    prm = make_params(q, k, v, r, P, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=max_seqlen_q,
                      max_seqlen_k=max_seqlen_k, alpha=alpha, window=window,
                      log_scale_base=log_scale_base, out=out, lse=lse)
    _check(relattn_prefill(prm, _current_stream() if stream is None else stream), "relattn_prefill")
    return out, lse


def decode_workspace(params: RelattnParams, device):
    import torch
    st, nbytes = relattn_decode_workspace_size(params)
    _check(st, "relattn_decode_workspace_size")
    if nbytes == 0:
        return None
    return torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=device)


def decode(q, k, v, r, P, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q: int, max_seqlen_k: int,
           alpha: float, window: int = 0, log_scale_base: float = 0.0, num_splits: int = 0,
           out=None, lse=None, workspace=None, stream: Optional[int] = None):
    """Split-KV decode (<= 16 query rows per sequence); returns (out, lse[Hq, Tq])."""
    out, lse = _outputs(q, out, lse)
    prm = make_params(q, k, v, r, P, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=max_seqlen_q,
                      max_seqlen_k=max_seqlen_k, alpha=alpha, window=window,
                      log_scale_base=log_scale_base, out=out, lse=lse, num_splits=num_splits)
    if workspace is None:
        workspace = decode_workspace(prm, q.device)
    if workspace is not None:
        prm.workspace = workspace.data_ptr()
        prm.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(relattn_decode(prm, _current_stream() if stream is None else stream), "relattn_decode")
    return out, lse


def prologue(q, k, v, conv_k, conv_v, norm_q, norm_k, cu_seqlens_q, cu_seqlens_k, k_cache,
             v_cache, *, eps: float = 1e-6, q_out=None, conv_state_in=None,
             conv_state_out=None, total_k: Optional[int] = None, mxfp8=None,
             stream: Optional[int] = None):
    """ShortConv + Q/K RMSNorm + KV-cache write for one chunk, on device tensors.

    ``conv_state_in`` / ``conv_state_out`` are ``(k_state, v_state)`` pairs of
    bf16 [batch, 3, Hkv*128] tensors, or None.  Writes ``k_cache`` / ``v_cache``
    rows in place and returns ``q_out`` (a new tensor unless given; pass
    ``q_out=q`` to normalise in place).  With ``mxfp8=(k8, v8, k_scale,
    v_scale)`` (uint8 [total_k, Hkv, 128] codes and [total_k, Hkv, 4] scales)
    the cache rows are also written as MXFP8 (relattn_prologue_mxfp8); the bf16
    caches may then be None.
    """
    import torch
    if q_out is None:
        q_out = torch.empty_like(q)

    def ptr(t):
        return None if t is None else t.data_ptr()
    sin = conv_state_in if conv_state_in is not None else (None, None)
    sout = conv_state_out if conv_state_out is not None else (None, None)
    prm = RelattnPrologueParams(
        q=ptr(q), k=ptr(k), v=ptr(v), conv_k=ptr(conv_k), conv_v=ptr(conv_v),
        norm_q=ptr(norm_q), norm_k=ptr(norm_k), eps=float(eps),
        cu_seqlens_q=ptr(cu_seqlens_q), cu_seqlens_k=ptr(cu_seqlens_k),
        batch=int(cu_seqlens_q.numel()) - 1, total_q=int(q.shape[0]),
        total_k=int((k_cache if k_cache is not None else mxfp8[0]).shape[0]) if total_k is None else int(total_k),
        num_heads_q=int(q.shape[1]), num_heads_kv=int(k.shape[1]), head_dim=int(q.shape[2]),
        q_out=ptr(q_out), k_cache=ptr(k_cache), v_cache=ptr(v_cache),
        conv_state_in_k=ptr(sin[0]), conv_state_in_v=ptr(sin[1]),
        conv_state_out_k=ptr(sout[0]), conv_state_out_v=ptr(sout[1]))
    st = _current_stream() if stream is None else stream
    if mxfp8 is None:
        _check(relattn_prologue(prm, st), "relattn_prologue")
    else:
        mx = RelattnKvMxfp8(k=ptr(mxfp8[0]), v=ptr(mxfp8[1]), k_scale=ptr(mxfp8[2]), v_scale=ptr(mxfp8[3]))
        _check(load_library().relattn_prologue_mxfp8(ctypes.byref(prm), ctypes.byref(mx), st),
               "relattn_prologue_mxfp8")
    return q_out


def relattn_decode_mxfp8(params: RelattnParams, kv: RelattnKvMxfp8, stream: int = 0) -> int:
    return load_library().relattn_decode_mxfp8(ctypes.byref(params), ctypes.byref(kv), stream)


def relattn_quantize_mxfp8(x: int, n_blocks: int, codes: int, scales: int, stream: int = 0) -> int:
    return load_library().relattn_quantize_mxfp8(x, n_blocks, codes, scales, stream)


def quantize_mxfp8(x, stream: Optional[int] = None):
    """MXFP8 of a contiguous bf16 CUDA tensor whose last dimension is a multiple
    of 32: (codes uint8 with x's shape, scales uint8 with the last dimension
    divided by 32)."""
    import torch
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.shape[-1] % 32:
        raise ValueError("x must be a contiguous bf16 tensor with a last dimension divisible by 32")
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty(*x.shape[:-1], x.shape[-1] // 32, dtype=torch.uint8, device=x.device)
    _check(relattn_quantize_mxfp8(x.data_ptr(), x.numel() // 32, codes.data_ptr(), scales.data_ptr(),
                                  _current_stream() if stream is None else stream),
           "relattn_quantize_mxfp8")
    return codes, scales


def decode_mxfp8(q, k8, v8, k_scale, v_scale, r, P, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q: int,
                 max_seqlen_k: int, alpha: float, window: int = 0, log_scale_base: float = 0.0,
                 num_splits: int = 0, out=None, lse=None, workspace=None, stream: Optional[int] = None):
    """Split-KV decode against an MXFP8 K / V cache: k8 / v8 uint8 E4M3 codes
    [total_k, Hkv, 128], k_scale / v_scale uint8 E8M0 [total_k, Hkv, 4].
    Returns (out, lse)."""
    out, lse = _outputs(q, out, lse)
    prm = make_params(q, k8, v8, r, P, cu_seqlens_q, cu_seqlens_k,
                      max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k, alpha=alpha,
                      window=window, log_scale_base=log_scale_base, out=out, lse=lse,
                      num_splits=num_splits)
    if workspace is None:
        workspace = decode_workspace(prm, q.device)
    if workspace is not None:
        prm.workspace = workspace.data_ptr()
        prm.workspace_bytes = workspace.numel() * workspace.element_size()
    kv = RelattnKvMxfp8(k=k8.data_ptr(), v=v8.data_ptr(), k_scale=k_scale.data_ptr(),
                        v_scale=v_scale.data_ptr())
    _check(relattn_decode_mxfp8(prm, kv, _current_stream() if stream is None else stream),
           "relattn_decode_mxfp8")
    return out, lse


def decode_paged(q, k_pool, v_pool, r, P, cu_seqlens_q, cu_seqlens_k, block_table, *,
                 page_size: int, max_seqlen_q: int, max_seqlen_k: int, alpha: float,
                 window: int = 0, log_scale_base: float = 0.0, num_splits: int = 0,
                 total_k: Optional[int] = None, out=None, lse=None, workspace=None,
                 stream: Optional[int] = None):
    """Split-KV decode against a paged KV cache: k_pool / v_pool [num_pages *
    page_size, Hkv, 128], block_table int32 [batch, max_pages_per_seq] on the
    device; cu_seqlens_k holds cumulative key counts.  ``total_k`` (their
    sum) sizes the split plan; when it is not given it is read back from
    cu_seqlens_k, which waits for the stream.  Returns (out, lse)."""
    out, lse = _outputs(q, out, lse)
    if total_k is None:
        total_k = int(cu_seqlens_k[-1].item())
    prm = make_params(q, k_pool, v_pool, r, P, cu_seqlens_q, cu_seqlens_k,
                      max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k, alpha=alpha,
                      window=window, log_scale_base=log_scale_base, out=out, lse=lse,
                      num_splits=num_splits, total_k=total_k)
    if workspace is None:
        workspace = decode_workspace(prm, q.device)
    if workspace is not None:
        prm.workspace = workspace.data_ptr()
        prm.workspace_bytes = workspace.numel() * workspace.element_size()
    kv = RelattnPagedKV(block_table=block_table.data_ptr(),
                        max_pages_per_seq=int(block_table.shape[1]), page_size=int(page_size),
                        num_pages=int(k_pool.shape[0]) // int(page_size))
    _check(relattn_decode_paged(prm, kv, _current_stream() if stream is None else stream),
           "relattn_decode_paged")
    return out, lse


def backward(q, k, v, r, P, out, lse, dout, cu_seqlens_q, cu_seqlens_k, *, max_seqlen_q: int,
             max_seqlen_k: int, alpha: float, window: int = 0, log_scale_base: float = 0.0,
             dq=None, dk=None, dv=None, dr=None, workspace=None, stream: Optional[int] = None):
    """Gradients of sum(dout * out) w.r.t. q, k, v and r (P frozen), from the
    forward's inputs and its saved out / lse.  Returns (dq, dk, dv, dr); dr is
    None when r has no channels."""
    import torch
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    r_dim = int(r.shape[-1]) if r is not None and r.dim() == 3 else 0
    if dr is None and r_dim > 0:
        dr = torch.empty_like(r)
    prm = RelattnBwdParams(
        fwd=make_params(q, k, v, r, P, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=max_seqlen_q,
                        max_seqlen_k=max_seqlen_k, alpha=alpha, window=window,
                        log_scale_base=log_scale_base, out=out, lse=lse),
        dout=dout.data_ptr(), dq=dq.data_ptr(), dk=dk.data_ptr(), dv=dv.data_ptr(),
        dr=None if dr is None else dr.data_ptr())
    if workspace is None:
        st, nbytes = relattn_backward_workspace_size(prm)
        _check(st, "relattn_backward_workspace_size")
        workspace = torch.empty(max(1, nbytes // 4), dtype=torch.float32, device=q.device)
    prm.workspace = workspace.data_ptr()
    prm.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(relattn_backward(prm, _current_stream() if stream is None else stream),
           "relattn_backward")
    return dq, dk, dv, dr
