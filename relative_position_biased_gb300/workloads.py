"""Seeded synthetic inputs for relative attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (tests, bench) and the fp64 oracle read
the tensors it returns, so the two always see identical bf16 bits.

Recipe (every workload): ``torch.Generator('cpu').manual_seed(seed)``; draw, in
this order, (1) sequence lengths if the workload has any, (2) q, (3) k, (4) v,
(5) r, all N(0, 1), then (6) P ~ N(0, p_std^2); each is drawn in fp32 and
rounded to bf16.  Shapes follow the Inkling attention facts: GQA with head size
128 (vLLM page, attention section), an 8K packed sequence with relative extent
1024 (Miles section, relative-attention paragraph), 1M context (highlights),
and a 9-position MTP verify (8 MTP heads plus the base token).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    q_lens: tuple            # query rows per sequence
    k_lens: tuple            # keys per sequence (k_len >= q_len, bottom-right aligned)
    Hq: int
    Hkv: int
    r_dim: int
    rel_extent: int
    window: int = 0          # <= 0: full attention
    log_scale_base: float = 0.0   # <= 0: no log-scale
    alpha: float = 1.0 / math.sqrt(HEAD_DIM)
    p_std: float = 0.02
    seed: int = 0
    head_dim: int = HEAD_DIM
    len_draw: tuple = ()     # (lo, hi, n) when the lengths were drawn from the seed

    @property
    def batch(self) -> int:
        return len(self.q_lens)

    @property
    def is_decode(self) -> bool:
        """Decode workloads have a few query rows per sequence against a longer KV."""
        return max(self.q_lens) <= 16 and any(lq < lk for lq, lk in zip(self.q_lens, self.k_lens))


def _uniform_lengths(gen: torch.Generator, n: int, lo: int, hi: int) -> List[int]:
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def tiny_full(seed: int = 0) -> Workload:
    """1 sequence, T=256, Hq=4, Hkv=1, r_dim=32, E=64, full causal."""
    return Workload("tiny_full_T256", (256,), (256,), 4, 1, 32, 64, seed=seed)


def swa_prefill(seed: int = 0, batch: int = 4, T: int = 8192) -> Workload:
    """4 x 8192 packed prefill, Hq=16, Hkv=2, window 4096, r_dim 64, E 1024."""
    return Workload(f"swa_prefill_{batch}x{T}_w4096", (T,) * batch, (T,) * batch,
                    16, 2, 64, 1024, window=4096, seed=seed)


def full_prefill_logscale(seed: int = 0) -> Workload:
    """4 sequences with lengths U[16384, 65536], full attention, log-scale base 65536."""
    gen = torch.Generator().manual_seed(seed)
    lens = tuple(_uniform_lengths(gen, 4, 16384, 65536))
    return Workload("full_prefill_varlen4_16k_64k_logscale", lens, lens, 16, 2, 64, 1024,
                    log_scale_base=65536.0, seed=seed, len_draw=(16384, 65536, 4))


def decode_batched(seed: int = 0, window: int = 0) -> Workload:
    """64 sequences, 1 query token each, KV lengths U[1024, 32768]."""
    gen = torch.Generator().manual_seed(seed)
    ks = tuple(_uniform_lengths(gen, 64, 1024, 32768))
    name = "decode_b64_kv1k_32k" + (f"_w{window}" if window > 0 else "_full")
    return Workload(name, (1,) * 64, ks, 16, 2, 64, 1024, window=window,
                    log_scale_base=0.0 if window > 0 else 65536.0, seed=seed,
                    len_draw=(1024, 32768, 64))


def decode_mtp_long(seed: int = 0, kv_len: int = 1 << 20) -> Workload:
    """1 sequence, 9 query rows (MTP verify width) against 1M keys, log-scale."""
    return Workload(f"decode_mtp9_kv{kv_len}", (9,), (kv_len,), 16, 2, 64, 1024,
                    log_scale_base=65536.0, seed=seed)


def make_inputs(w: Workload, device: Optional[str] = None,
                with_dout: bool = False) -> Dict[str, torch.Tensor]:
    """Draw q, k, v, r, P for workload ``w`` (CPU bf16 unless ``device`` given).

    Returns dict with q [Tq,Hq,D], k/v [Tk,Hkv,D], r [Tq,Hq,r_dim], P [r_dim,E]
    (bf16) and cu_seqlens_q / cu_seqlens_k (int32, [B+1]).  With ``with_dout``
    a step (7) draws the upstream gradient dout [Tq,Hq,D] ~ N(0, 1) in bf16
    (after P, so the other tensors are unchanged).
    """
    gen = torch.Generator().manual_seed(w.seed)
    if w.len_draw:
        # step (1): the lengths came from this seed; redraw them to keep the stream aligned
        lo, hi, n = w.len_draw
        _uniform_lengths(gen, n, lo, hi)
    Tq, Tk = sum(w.q_lens), sum(w.k_lens)
    D = w.head_dim

    def normal(*shape, std=1.0):
        x = torch.randn(*shape, generator=gen, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    out = {
        "q": normal(Tq, w.Hq, D),
        "k": normal(Tk, w.Hkv, D),
        "v": normal(Tk, w.Hkv, D),
        "r": normal(Tq, w.Hq, w.r_dim),
        "P": normal(w.r_dim, w.rel_extent, std=w.p_std),
        "cu_seqlens_q": cu_seqlens(w.q_lens),
        "cu_seqlens_k": cu_seqlens(w.k_lens),
    }
    if with_dout:
        out["dout"] = normal(Tq, w.Hq, D)
    if device is not None:
        out = {k: v.to(device) for k, v in out.items()}
    return out


def make_prologue_inputs(w: Workload, with_state: bool = False,
                         device: Optional[str] = None) -> Dict[str, torch.Tensor]:
    """Draw the inputs of the attention prologue for the chunk rows of ``w``.

    Recipe: ``torch.Generator('cpu').manual_seed(w.seed)``; draw, in this order,
    (1) the lengths if ``w`` drew them, (2) q [Tq,Hq,D], (3) k, (4) v
    [Tq,Hkv,D], all N(0, 1) rounded to bf16 (the pre-norm / pre-conv
    projections of the chunk's rows); (5) conv_k, (6) conv_v [Hkv*D, 4] fp32
    ~ N(0, 0.3^2) (taps of the order of a uniform(-1/sqrt(4), 1/sqrt(4))
    initialisation); (7) norm_q, (8) norm_k [D] fp32 ~ 1 + N(0, 0.1^2);
    then, with ``with_state``, (9) state_k, (10) state_v [B,3,Hkv*D] ~ N(0, 1)
    in bf16.  Also returns cu_seqlens_q / cu_seqlens_k (int32, [B+1]).
    """
    gen = torch.Generator().manual_seed(w.seed)
    if w.len_draw:
        lo, hi, n = w.len_draw
        _uniform_lengths(gen, n, lo, hi)
    Tq, D, C = sum(w.q_lens), w.head_dim, w.Hkv * w.head_dim

    def normal(*shape, std=1.0, mean=0.0, bf16=True):
        x = torch.randn(*shape, generator=gen, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if mean != 0.0:
            x.add_(mean)
        return x.to(torch.bfloat16) if bf16 else x

    out = {
        "q": normal(Tq, w.Hq, D),
        "k": normal(Tq, w.Hkv, D),
        "v": normal(Tq, w.Hkv, D),
        "conv_k": normal(C, 4, std=0.3, bf16=False),
        "conv_v": normal(C, 4, std=0.3, bf16=False),
        "norm_q": normal(D, std=0.1, mean=1.0, bf16=False),
        "norm_k": normal(D, std=0.1, mean=1.0, bf16=False),
        "cu_seqlens_q": cu_seqlens(w.q_lens),
        "cu_seqlens_k": cu_seqlens(w.k_lens),
    }
    if with_state:
        out["state_k"] = normal(w.batch, 3, C)
        out["state_v"] = normal(w.batch, 3, C)
    if device is not None:
        out = {k: v.to(device) for k, v in out.items()}
    return out


def page_kv(k: torch.Tensor, v: torch.Tensor, k_lens, page_size: int, seed: int = 0,
            spare_pages: int = 3):
    """Scatter contiguous K / V rows into a paged pool with a shuffled page
    order (pure layout: copies of the same bf16 rows).

    Returns (k_pool, v_pool [num_pages*page_size, Hkv, D], block_table int32
    [B, max_pages]).  Unused block-table slots hold -1; ``spare_pages`` extra
    pages, never referenced, sit in the pool; pool rows past a sequence's end
    inside its last page are filled with a large value so that reading them
    by mistake shows up in the output.
    """
    gen = torch.Generator().manual_seed(seed + 7777)
    pages = [(n + page_size - 1) // page_size for n in k_lens]
    n_pages = sum(pages) + spare_pages
    perm = torch.randperm(n_pages, generator=gen)
    Hkv, D = k.shape[1], k.shape[2]
    k_pool = torch.full((n_pages * page_size, Hkv, D), 1e4, dtype=k.dtype)
    v_pool = torch.full_like(k_pool, 1e4)
    max_pages = max(pages) if pages else 1
    table = torch.full((len(k_lens), max(1, max_pages)), -1, dtype=torch.int32)
    used, start = 0, 0
    for b, n in enumerate(k_lens):
        for i in range(pages[b]):
            pg = int(perm[used])
            used += 1
            table[b, i] = pg
            lo, hi = start + i * page_size, min(start + n, start + (i + 1) * page_size)
            k_pool[pg * page_size: pg * page_size + (hi - lo)] = k[lo:hi]
            v_pool[pg * page_size: pg * page_size + (hi - lo)] = v[lo:hi]
        start += n
    return k_pool, v_pool, table


def cu_seqlens(lens) -> torch.Tensor:
    c = [0]
    for n in lens:
        c.append(c[-1] + int(n))
    return torch.tensor(c, dtype=torch.int32)


def custom(name: str, q_lens, k_lens, Hq: int, Hkv: int, r_dim: int, rel_extent: int,
           **kw) -> Workload:
    """A workload with explicit lengths (tests and edge cases)."""
    return Workload(name, tuple(int(x) for x in q_lens), tuple(int(x) for x in k_lens),
                    Hq, Hkv, r_dim, rel_extent, **kw)


ALL = {
    "tiny": tiny_full,
    "swa_prefill": swa_prefill,
    "full_prefill_logscale": full_prefill_logscale,
    "decode_batched": decode_batched,
    "decode_mtp_long": decode_mtp_long,
}
