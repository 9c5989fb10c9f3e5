#!/usr/bin/env python3
"""Benchmark of the relative-attention forward on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
for every workload of the benchmark set:
  1. prefill of the full-attention varlen workload with log-scale (4
     sequences, lengths U[16384, 65536] from seed 0, Hq=16, Hkv=2, r_dim 64,
     E 1024) -- rel projection, QK^T, bias gather, mask, online softmax, PV,
     epilogue.  This is the largest single-GPU prefill, and `value` is its
     throughput (TFLOP/s, algorithmic flops over the call time);
  2. prefill of the sliding-window workload (4 x 8192 tokens, window 4096),
     reported under `prefill_swa` with its own roofline;
  3. split-KV decode + LSE combine of the long-context MTP verify
     (9 query rows against 1,048,576 keys, log-scale): `decode`;
  4. split-KV decode + LSE combine of the batched decode (64 sequences, 1
     query row each, KV lengths U[1024, 32768], log-scale):
     `decode.batched`;
  5. the same batch with a 4096-key window: `decode.batched_window`.
Each phase is timed with CUDA events around the call on the launching
stream; the per-phase figure is the median over the timed steps.  Decode
throughput is GB/s of visible K/V over the call time (split kernel +
combine).

The attention prologue of the SWA chunk (ShortConv of k / v, RMSNorm of q /
k, KV-cache write, conv state) is timed after the step, on its own, and
reported under `prologue` in GB/s of the bytes it must move; the backward of
the SWA prefill (dq, dk, dv, dr from the saved out / lse) likewise under
`backward`, in TFLOP/s of its algorithmic flops (five 128-deep products per
visible pair and head, plus dr in the bias band).  Two decodes are also
timed through a paged copy of their K / V (128-key pages in a shuffled pool)
and reported under `decode.paged`.  L2 is flushed by a 256 MiB write before
every timed call; the flush is outside the timed events.  Before the flush
the stream is held busy for about half a millisecond, so the host has queued
the timed call (argument marshalling, tensor-map encoding, launch) before
the device reaches it: the device-timed window holds device work only.

`e2e` is the headline metric through the C ABI from host buffers. Every step
uploads its inputs from pinned host memory and reads out / lse back, and
the timed window covers it all:
- `value`: the copies overlap the calls, as a serving loop would run them.
  Step k+1's inputs go up and step k-1's outputs come back while step k
  computes, on two copy streams with two device buffer sets.
- `serial_value`: one step at a time, copies and call back to back.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (independent replicas, weak scaling); ranks meet only for the timing
barrier and the max-over-ranks of the elapsed time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from relative_position_biased_gb300 import accounting as A  # noqa: E402
from relative_position_biased_gb300 import workloads as W  # noqa: E402

METRIC = "relattn prefill TFLOP/s & decode HBM GB/s at 1 GB300; % of roofline"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
_FWD = ["relative_position_biased_gb300/csrc/fwd_tc.cu",
        "relative_position_biased_gb300/csrc/tc_common.cuh",
        "relative_position_biased_gb300/csrc/common.cuh"]
KERNEL_SOURCES = {
    "prefill": _FWD + ["relative_position_biased_gb300/csrc/fwd_tc_main.cu"],
    "decode": _FWD + ["relative_position_biased_gb300/csrc/combine.cu",
                      "relative_position_biased_gb300/csrc/decode_tc.cu",
                      "relative_position_biased_gb300/csrc/mxfp8.cuh"],
    "backward": ["relative_position_biased_gb300/csrc/bwd_mma.cu",
                 "relative_position_biased_gb300/csrc/bwd_tc.cu",
                 "relative_position_biased_gb300/csrc/tc_common.cuh",
                 "relative_position_biased_gb300/csrc/common.cuh"],
    "prologue": ["relative_position_biased_gb300/csrc/prologue.cu",
                 "relative_position_biased_gb300/csrc/tc_common.cuh",
                 "relative_position_biased_gb300/csrc/common.cuh"],
}
L2_FLUSH_BYTES = 256 << 20
HOLD_CYCLES = 1_000_000   # device-side hold before each timed call (~0.5 ms)


def src_sha(kind: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    if os.path.exists(PEAKS_PATH):
        return json.load(open(PEAKS_PATH)), "measured"
    return FALLBACK_PEAKS, "fallback"


def load_traffic(phase: str, kind: str):
    """dram bytes per call of `phase` from a committed ncu summary, if the
    sources of its kernels (`kind`) are unchanged since the capture."""
    try:
        t = json.load(open(TRAFFIC_PATH)).get(phase)
    except (OSError, ValueError):
        return None
    if not t or t.get("src_sha") != src_sha(kind):
        return None
    return t.get("bytes_per_launch")


def median(xs):
    return statistics.median(xs) if xs else float("nan")


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def init_dist(ws: int, local: int):
    if ws <= 1:
        return None
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return dist


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def job_rate(units_per_rank: float, ms_max: float, ws: int, scale: float) -> float:
    """Whole-job throughput: every rank processed `units_per_rank` units and
    the slowest took `ms_max` ms (replicas, weak scaling); in units of `scale`."""
    return ws * units_per_rank / (ms_max * 1e-3) / scale


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workloads

# phases of one step, in order: (name, workload); the first is the headline
def step_workloads():
    return {"prefill": W.full_prefill_logscale(), "prefill_swa": W.swa_prefill(),
            "decode_long": W.decode_mtp_long(), "decode_batched": W.decode_batched(),
            "decode_batched_w": W.decode_batched(window=4096)}


STEP_PHASES = ("prefill", "prefill_swa", "decode_long", "decode_batched", "decode_batched_w")


def _kw(w):
    return dict(max_seqlen_q=max(w.q_lens), max_seqlen_k=max(w.k_lens), alpha=w.alpha,
                window=w.window, log_scale_base=w.log_scale_base)


ARG_ORDER = ("q", "k", "v", "r", "P", "cu_seqlens_q", "cu_seqlens_k")


def decode_prepass(w, mxfp8):
    """Whether a decode call of w launches the decode-row bias kernel first:
    few-row items (<= 16 rows per kv head) with a bias, unless the bf16
    few-row kernel computes the bias itself (r_dim a multiple of 8 and at
    most 64, rel_extent a multiple of 8 and at most 1024)."""
    few = max(w.q_lens) * (w.Hq // w.Hkv) <= 16
    if not (few and w.r_dim > 0 and w.rel_extent > 0):
        return False
    in_kernel = (not mxfp8 and w.r_dim % 8 == 0 and w.r_dim <= 64 and w.rel_extent % 8 == 0
                 and w.rel_extent <= 1024)
    return not in_kernel


class Phase:
    """One timed call of the library on device-resident inputs."""

    def __init__(self, name, w, host_inputs, rpb):
        self.name, self.w, self.rpb = name, w, rpb
        self.host = host_inputs
        self.dev = {k: v.cuda() for k, v in host_inputs.items()}
        self.args = [self.dev[k] for k in ARG_ORDER]
        self.out = torch.empty_like(self.dev["q"])
        self.lse = torch.empty(self.dev["q"].shape[1], self.dev["q"].shape[0],
                               dtype=torch.float32, device="cuda")
        self.decode = w.is_decode
        self.kind = "decode" if self.decode else "prefill"
        self.ws = None
        # prefill with a bias band: the band kernel, then the main kernel
        self.launches = 2 if (w.r_dim > 0 and w.rel_extent > 0) else 1
        if self.decode:
            prm = rpb.make_params(*self.args, out=self.out, lse=self.lse, **_kw(w))
            self.ws = rpb.decode_workspace(prm, "cuda")
            st, splits = rpb.relattn_decode_num_splits(prm)
            self.splits = splits
            # the decode, the combine when split, and the decode-row bias pre-pass
            # when the few-row kernel cannot compute the bias itself
            self.split_launch = 1 if splits > 1 else 0
            self.launches = 1 + self.split_launch + (1 if decode_prepass(w, mxfp8=False) else 0)
        self.flops = A.flops(w)
        self.bytes = A.kv_bytes(w)
        io = A.io_bytes(w)
        self.h2d, self.d2h = io["h2d"], io["d2h"]

    def run(self, args=None, out=None, lse=None):
        args = self.args if args is None else args
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        if self.decode:
            self.rpb.decode(*args, out=out, lse=lse, workspace=self.ws, **_kw(self.w))
        else:
            self.rpb.prefill(*args, out=out, lse=lse, **_kw(self.w))


class ProloguePhase:
    """The attention prologue over the prefill workload's chunk rows: ShortConv
    of k / v, RMSNorm of q / k, cache write and conv state out (the sequences
    start with the chunk, so no state in)."""

    def __init__(self, w, rpb, mxfp8=False):
        self.name, self.w, self.rpb = "prologue" + ("_mxfp8" if mxfp8 else ""), w, rpb
        self.decode = True   # reported in GB/s
        self.host = W.make_prologue_inputs(w)
        d = {k: v.cuda() for k, v in self.host.items()}
        self.dev = d
        Tk = sum(w.k_lens)
        self.k_cache = torch.empty(Tk, w.Hkv, 128, dtype=torch.bfloat16, device="cuda")
        self.v_cache = torch.empty_like(self.k_cache)
        self.q_out = torch.empty_like(d["q"])
        self.state = tuple(torch.empty(w.batch, 3, w.Hkv * 128, dtype=torch.bfloat16,
                                       device="cuda") for _ in range(2))
        self.launches = 2   # rows kernel + state kernel
        self.bytes = A.prologue_bytes(w, state_in=False, state_out=True)
        self.mx = None
        if mxfp8:
            # the MXFP8 cache written as well (codes + scales: 132 bytes a 128-dim row)
            k8 = torch.empty(Tk, w.Hkv, 128, dtype=torch.uint8, device="cuda")
            ks = torch.empty(Tk, w.Hkv, 4, dtype=torch.uint8, device="cuda")
            self.mx = (k8, torch.empty_like(k8), ks, torch.empty_like(ks))
            self.bytes += 2 * sum(w.q_lens) * w.Hkv * (128 + 4)

    def run(self):
        d = self.dev
        self.rpb.prologue(d["q"], d["k"], d["v"], d["conv_k"], d["conv_v"], d["norm_q"],
                          d["norm_k"], d["cu_seqlens_q"], d["cu_seqlens_k"], self.k_cache,
                          self.v_cache, q_out=self.q_out, conv_state_out=self.state, mxfp8=self.mx)


class PagedDecodePhase:
    """A decode phase re-run against a paged copy of its K / V (128-key pages
    in a shuffled pool, built once outside the timing)."""

    def __init__(self, base, page_size, rpb):
        self.name, self.w, self.rpb = base.name + "_paged", base.w, rpb
        self.decode = True
        self.base = base
        kp, vp, table = W.page_kv(base.host["k"], base.host["v"], base.w.k_lens, page_size)
        self.k_pool, self.v_pool, self.table = kp.cuda(), vp.cuda(), table.cuda()
        self.page_size = page_size
        self.launches = base.launches
        self.bytes = base.bytes

    def run(self):
        a = self.base.args
        self.rpb.decode_paged(a[0], self.k_pool, self.v_pool, a[3], a[4], a[5], a[6], self.table,
                              page_size=self.page_size, total_k=sum(self.w.k_lens),
                              out=self.base.out, lse=self.base.lse, workspace=self.base.ws,
                              **_kw(self.w))


class Mxfp8DecodePhase:
    """A decode phase re-run against an MXFP8 copy of its K / V (E4M3 codes and
    E8M0 scales per 32 dims, quantised once on the device outside the timing)."""

    def __init__(self, base, rpb):
        self.name, self.w, self.rpb = base.name + "_mxfp8", base.w, rpb
        self.decode = True
        self.base = base
        a = base.args
        self.k8, self.ks = rpb.quantize_mxfp8(a[1])
        self.v8, self.vs = rpb.quantize_mxfp8(a[2])
        self.launches = 1 + base.split_launch + (1 if decode_prepass(base.w, mxfp8=True) else 0)
        self.bytes = A.kv_bytes_mxfp8(base.w)      # bytes the kernel must read
        self.bytes_bf16 = base.bytes                 # the same keys in bf16

    def run(self):
        a = self.base.args
        self.rpb.decode_mxfp8(a[0], self.k8, self.v8, self.ks, self.vs, a[3], a[4], a[5], a[6],
                              out=self.base.out, lse=self.base.lse, workspace=self.base.ws,
                              **_kw(self.w))


class BackwardPhase:
    """The backward of the prefill workload: gradients of sum(dout * out)
    w.r.t. q, k, v, r from the forward's saved out / lse (computed once,
    outside the timing)."""

    def __init__(self, w, rpb):
        self.name, self.w, self.rpb = "backward", w, rpb
        self.decode = False   # reported in TFLOP/s
        host = W.make_inputs(w, with_dout=True)
        d = {k: v.cuda() for k, v in host.items()}
        self.d = d
        self.args = [d[k] for k in ARG_ORDER]
        self.out, self.lse = rpb.prefill(*self.args, **_kw(w))
        self.dq, self.dk, self.dv = (torch.empty_like(d["q"]), torch.empty_like(d["k"]),
                                     torch.empty_like(d["v"]))
        self.dr = torch.empty_like(d["r"])
        prm = rpb.RelattnBwdParams(fwd=rpb.make_params(*self.args, out=self.out, lse=self.lse,
                                                        **_kw(w)))
        st, nbytes = rpb.relattn_backward_workspace_size(prm)
        if st != 0:
            raise SystemExit("relattn_backward_workspace_size failed")
        self.ws = torch.empty(max(1, nbytes // 4), dtype=torch.float32, device="cuda")
        # on the tcgen05 path: R, D, dq outside the band, dq / dr of the band, dk / dv
        # (without a bias: D, dq, dk / dv), and the dk / dv reduce when an even
        # GQA group of 4 or more heads is split between two CTAs
        group = w.Hq // w.Hkv
        self.launches = ((5 if (w.r_dim > 0 and w.rel_extent > 0) else 3) +
                         (1 if group >= 4 and group % 2 == 0 else 0))
        self.flops = A.bwd_flops(w)

    def run(self):
        a = self.args
        self.rpb.backward(a[0], a[1], a[2], a[3], a[4], self.out, self.lse, self.d["dout"],
                          a[5], a[6], dq=self.dq, dk=self.dk, dv=self.dv, dr=self.dr,
                          workspace=self.ws, **_kw(self.w))


def timed_steps(phases, steps, flush):
    """Run `steps` steps; return per-phase lists of kernel times (ms)."""
    stream = torch.cuda.current_stream()
    times = {p.name: [] for p in phases}
    events = []
    for _ in range(steps):
        for p in phases:
            torch.cuda._sleep(HOLD_CYCLES)
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            p.run()
            b.record(stream)
            events.append((p.name, a, b))
    torch.cuda.synchronize()
    for name, a, b in events:
        times[name].append(a.elapsed_time(b))
    return times


def e2e_steps(phases, steps, flush):
    """Same step with host buffers: pinned H2D of every input, the call, and a
    D2H read of out and lse, all inside the timed events."""
    stream = torch.cuda.current_stream()
    pinned = {}
    for p in phases:
        pinned[p.name] = ({k: v.pin_memory() for k, v in p.host.items()},
                          torch.empty(p.out.shape, dtype=p.out.dtype).pin_memory(),
                          torch.empty(p.lse.shape, dtype=p.lse.dtype).pin_memory())
    staging = {p.name: {k: torch.empty_like(v) for k, v in p.dev.items()} for p in phases}
    times = {p.name: [] for p in phases}
    events = []
    for _ in range(steps):
        for p in phases:
            hin, hout, hlse = pinned[p.name]
            dst = staging[p.name]
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k in ARG_ORDER:
                dst[k].copy_(hin[k], non_blocking=True)
            p.run(args=[dst[k] for k in ARG_ORDER])
            hout.copy_(p.out, non_blocking=True)
            hlse.copy_(p.lse, non_blocking=True)
            b.record(stream)
            events.append((p.name, a, b))
    torch.cuda.synchronize()
    for name, a, b in events:
        times[name].append(a.elapsed_time(b))
    return times


def e2e_pipelined(phases, steps, flush):
    """Host-buffer throughput with the copies overlapped, per phase.

    Every step still uploads its inputs from pinned host memory and reads
    out / lse back.  Step k+1's inputs go up on one copy stream while step k
    computes, and step k's outputs come back on another while step k+1
    computes.  Two device input / output sets alternate.  Returns the ms per
    step between events bracketing all `steps` steps (the uploads move far
    more than L2 holds, so no flush between steps).
    """
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    res = {}
    for p in phases:
        hin = {k: v.pin_memory() for k, v in p.host.items()}
        dev = [{k: torch.empty_like(v) for k, v in p.dev.items()} for _ in range(2)]
        outs = [(torch.empty_like(p.out), torch.empty_like(p.lse)) for _ in range(2)]
        hout = [(torch.empty(p.out.shape, dtype=p.out.dtype).pin_memory(),
                 torch.empty(p.lse.shape, dtype=p.lse.dtype).pin_memory()) for _ in range(2)]
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        flush.zero_()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(comp)
        cin.wait_stream(comp)
        cout.wait_stream(comp)

        def upload(k):
            s = k % 2
            with torch.cuda.stream(cin):
                if k >= 2:
                    cin.wait_event(comp_done[s])   # step k-2 has finished reading set s
                for name in ARG_ORDER:
                    dev[s][name].copy_(hin[name], non_blocking=True)
                in_ready[s].record(cin)

        upload(0)
        for k in range(steps):
            s = k % 2
            if k + 1 < steps:
                upload(k + 1)
            comp.wait_event(in_ready[s])
            if k >= 2:
                comp.wait_event(out_done[s])       # step k-2's outputs are back on the host
            p.run(args=[dev[s][n] for n in ARG_ORDER], out=outs[s][0], lse=outs[s][1])
            comp_done[s].record(comp)
            with torch.cuda.stream(cout):
                cout.wait_event(comp_done[s])
                hout[s][0].copy_(outs[s][0], non_blocking=True)
                hout[s][1].copy_(outs[s][1], non_blocking=True)
                out_done[s].record(cout)
        comp.wait_stream(cin)
        comp.wait_stream(cout)
        end.record(comp)
        torch.cuda.synchronize()
        res[p.name] = start.elapsed_time(end) / steps
    return res


# ------------------------------------------------------------------ CPU oracle timing

def oracle_sample_rows(w, n_rows, seed=7):
    rng = np.random.default_rng(seed)
    total = sum(w.q_lens)
    return np.sort(rng.choice(total, size=min(n_rows, total), replace=False)).astype(np.int64)


def time_oracle(w, inp, rows):
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.forward(inp["q"], inp["k"], inp["v"], inp["r"], inp["P"], inp["cu_seqlens_q"],
                   inp["cu_seqlens_k"], alpha=w.alpha, window=w.window,
                   log_scale_base=w.log_scale_base, rows=rows)
    dt = time.perf_counter() - t0
    return dt, A.flops(w, rows), oracle.max_threads()


def decode_rows_bytes(w, rows):
    """K/V bytes the selected decode rows read (each row streams its visible keys)."""
    return A.visible_pairs(w, rows) * w.Hkv * w.head_dim * 2 * 2 // max(1, len(rows))


# ------------------------------------------------------------------ arms

def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = step_workloads()["prefill"]
    inp = W.make_inputs(w)
    # each step: a sample of query rows sized to about a second of oracle work
    cal = oracle_sample_rows(w, 16, seed=3)
    for _ in range(args.warmup):
        cdt, _, _ = time_oracle(w, inp, cal)
    n_step = int(min(sum(w.q_lens), max(16, 16 * 1.0 / max(cdt, 1e-3))))
    dts, fl = [], 0
    t_all0 = time.perf_counter()
    for s in range(args.steps):
        r = oracle_sample_rows(w, n_step, seed=100 + s)
        dt, f, cores = time_oracle(w, inp, r)
        dts.append(dt)
        fl += f
    elapsed = sum(dts)
    value = fl / elapsed / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": f"{n_step} random query rows x {w.Hq} heads per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x {n_step} random query rows x {w.Hq} heads of {w.name}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_all0,
    }
    print(json.dumps(line), flush=True)
    return 0


CPU_SAMPLE_SECONDS = 10.0   # oracle work for the cpu_baseline (bounded sample)


def cpu_baseline(wl, host):
    """Oracle on the host cores over a bounded sample of the headline prefill
    workload: a short calibration sizes the sample to about
    CPU_SAMPLE_SECONDS.  Beside it: every row of the MTP decode, one sequence
    of the SWA chunk's prologue, and the last 64 rows of one SWA sequence's
    backward."""
    w = wl["prefill"]
    cal = oracle_sample_rows(w, 16, seed=3)
    cdt, _, _ = time_oracle(w, host["prefill"], cal)
    n = int(min(sum(w.q_lens), max(16, 16 * CPU_SAMPLE_SECONDS / max(cdt, 1e-3))))
    rows = oracle_sample_rows(w, n)
    dt, f, cores = time_oracle(w, host["prefill"], rows)
    wd = wl["decode_long"]
    drows = np.arange(sum(wd.q_lens), dtype=np.int64)   # every MTP row
    ddt, _, _ = time_oracle(wd, host["decode_long"], drows)
    # the prologue oracle over the first sequence of the SWA chunk
    from oracle import prologue as OP
    ws_ = wl["prefill_swa"]
    wp = W.custom("prologue_sample", ws_.q_lens[:1], ws_.k_lens[:1], ws_.Hq, ws_.Hkv, 0, 0)
    pin = W.make_prologue_inputs(wp)
    t0 = time.perf_counter()
    OP.prologue(pin["q"], pin["k"], pin["v"], pin["conv_k"], pin["conv_v"], pin["norm_q"],
                pin["norm_k"], pin["cu_seqlens_q"], pin["cu_seqlens_k"])
    pdt = time.perf_counter() - t0
    pro = {"value": A.prologue_bytes(wp) / pdt / 1e9, "unit": "GB/s",
           "sample": f"one {wp.q_lens[0]}-row sequence x ({ws_.Hq} q + 2x{ws_.Hkv} kv) heads "
                     f"({pdt:.1f} s)"}
    # the backward oracle over the last 64 rows of the first SWA sequence (a
    # chunk at the end of its 8,192 keys)
    import oracle
    T0 = ws_.q_lens[0]
    wb = W.custom("bwd_sample", [64], [T0], ws_.Hq, ws_.Hkv, ws_.r_dim, ws_.rel_extent,
                  window=ws_.window)
    bin_ = W.make_inputs(ws_, with_dout=True)
    sl = slice(T0 - 64, T0)
    t0 = time.perf_counter()
    oracle.backward(bin_["q"][sl], bin_["k"][:T0], bin_["v"][:T0], bin_["r"][sl], bin_["P"],
                    bin_["dout"][sl], [0, 64], [0, T0], alpha=ws_.alpha, window=ws_.window)
    bdt = time.perf_counter() - t0
    bwd = {"value": A.bwd_flops(wb) / bdt / 1e12, "unit": "TFLOP/s",
           "sample": f"the last 64 rows x {ws_.Hq} heads of one {T0}-token sequence ({bdt:.1f} s, "
                     f"{ws_.Hkv} threads: one task per kv head)"}
    return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "prologue": pro, "backward": bwd,
            "sample": f"{n} random query rows x {w.Hq} heads of {w.name} ({dt:.1f} s)",
            "decode": {"value": decode_rows_bytes(wd, drows) / ddt / 1e9, "unit": "GB/s",
                       "sample": f"all {len(drows)} query rows x {wd.Hq} heads of {wd.name} ({ddt:.1f} s)"}}


def _roofline(bound, achieved, peak, unit, traffic, peak_kind, **extra):
    r = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
         "frac": achieved / peak, "traffic": traffic}
    r.update(extra)
    r["peak_source"] = peak_kind
    return r


def gpu_arm(args):
    ws, rank, local = dist_env()
    dist = init_dist(ws, local)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local if ws > 1 else 0)
    import relative_position_biased_gb300 as rpb
    rpb.build()
    rpb.load_library()

    wl = step_workloads()
    if args.only == "prologue":
        return single_phase(args, ProloguePhase(wl["prefill_swa"], rpb))
    if args.only == "backward":
        return single_phase(args, BackwardPhase(wl["prefill_swa"], rpb))
    if args.only and args.only.endswith("_mxfp8"):
        n = args.only[:-len("_mxfp8")]
        mx = Mxfp8DecodePhase(Phase(n, wl[n], W.make_inputs(wl[n]), rpb), rpb)
        return single_phase(args, mx)
    if args.only:
        return single_phase(args, Phase(args.only, wl[args.only], W.make_inputs(wl[args.only]), rpb))
    host = {k: W.make_inputs(w) for k, w in wl.items()}
    phases = [Phase(k, wl[k], host[k], rpb) for k in STEP_PHASES]
    ph = {p.name: p for p in phases}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    for _ in range(args.warmup):
        for p in phases:
            p.run()
    torch.cuda.synchronize()
    if rpb.relattn_get_device_error() != 0:
        raise SystemExit("device error word set during warm-up")

    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = time.perf_counter()
        times = timed_steps(phases, args.steps, flush)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(dist)
    clocks = clk.summary()
    if rpb.relattn_get_device_error() != 0:
        raise SystemExit("device error word set during the timed steps")

    # the attention prologue of the SWA chunk, timed on its own
    pro = ProloguePhase(wl["prefill_swa"], rpb)
    for _ in range(args.warmup):
        pro.run()
    torch.cuda.synchronize()
    pro_mx = ProloguePhase(wl["prefill_swa"], rpb, mxfp8=True)
    for _ in range(args.warmup):
        pro_mx.run()
    torch.cuda.synchronize()
    pro_tt = timed_steps([pro, pro_mx], args.steps, flush)
    pro_t = pro_tt["prologue"]
    torch.cuda.synchronize()
    if rpb.relattn_get_device_error() != 0:
        raise SystemExit("device error word set by the prologue")
    # two decodes again through 128-key pages of a shuffled pool
    paged = [PagedDecodePhase(ph[n], 128, rpb) for n in ("decode_long", "decode_batched")]
    for _ in range(args.warmup):
        for p in paged:
            p.run()
    torch.cuda.synchronize()
    pg_t = timed_steps(paged, args.steps, flush)
    torch.cuda.synchronize()
    if rpb.relattn_get_device_error() != 0:
        raise SystemExit("device error word set by the paged decode")
    for p in paged:
        del p.k_pool, p.v_pool
    # the two batched decodes again on an MXFP8 K / V cache
    mx = [Mxfp8DecodePhase(ph[n], rpb) for n in ("decode_batched", "decode_batched_w")]
    for _ in range(args.warmup):
        for p in mx:
            p.run()
    torch.cuda.synchronize()
    mx_t = timed_steps(mx, args.steps, flush)
    torch.cuda.synchronize()
    if rpb.relattn_get_device_error() != 0:
        raise SystemExit("device error word set by the MXFP8 decode")
    for p in mx:
        del p.k8, p.v8, p.ks, p.vs
    # the backward of the SWA prefill, timed on its own
    bwd = BackwardPhase(wl["prefill_swa"], rpb)
    for _ in range(args.warmup):
        bwd.run()
    torch.cuda.synchronize()
    bwd_t = timed_steps([bwd], max(2, min(args.steps, 5)), flush)["backward"]
    torch.cuda.synchronize()
    if rpb.relattn_get_device_error() != 0:
        raise SystemExit("device error word set by the backward")
    del bwd.d, bwd.dq, bwd.dk, bwd.dv, bwd.dr, bwd.out, bwd.lse, bwd.args

    e2e_t = e2e_steps(phases, max(1, min(args.steps, 5)), flush)
    torch.cuda.synchronize()
    e2e_steps_pipe = max(4, min(args.steps, 8))
    e2e_p = e2e_pipelined(phases, e2e_steps_pipe, flush)

    # per-phase device time: the median of the timed steps, max over ranks
    ms = {n: max_over_ranks(median(times[n]), dist) for n in STEP_PHASES}
    step_ms = max_over_ranks(sum(median(times[n]) for n in STEP_PHASES), dist)
    pro_ms = max_over_ranks(median(pro_t), dist)
    pro_mx_ms = max_over_ranks(median(pro_tt["prologue_mxfp8"]), dist)
    pg_ms = {p.name: max_over_ranks(median(pg_t[p.name]), dist) for p in paged}
    mx_ms = {p.name: max_over_ranks(median(mx_t[p.name]), dist) for p in mx}
    bwd_ms = max_over_ranks(median(bwd_t), dist)
    e2e_ser = {n: max_over_ranks(median(e2e_t[n]), dist) for n in STEP_PHASES}
    e2e_pipe = {n: max_over_ranks(e2e_p[n], dist) for n in STEP_PHASES}
    if rank != 0:
        return 0
    peaks, peak_kind = load_peaks()
    tf_peak, hbm_peak = peaks["bf16_tflops"], peaks["hbm_gbs"]
    tf_src = f"{peak_kind} bf16 dense (burst)"
    hbm_src = f"{peak_kind} HBM copy"

    def tflops(p):   # one GPU's rate
        return p.flops / (ms[p.name] * 1e-3) / 1e12

    def gbs(p):
        return p.bytes / (ms[p.name] * 1e-3) / 1e9

    pre, swa, dl, db, dbw = (ph[n] for n in STEP_PHASES)
    prefill_kernels = ("relattn_fwd_tc_kernel<prefill, band> + relattn_fwd_tc_main_kernel "
                       "(the two launches of one prefill call)")
    pro_gbs = pro.bytes / (pro_ms * 1e-3) / 1e9
    bwd_tf = bwd.flops / (bwd_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": job_rate(pre.flops, ms["prefill"], ws, 1e12),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": pre.w.name,
            "step": " + ".join(ph[n].w.name for n in STEP_PHASES),
            "prefill": {"batch": pre.w.batch, "seq_lens": list(pre.w.q_lens), "Hq": pre.w.Hq,
                        "Hkv": pre.w.Hkv, "head_dim": 128, "r_dim": pre.w.r_dim,
                        "rel_extent": pre.w.rel_extent, "window": pre.w.window,
                        "log_scale_base": pre.w.log_scale_base, "flops": pre.flops},
            "prefill_swa": {"batch": swa.w.batch, "seq_len": swa.w.q_lens[0],
                            "window": swa.w.window, "flops": swa.flops},
            "decode_long": {"q_rows": dl.w.q_lens[0], "kv_len": dl.w.k_lens[0],
                            "log_scale_base": dl.w.log_scale_base, "kv_bytes": dl.bytes,
                            "splits": dl.splits},
            "decode_batched": {"batch": db.w.batch, "kv_lens": "U[1024,32768]",
                               "kv_bytes": db.bytes, "splits": db.splits},
            "decode_batched_w": {"batch": dbw.w.batch, "kv_lens": "U[1024,32768]",
                                 "window": dbw.w.window, "kv_bytes": dbw.bytes,
                                 "splits": dbw.splits},
            "statistic": f"median of {args.steps} timed steps per phase",
            "l2": "flushed by a 256 MiB write before every timed call",
            "parallelism": f"replicas x{ws}",
        },
        "phases_ms": dict(ms),
        "roofline": _roofline("tensor", tflops(pre), tf_peak, "TFLOP/s",
                              load_traffic("prefill_full", "prefill"), tf_src,
                              kernel=prefill_kernels, workload=pre.w.name),
        "prefill_swa": {
            "value": job_rate(swa.flops, ms["prefill_swa"], ws, 1e12), "unit": "TFLOP/s",
            "ms": ms["prefill_swa"], "workload": swa.w.name, "flops": swa.flops,
            "roofline": _roofline("tensor", tflops(swa), tf_peak, "TFLOP/s",
                                  load_traffic("prefill_swa", "prefill"), tf_src,
                                  kernel=prefill_kernels)},
        "decode": {
            "value": job_rate(dl.bytes, ms["decode_long"], ws, 1e9), "unit": "GB/s",
            "workload": dl.w.name, "ms": ms["decode_long"],
            "roofline": _roofline("hbm", gbs(dl), hbm_peak, "GB/s",
                                  load_traffic("decode_long", "decode"), hbm_src,
                                  frac_vs_8tbs=gbs(dl) / 8000.0,
                                  kernel="relattn_fwd_tc_kernel<decode> + relattn_combine_kernel"),
            "batched": {"value": job_rate(db.bytes, ms["decode_batched"], ws, 1e9), "unit": "GB/s",
                        "workload": db.w.name, "ms": ms["decode_batched"],
                        "frac": gbs(db) / hbm_peak,
                        "roofline": _roofline("hbm", gbs(db), hbm_peak, "GB/s",
                                              load_traffic("decode_batched", "decode"), hbm_src,
                                              frac_vs_8tbs=gbs(db) / 8000.0)},
            "batched_window": {"value": job_rate(dbw.bytes, ms["decode_batched_w"], ws, 1e9),
                               "unit": "GB/s", "workload": dbw.w.name,
                               "ms": ms["decode_batched_w"], "frac": gbs(dbw) / hbm_peak,
                               "roofline": _roofline("hbm", gbs(dbw), hbm_peak, "GB/s",
                                                     load_traffic("decode_batched_w4096", "decode"),
                                                     hbm_src, frac_vs_8tbs=gbs(dbw) / 8000.0)},
            "paged": {p.name: {"value": p.bytes / (pg_ms[p.name] * 1e-3) / 1e9, "unit": "GB/s",
                               "ms": pg_ms[p.name], "page_size": p.page_size,
                               "frac": p.bytes / (pg_ms[p.name] * 1e-3) / 1e9 / hbm_peak}
                      for p in paged},
            "mxfp8": {p.name: {"value": p.bytes / (mx_ms[p.name] * 1e-3) / 1e9, "unit": "GB/s",
                               "ms": mx_ms[p.name], "bytes": p.bytes,
                               "traffic": load_traffic(p.name, "decode"),
                               "frac": p.bytes / (mx_ms[p.name] * 1e-3) / 1e9 / hbm_peak,
                               "bf16_equivalent": p.bytes_bf16 / (mx_ms[p.name] * 1e-3) / 1e9,
                               "what": "E4M3 K / V codes + E8M0 scales per 32 dims; q quantised "
                                       "in the kernel, Q K^T as E4M3 products, V dequantised "
                                       "to bf16 for P V"}
                      for p in mx},
        },
        "prologue": {
            "value": job_rate(pro.bytes, pro_ms, ws, 1e9), "unit": "GB/s", "ms": pro_ms,
            "workload": swa.w.name,
            "what": "ShortConv k/v + RMSNorm q/k + KV-cache write + conv state out",
            "bytes": pro.bytes, "launches": args.steps * pro.launches,
            "roofline": _roofline("hbm", pro_gbs, hbm_peak, "GB/s",
                                  load_traffic("prologue", "prologue"), hbm_src),
            "mxfp8": {"ms": pro_mx_ms, "value": pro_mx.bytes / (pro_mx_ms * 1e-3) / 1e9, "unit": "GB/s",
                      "bytes": pro_mx.bytes, "vs_bf16_only": pro_mx_ms / pro_ms,
                      "what": "the same prologue writing the MXFP8 cache (E4M3 codes + E8M0 scales) "
                              "beside the bf16 cache, quantise fused"}},
        "backward": {
            "value": job_rate(bwd.flops, bwd_ms, ws, 1e12), "unit": "TFLOP/s", "ms": bwd_ms,
            "workload": swa.w.name,
            "what": "dq, dk, dv, dr of sum(dout * out), P frozen", "flops": bwd.flops,
            "launches": len(bwd_t) * bwd.launches,
            "roofline": _roofline("tensor", bwd_tf, tf_peak, "TFLOP/s",
                                  load_traffic("backward", "backward"), tf_src,
                                  kernel="relattn_bwd_rel_kernel + relattn_bwd_dot_kernel + "
                                         "relattn_bwd_dq_tc_kernel + relattn_bwd_dq_kernel (band, "
                                         "mma.sync) + relattn_bwd_dkdv_tc_kernel (heads split "
                                         "over two CTAs) + relattn_bwd_dkv_reduce_kernel")},
        "e2e": {"value": job_rate(pre.flops, e2e_pipe["prefill"], ws, 1e12), "unit": "TFLOP/s",
                "workload": pre.w.name,
                "h2d_bytes_per_step": sum(p.h2d for p in phases),
                "d2h_bytes_per_step": sum(p.d2h for p in phases),
                "path": "pinned host buffers -> H2D -> relattn_* C ABI -> D2H out+lse",
                "overlap": f"{e2e_steps_pipe} steps per phase; step k+1's H2D and step k-1's D2H "
                           "on two copy streams while step k computes (two device buffer sets)",
                "serial_value": job_rate(pre.flops, e2e_ser["prefill"], ws, 1e12),
                "phases": {n: {"value": (job_rate(ph[n].flops, e2e_pipe[n], ws, 1e12) if not ph[n].decode
                                         else job_rate(ph[n].bytes, e2e_pipe[n], ws, 1e9)),
                               "serial_value": (job_rate(ph[n].flops, e2e_ser[n], ws, 1e12)
                                                if not ph[n].decode
                                                else job_rate(ph[n].bytes, e2e_ser[n], ws, 1e9)),
                               "unit": "GB/s" if ph[n].decode else "TFLOP/s",
                               "h2d_bytes": ph[n].h2d, "d2h_bytes": ph[n].d2h}
                           for n in STEP_PHASES}},
        "gpu_launches": args.steps * sum(p.launches for p in phases),
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, host)
    print(json.dumps(line), flush=True)
    return 0


def splits_sweep(args):
    """Decode time against the split count, for the heuristic's choice
    (num_splits = 0) and fixed counts around it; one JSON line per point."""
    import relative_position_biased_gb300 as rpb
    rpb.build()
    rpb.load_library()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    cases = (("decode_batched", W.decode_batched(), [0, 1, 2, 3, 4, 6, 8, 12, 16]),
             ("decode_batched_w4096", W.decode_batched(window=4096), [0, 1, 2, 3, 4, 6, 8]),
             ("decode_long", W.decode_mtp_long(), [0, 38, 76, 152, 228]))
    for name, w, counts in cases:
        d = {k: v.cuda() for k, v in W.make_inputs(w).items()}
        args_ = [d[k] for k in ARG_ORDER]
        out = torch.empty_like(d["q"])
        lse = torch.empty(w.Hq, sum(w.q_lens), dtype=torch.float32, device="cuda")
        nbytes = A.kv_bytes(w)
        for ns in counts:
            prm = rpb.make_params(*args_, out=out, lse=lse, num_splits=ns, **_kw(w))
            ws = rpb.decode_workspace(prm, "cuda")
            _, splits = rpb.relattn_decode_num_splits(prm)

            def run(ns=ns, ws=ws):
                rpb.decode(*args_, out=out, lse=lse, workspace=ws, num_splits=ns, **_kw(w))
            ph = types.SimpleNamespace(name=f"{name}_s{ns}", run=run)   # a phase with this split count
            for _ in range(max(3, args.warmup)):
                ph.run()
            t = sorted(timed_steps([ph], args.steps, flush)[ph.name])
            ms = t[len(t) // 2]
            print(json.dumps({"workload": w.name, "num_splits": ns, "splits": splits,
                              "ms_median": ms, "GBs": nbytes / (ms * 1e-3) / 1e9}), flush=True)
    return 0


def single_phase(args, p):
    """One phase alone (used for profiling captures): warm-up, K timed calls."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        p.run()
    torch.cuda.synchronize()
    t = timed_steps([p], args.steps, flush)[p.name]
    ms = median(t)
    rate = (p.bytes / (ms * 1e-3) / 1e9, "GB/s") if p.decode else \
        (p.flops / (ms * 1e-3) / 1e12, "TFLOP/s")
    print(json.dumps({"phase": p.name, "workload": p.w.name, "ms": ms, "value": rate[0],
                      "unit": rate[1], "steps": args.steps, "warmup": args.warmup}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=list(STEP_PHASES) + ["prologue", "backward", "decode_batched_mxfp8",
                                                           "decode_batched_w_mxfp8"],
                    help="time one phase alone (profiling captures)")
    ap.add_argument("--splits-sweep", action="store_true",
                    help="time the decodes at fixed split counts beside the heuristic's choice")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.splits_sweep:
        return splits_sweep(args)
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
