#!/usr/bin/env python
"""Benchmark of the causal depthwise conv1d forward family on one GB300 (or N
independent replicas under torchrun).

One step is one pass over the whole hot path, on inputs already resident in
HBM:
  1. ccv_fwd   large prefill, 4 sequences x 4096 tokens, dim 8192, W 4,
               x stored (tokens, dim)  [channel-last]
  2. ccv_fwd   the same batch stored (dim, tokens)  [channel-first]
  3. ccv_update decode, 256 rows x dim 8192, state pool (512, 8192, 3)
  4. paged_sconv_seq_metadata + paged_sconv_fwd: H=16 x ws=128, W 4,
     cache [1024,16,16,512], 32 mixed requests
All inputs are seeded synthetic N(0, 0.02^2) bf16 (see workloads.py).  The
headline value is algorithmic HBM bytes of the step / device time of the step
(GB/s); the parts, prefill Mtok/s and decode us/call ride in the same line.
Prefill inputs (2 x 268 MB in, 2 x 268 MB out) exceed the 129 MB L2, so every
part of every step starts L2-cold without an explicit flush.

--impl reference times the CPU oracle on the host cores on a bounded channel
sample of the same workload, in the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "varlen causal_conv1d HBM GB/s & Mtok/s at dim 8192 bf16; decode us/call"
WORKLOAD = ("prefill 4x4096 tokens dim 8192 W4 (tokens,dim) + same in (dim,tokens) "
            "+ paged short conv H16 ws128 32 requests + decode 256x8192")


# ----------------------------------------------------------- byte counts ----

def prefill_bytes(case) -> int:
    """x read + out write + state read (has_init) and write + weight + bias +
    index vectors, for the non-pad sequences that own tokens."""
    W, dim = case.width, case.dim
    tokens = 0
    state = 0
    for i, L in enumerate(case.lengths):
        pad = case.cache_indices is not None and int(case.cache_indices[i]) == case.pad_slot_id
        if pad or L == 0:
            continue
        tokens += L
        init = case.has_initial_state is not None and bool(case.has_initial_state[i])
        state += dim * (W - 1) * 2 * (2 if init else 1)
    small = dim * W * 2 + (dim * 2 if case.bias is not None else 0)
    small += 4 * (len(case.lengths) + 1) + 4 * len(case.lengths) + len(case.lengths)
    return 4 * dim * tokens + state + small


def prefill_tokens(case) -> int:
    return sum(L for i, L in enumerate(case.lengths)
               if not (case.cache_indices is not None
                       and int(case.cache_indices[i]) == case.pad_slot_id))


def decode_bytes(case) -> int:
    x3 = case.x if case.x.dim() == 3 else case.x.unsqueeze(-1)
    B, dim, S = x3.shape
    W = case.weight.shape[1]
    rows = B if case.conv_state_indices is None else int(
        (case.conv_state_indices != case.pad_slot_id).sum())
    per_row = dim * 2 * (2 * S + (W - 1) + (W - 2 + S))
    return rows * per_row + dim * W * 2 + dim * 2 + 4 * B


def spec_bytes(case) -> int:
    """Speculative verify: per non-pad row x read + out write + the window
    read + the intermediate windows + the output-line windows (+ the shifted
    columns when no buffer is given), plus weights, bias and indices."""
    B, dim, S = case.x.shape
    W = case.weight.shape[1]
    rows = [b for b in range(B) if int(case.conv_state_indices[b]) != case.pad_slot_id]
    per_row = dim * 2 * (2 * S + (W - 1))
    total = 0
    for b in rows:
        total += per_row
        if case.intermediate_conv_window is not None:
            total += S * dim * (W - 1) * 2
        if case.output_state_indices is not None:
            total += int((case.output_state_indices[b, :S] >= 0).sum()) * dim * (W - 1) * 2
        if case.intermediate_conv_window is None and case.output_state_indices is None:
            total += dim * (W - 2 + S) * 2
    idx_bytes = 4 * B * (1 + (case.num_accepted_tokens is not None)
                         + (S if case.output_state_indices is not None else 0))
    return total + dim * W * 2 + dim * 2 + idx_bytes


_PAGED_BYTES = {}


def paged_bytes(case) -> int:
    """x read + out write + cache insert + pre-forward cache taps + weights +
    per-token metadata + block-table reads."""
    key = (id(case), case.x.shape, case.weight.shape)
    if key not in _PAGED_BYTES:
        _PAGED_BYTES[key] = _paged_bytes(case)
    return _PAGED_BYTES[key]


def _paged_bytes(case) -> int:
    """x read + out write for every row, the insert of every real token, each
    distinct cached (request, position) the pre-forward taps read, each
    distinct block-table entry those reads resolve through, the weights, the
    four per-token index values and the query_start_loc of the metadata."""
    C = case.x.shape[1]
    W = case.weight.shape[1]
    T = case.T
    N = case.block_size
    max_blocks = case.block_table.shape[1]
    real = (case.slot_mapping >= 0)
    n_real = int(real.sum())
    cached, entries = set(), set()
    for t in range(T):
        if not bool(real[t]):
            continue
        pos = int(case.positions[t])
        qs = int(case.query_start[t])
        req = int(case.seq_idx[t])
        for iw in range(W):
            src = pos - (W - 1) + iw
            row = t - (W - 1) + iw
            if src >= 0 and row < qs:
                cached.add((req, src))
                entries.add((req, min(src // N, max_blocks - 1)))
    return (2 * T * C * 2 + n_real * C * 2 + len(cached) * C * 2 + C * W * 2
            + T * (8 + 4 + 8 + 4) + len(entries) * 4 + 4 * (len(case.req_lengths) + 1))


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms (read only).
    Only samples taken between mark("start") and mark("end") are summarised
    (all samples if none fell inside a very short timed region)."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.gpu_id = gpu_id_for_smi(device)
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def mark(self, which: str):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        return summarize_clocks(rows, self.t0, self.t1)


def gpu_id_for_smi(device) -> str:
    """The id nvidia-smi knows this CUDA device by (its UUID when available)."""
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except (AttributeError, RuntimeError):
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    idx = device.index or 0
    if vis:
        return vis.split(",")[idx].strip()
    return str(idx)


def _is_active(v: str) -> bool:
    return v.strip().lower() in ("active", "1", "yes")


def _stamp(ts: str):
    from datetime import datetime

    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.strptime(ts, fmt).timestamp()
        except ValueError:
            continue
    return None


def summarize_clocks(rows, t0=None, t1=None) -> dict:
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    parsed = []
    for r in rows:
        try:
            parsed.append((_stamp(r[0]), float(r[1]), float(r[2]), r[5:9]))
        except ValueError:
            continue
    inside = [p for p in parsed
              if t0 is not None and t1 is not None and p[0] is not None and t0 <= p[0] <= t1]
    use = inside if inside else parsed
    sm = [p[1] for p in use if p[1] > 0]
    reasons = sorted({n for p in use for n, v in zip(names, p[3]) if _is_active(v)})
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max((p[2] for p in use), default=None),
            "reasons": reasons, "samples": len(use),
            "window": "timed region" if inside else "whole run (timed region shorter than 100 ms)"}


# ----------------------------------------------------------- distributed ----

def dist_env():
    """(rank, world_size, local_rank) from torchrun's environment, or (0, 1, 0)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(value: float, device=None) -> float:
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Weak scaling: every rank processes its own replica of the step."""
    return units_per_rank_step * steps * world / max_seconds


# ------------------------------------------------------------- roofline ----

# Translation unit that defines each kernel the bench times.
KERNEL_SOURCE = {
    "fwd_cl_async_kernel": "ccv_fwd.cu",
    "fwd_cf_async_kernel": "ccv_fwd.cu",
    "fwd_cl_short_kernel": "ccv_fwd.cu",
    "fwd_cf_short_kernel": "ccv_fwd.cu",
    "fwd_cf_rows_kernel": "ccv_fwd.cu",
    "update_kernel": "ccv_update.cu",
    "spec_kernel": "ccv_update.cu",
    "paged_row_kernel": "paged_sconv.cu",
    "seq_metadata_kernel": "paged_sconv.cu",
}


def kernel_sources_sha(kernel: str) -> str:
    """Hash of the sources `kernel` is built from: its own .cu file and the
    shared device headers (the C header declares the ABI; no device code
    depends on it)."""
    from causal_depthwise_conv1d_fwd_gb300 import build as lib_build

    own = KERNEL_SOURCE[kernel]
    h = hashlib.sha256()
    for f in sorted(lib_build._inputs()):
        name = os.path.basename(f)
        if not (name == own or name.endswith(".cuh")):
            continue
        with open(f, "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from a committed ncu summary, if the
    summary was taken on the current kernel sources; else None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    if kernel not in KERNEL_SOURCE:
        return None
    sha = kernel_sources_sha(kernel)
    pat = re.compile(r"bench-traffic:\s*kernel=(\S+)\s+bytes_per_launch=(\d+)\s+"
                     r"source_sha=([0-9a-f]+)")
    for f in sorted(os.listdir(pdir)):
        if not f.endswith((".md", ".txt")):
            continue
        for m in pat.finditer(open(os.path.join(pdir, f)).read()):
            if m.group(1) == kernel and m.group(3) == sha:
                return int(m.group(2))
    return None


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# --------------------------------------------------------------- our arm ----

class Part:
    """One part of the step: `fn_on(handle)` enqueues its launches on the
    given stream handle, `fn()` on the stream current at set-up."""

    def __init__(self, name, kernel, launches, nbytes, tokens, fn_on, stream):
        self.name, self.kernel, self.launches = name, kernel, launches
        self.nbytes, self.tokens, self.fn_on = nbytes, tokens, fn_on
        self.stream = stream
        self.ms = 0.0

    def fn(self):
        self.fn_on(self.stream)


def make_parts(dev, rank):
    """The four parts of a step as pre-marshalled launches on the current stream,
    in step order: the two prefill layouts, then paged, then decode.  The
    parts share no buffer, so any order computes the same; the order sets
    which launch absorbs which predecessor's pending writes.  Over all six
    cyclic orders the step measured 191.6-201.2 us on one box: the two
    prefill launches side by side, then paged, then decode, is within 0.1 us
    of the fastest (decode before paged is the slowest)."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    seed_off = 100 * rank
    cases = {
        "prefill_tokens_dim": wl.config_large_prefill(1003 + seed_off, layout="tokens_dim"),
        "prefill_dim_tokens": wl.config_large_prefill(1003 + seed_off, layout="dim_tokens"),
        "decode": wl.config_decode(1002 + seed_off),
        "paged": wl.config_paged(1004 + seed_off),
    }
    stream = torch.cuda.current_stream().cuda_stream
    dev_args = {}
    parts = []
    for name in ("prefill_tokens_dim", "prefill_dim_tokens"):
        c = cases[name]
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16, device=dev)
        dev_args[name] = (d, out)
        launch = ccv.prepare_ccv_fwd(**d, out=out)
        parts.append(Part(name, "fwd_cl_async_kernel" if name.endswith("tokens_dim") else "fwd_cf_async_kernel",
                          1, prefill_bytes(c), prefill_tokens(c), launch, stream))
    c = cases["paged"]
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
    qsl = c.query_start_loc.to(dev)
    n_req = len(c.req_lengths)
    seq = torch.empty(c.T, dtype=torch.int32, device=dev)
    qs = torch.empty(c.T, dtype=torch.int32, device=dev)
    d["seq_idx"], d["query_start"] = seq, qs
    out = torch.empty_like(d["x"])
    dev_args["paged"] = (d, out)
    # One launch that resolves each token's request from query_start_loc and
    # writes the metadata out, instead of the metadata launch and the conv:
    # in this step order it ran the step 2.3 us faster (192.4 against
    # 194.7 us per step, same box).
    d1 = {k: v for k, v in d.items() if k not in ("seq_idx", "query_start")}
    paged = ccv.prepare_paged_sconv_fwd_with_metadata(
        query_start_loc=qsl, num_reqs=n_req, num_actual_tokens=c.num_actual_tokens,
        seq_idx_out=seq, query_start_out=qs, out=out, **d1)
    parts.append(Part("paged", "paged_row_kernel", 1, paged_bytes(c), c.T, paged, stream))
    c = cases["decode"]
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
    dev_args["decode"] = (d, d["x"])
    launch = ccv.prepare_ccv_update(**d)
    parts.append(Part("decode", "update_kernel", 1, decode_bytes(c), c.x.shape[0], launch, stream))
    return parts, cases, dev_args


def run_e2e(dev, cases, dev_args, steps):
    """The same step through the public API with host buffers: each step copies
    its inputs from pinned host memory and reads its outputs back, pipelined
    over a copy-in, a compute and a copy-out stream."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv

    stream = torch.cuda.current_stream()
    host_in, host_out, h2d, d2h = [], [], 0, 0

    def pinned_like(t):
        h = torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, pin_memory=True)
        return h

    plan = []
    for name in ("prefill_tokens_dim", "prefill_dim_tokens"):
        d, out = dev_args[name]
        hx = pinned_like(d["x"])
        hx.copy_(cases[name].x)
        ho = pinned_like(out)
        plan.append((name, d, out, hx, ho))
        h2d += hx.numel() * 2
        d2h += ho.numel() * 2
    d, out = dev_args["paged"]
    c = cases["paged"]
    hx = pinned_like(d["x"])
    hx.copy_(c.x)
    ho = pinned_like(out)
    hmeta = {k: getattr(c, k).pin_memory() for k in ("positions", "slot_mapping")}
    hq = c.query_start_loc.pin_memory()
    qsl_dev = torch.empty_like(hq, device=dev)
    plan.append(("paged", d, out, hx, ho))
    h2d += hx.numel() * 2 + sum(v.numel() * v.element_size() for v in hmeta.values()) + hq.numel() * 4
    d2h += ho.numel() * 2
    d, out = dev_args["decode"]
    hx = pinned_like(d["x"])
    hx.copy_(cases["decode"].x)
    ho = pinned_like(out)
    plan.append(("decode", d, out, hx, ho))
    h2d += hx.numel() * 2
    d2h += ho.numel() * 2

    # Copy-in streams, a compute stream and copy-out streams.  Part i's
    # copy-in waits until the previous step's compute and copy-out of part i
    # are done with its buffers; its compute waits for its copy-in and for the
    # previous copy-out of its output; its copy-out waits for its compute.
    # Copies in both directions and kernels of different parts overlap.
    # KCOPY > 1 splits each copy over that many streams per direction; on
    # GB300 that measured slower (the host link, not the copy engines, is the
    # limit), so one stream per direction is used.
    KCOPY = 1
    s_in = [torch.cuda.Stream() for _ in range(KCOPY)]
    s_out = [torch.cuda.Stream() for _ in range(KCOPY)]
    s_comp = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(KCOPY)] for _ in plan]
    ev_out = [[torch.cuda.Event() for _ in range(KCOPY)] for _ in plan]
    ev_done = [torch.cuda.Event() for _ in plan]

    def flat(t):
        # the host and device buffers share shape and strides and are dense,
        # so their storage can be copied as flat element ranges
        return t.as_strided((t.numel(),), (1,))

    def pieces(n):
        step = (n + KCOPY - 1) // KCOPY
        return [(k * step, min(n, (k + 1) * step)) for k in range(KCOPY)]

    def one_step():
        for i, (name, d, out, hx, ho) in enumerate(plan):
            src, dst = flat(hx), flat(d["x"])
            for k, (lo, hi) in enumerate(pieces(src.numel())):
                with torch.cuda.stream(s_in[k]):
                    s_in[k].wait_event(ev_done[i])
                    for e in ev_out[i]:
                        s_in[k].wait_event(e)
                    dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                    if name == "paged" and k == 0:
                        for key, v in hmeta.items():
                            d[key].copy_(v, non_blocking=True)
                        qsl_dev.copy_(hq, non_blocking=True)
                    ev_in[i][k].record(s_in[k])
            with torch.cuda.stream(s_comp):
                for e in ev_in[i] + ev_out[i]:
                    s_comp.wait_event(e)
                if name == "decode":
                    ccv.ccv_update(**d)
                elif name == "paged":
                    d1 = {k: v for k, v in d.items() if k not in ("seq_idx", "query_start")}
                    ccv.paged_sconv_fwd_with_metadata(
                        query_start_loc=qsl_dev, num_reqs=len(c.req_lengths),
                        num_actual_tokens=c.num_actual_tokens, seq_idx_out=d["seq_idx"],
                        query_start_out=d["query_start"], out=out, **d1)
                else:
                    ccv.ccv_fwd(**d, out=out)
                ev_done[i].record(s_comp)
            src, dst = flat(out), flat(ho)
            for k, (lo, hi) in enumerate(pieces(src.numel())):
                with torch.cuda.stream(s_out[k]):
                    s_out[k].wait_event(ev_done[i])
                    dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                    ev_out[i][k].record(s_out[k])

    all_streams = s_in + [s_comp] + s_out

    def join():
        for st in all_streams:
            stream.wait_stream(st)

    for st in all_streams:
        st.wait_stream(stream)
    for _ in range(3):
        one_step()
    join()
    torch.cuda.synchronize()
    # Three timed windows of `steps` steps each; the median window is the
    # result (single windows varied by up to 12% from run to run).
    windows = []
    for _ in range(3):
        barrier(dev)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for st in all_streams:
            st.wait_stream(stream)
        for _ in range(steps):
            one_step()
        join()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(dev)
        windows.append(start.elapsed_time(end) / 1e3)
    return sorted(windows)[1], h2d, d2h, windows


GRAPH_CALLS = 20  # calls captured per graph, so replay measures the GPU, not the host launch


def graph_us_per_call(launch, replays=50):
    """Warm (L2-resident) CUDA-graph replay: GRAPH_CALLS launches of `launch`
    captured in one graph, us per call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        launch(s.cuda_stream)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream().cuda_stream
        for _ in range(GRAPH_CALLS):
            launch(cs)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (replays * GRAPH_CALLS)


def decode_graph_us(dev_args):
    """Warm CUDA-graph replay of the decode call, us per call."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv

    d, _ = dev_args["decode"]
    launch = ccv.prepare_ccv_update(**d)
    return graph_us_per_call(lambda st: launch(st))


class L2Flush:
    """Leaves L2 holding only clean, unrelated lines: a write of a buffer
    larger than L2 evicts everything, then a read of a second such buffer
    evicts the dirty lines the write left (so the next kernel does not pay
    for their write-back)."""

    def __init__(self, dev, nbytes=256 << 20):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def spec_verify_timing(dev, rank, calls=100):
    """The speculative-verify update (not part of the step): us per call
    L2-cold (L2Flush between calls, outside the timed window) and as warm
    CUDA-graph replay."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    c = wl.config_spec_decode(1005 + 100 * rank)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
    src = c.intermediate_conv_window
    inter = torch.empty_strided(src.shape, src.stride(), dtype=src.dtype, device=dev)
    inter.copy_(src)
    d["intermediate_conv_window"] = inter
    launch = ccv.prepare_ccv_update_spec(**d)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    for _ in range(3):
        launch(stream.cuda_stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(calls)]
    for a, b in evs:
        flush()
        a.record()
        launch(stream.cuda_stream)
        b.record()
    torch.cuda.synchronize()
    # mean, not median: single event pairs resolve only about 2 us here, and
    # the mean of many quantised readings is unbiased
    cold = sum(a.elapsed_time(b) * 1e3 for a, b in evs) / calls
    warm = graph_us_per_call(lambda st: launch(st))
    nbytes = spec_bytes(c)
    return {"workload": c.name, "kernel": "spec_kernel", "bytes": nbytes,
            "us_l2_cold": round(cold, 2), "gbs_l2_cold": round(nbytes / (cold * 1e-6) / 1e9, 1),
            "us_graph_warm": round(warm, 2)}


def atrex_shapes_timing(dev, calls=100):
    """The nine atrex-bench #003 shapes (one channel-first sequence, not part
    of the step): us per call L2-cold (L2Flush between calls, outside the
    timed window) and algorithmic GB/s."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    rows = []
    for tokens, dim in wl.ATREX_SHAPES:
        c = wl.config_atrex(tokens, dim)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16, device=dev)
        launch = ccv.prepare_ccv_fwd(**d, out=out)
        for _ in range(3):
            launch(stream.cuda_stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(calls)]
        for a, b in evs:
            flush()
            a.record()
            launch(stream.cuda_stream)
            b.record()
        torch.cuda.synchronize()
        us = sum(a.elapsed_time(b) * 1e3 for a, b in evs) / calls  # mean, see above
        nbytes = prefill_bytes(c)
        rows.append({"tokens": tokens, "dim": dim, "us_l2_cold": round(us, 2),
                     "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "bytes": nbytes})
        del d, out, launch
    return rows


def paged_streams_timing(dev, calls=100):
    """A layer's four conv streams on one paged cache (not part of the step):
    one fused launch vs one paged_sconv_fwd per stream, us per call L2-cold
    (L2Flush between calls, outside the timed window), mean of many calls."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    base, streams = wl.config_paged_streams()
    cache = base.cache.to(dev)
    meta = {k: getattr(base, k).to(dev) for k in
            ("positions", "block_table", "seq_idx", "slot_mapping", "query_start")}
    ds = [{"x": st["x"].to(dev), "weight": st["weight"].to(dev), "off_s": st["off_s"],
           "ws": st["ws"]} for st in streams]
    fused = ccv.prepare_paged_sconv_fwd_streams(ds, cache, block_size=base.block_size,
                                                activation="silu", use_residual=True, **meta)
    single = [ccv.prepare_paged_sconv_fwd(st["x"], st["weight"], cache, off_s=st["off_s"],
                                          ws=st["ws"], block_size=base.block_size,
                                          activation="silu", use_residual=True, **meta)
              for st in ds]
    stream = torch.cuda.current_stream().cuda_stream
    flush = L2Flush(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(calls)]
        for a, b in evs:
            flush()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) * 1e3 for a, b in evs) / calls

    us_fused = timed(lambda: fused(stream))
    us_sep = timed(lambda: [launch(stream) for launch in single])
    # every stream has the base case's channel count and token metadata
    nbytes = len(streams) * _paged_bytes(base)
    return {"workload": base.name, "kernel": "paged_row_kernel", "streams": len(streams),
            "bytes": nbytes, "us_fused_l2_cold": round(us_fused, 2),
            "us_separate_l2_cold": round(us_sep, 2),
            "gbs_fused": round(nbytes / (us_fused * 1e-6) / 1e9, 1)}


def paged_single_launch_timing(dev, calls=100):
    """The paged workload as one paged_sconv_fwd_with_metadata launch (the
    metadata resolved in the conv kernel) against paged_sconv_seq_metadata +
    paged_sconv_fwd: us per call L2-cold (L2Flush between calls, outside the
    timed window), mean of many calls."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    c = wl.config_paged()
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
    qsl = c.query_start_loc.to(dev)
    seq = torch.empty(c.T, dtype=torch.int32, device=dev)
    qs = torch.empty(c.T, dtype=torch.int32, device=dev)
    d["seq_idx"], d["query_start"] = seq, qs
    n_req = len(c.req_lengths)
    meta = ccv.prepare_paged_sconv_seq_metadata(qsl, n_req, c.num_actual_tokens, seq, qs, c.T)
    conv = ccv.prepare_paged_sconv_fwd(**d)
    d1 = {k: v for k, v in d.items() if k not in ("seq_idx", "query_start")}
    single = ccv.prepare_paged_sconv_fwd_with_metadata(
        query_start_loc=qsl, num_reqs=n_req, num_actual_tokens=c.num_actual_tokens,
        seq_idx_out=seq, query_start_out=qs, **d1)
    stream = torch.cuda.current_stream().cuda_stream
    flush = L2Flush(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(calls)]
        for a, b in evs:
            flush()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) * 1e3 for a, b in evs) / calls

    us_two = timed(lambda: (meta(stream), conv(stream)))
    us_one = timed(lambda: single(stream))
    nbytes = paged_bytes(c)
    return {"workload": c.name, "bytes": nbytes, "us_metadata_then_conv_l2_cold": round(us_two, 2),
            "us_single_launch_l2_cold": round(us_one, 2),
            "gbs_single_launch": round(nbytes / (us_one * 1e-6) / 1e9, 1)}


def width_variants_timing(dev, calls=20):
    """The large prefill in both layouts for every width 2..5, with bias and
    SiLU and without either (not part of the step).  Inputs are larger than
    L2, so calls run back to back; us per call is the mean of many calls."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    stream = torch.cuda.current_stream().cuda_stream
    rows = []
    for layout in ("tokens_dim", "dim_tokens"):
        c = wl.config_large_prefill(layout=layout)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16, device=dev)
        g = torch.Generator().manual_seed(1008)
        for width in (2, 3, 4, 5):
            w = (torch.randn(c.dim, width, generator=g) * 0.02).to(torch.bfloat16).to(dev)
            states = d["conv_states"]
            if states.shape[2] < width - 1:  # W = 5 needs a fourth state column
                states = wl.make_states(states.shape[0], c.dim, width - 1, "dim_contiguous",
                                        g).to(dev)
            for plain in (False, True):
                dd = dict(d, weight=w, conv_states=states, bias=None if plain else d["bias"],
                          activation=None if plain else "silu")
                launch = ccv.prepare_ccv_fwd(**dd, out=out)
                for _ in range(3):
                    launch(stream)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(calls):
                    launch(stream)
                b.record()
                torch.cuda.synchronize()
                us = a.elapsed_time(b) * 1e3 / calls
                case = wl.PrefillCase(c.name, c.x, torch.empty(c.dim, width, dtype=torch.bfloat16),
                                      None if plain else c.bias, c.conv_states,
                                      c.query_start_loc, c.cache_indices, c.has_initial_state,
                                      None if plain else "silu", lengths=c.lengths)
                nbytes = prefill_bytes(case)
                rows.append({"layout": layout, "width": width,
                             "bias_silu": not plain, "us": round(us, 2),
                             "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)})
        del d, out
    return rows


SHORT_SEQUENCE_MIXES = ((64, 1024), (256, 256), (16, 2048))


def short_sequences_timing(dev, calls=20):
    """Many short sequences at dim 8192, width 4, bias and SiLU, in both
    layouts (not part of the step): channel-first takes the multi-row kernel
    here.  Inputs are larger than L2, so calls run back to back; us per call
    is the mean of `calls` calls."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    stream = torch.cuda.current_stream().cuda_stream
    rows = []
    for batch, tokens in SHORT_SEQUENCE_MIXES:
        for layout in ("tokens_dim", "dim_tokens"):
            c = wl.varlen_prefill(1010, [tokens] * batch, 8192, 4, layout=layout, has_init="all")
            d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
            out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16,
                                      device=dev)
            launch = ccv.prepare_ccv_fwd(**d, out=out)
            for _ in range(3):
                launch(stream)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(calls):
                launch(stream)
            b.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / calls
            nbytes = prefill_bytes(c)
            rows.append({"sequences": batch, "tokens_each": tokens, "layout": layout,
                         "us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)})
            del d, out, launch
        torch.cuda.empty_cache()
    return rows


def small_configs_timing(dev, calls=100):
    """The single-sequence (dim 64, 16 tokens) and varlen continuous-batching
    (8 sequences, dim 4096) prefill configurations, not part of the step: us
    per call L2-cold (L2Flush between calls, outside the timed window), mean
    of many calls."""
    import causal_depthwise_conv1d_fwd_gb300 as ccv
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    stream = torch.cuda.current_stream().cuda_stream
    flush = L2Flush(dev)
    rows = []
    for c in (wl.config_single(), wl.config_varlen()):
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16, device=dev)
        launch = ccv.prepare_ccv_fwd(**d, out=out)
        for _ in range(3):
            launch(stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(calls)]
        for a, b in evs:
            flush()
            a.record()
            launch(stream)
            b.record()
        torch.cuda.synchronize()
        us = sum(a.elapsed_time(b) * 1e3 for a, b in evs) / calls
        nbytes = prefill_bytes(c)
        rows.append({"workload": c.name, "tokens": prefill_tokens(c), "us_l2_cold": round(us, 2),
                     "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "bytes": nbytes})
    return rows


def time_parts(parts, steps, stream):
    """K steps with an event between parts: adds each part's time to p.ms and
    returns the seconds of the whole loop."""
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)]
              for _ in range(steps)]
    torch.cuda.synchronize()
    for s in range(steps):
        ev = events[s]
        ev[0].record(stream)
        for i, p in enumerate(parts):
            p.fn()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    for s in range(steps):
        for i, p in enumerate(parts):
            p.ms += events[s][i].elapsed_time(events[s][i + 1])
    return events[0][0].elapsed_time(events[-1][-1]) / 1e3


def graph_step_timing(parts, steps):
    """The step captured as one CUDA graph and replayed K times: ms per step,
    and each part's us per call from timing events recorded inside the graph
    (where this torch records events as graph nodes; their nodes also
    serialise the launches around them, so the part figures add up to more
    than the event-free step)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()

    def capture(with_events):
        g = torch.cuda.CUDAGraph()
        evs = None
        with torch.cuda.graph(g, stream=s):
            if with_events:
                evs = [torch.cuda.Event(enable_timing=True, external=True)
                       for _ in range(len(parts) + 1)]
                evs[0].record()
            for i, p in enumerate(parts):
                p.fn_on(torch.cuda.current_stream().cuda_stream)
                if with_events:
                    evs[i + 1].record()
        return g, evs

    def replay(g, n):
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    g, _ = capture(False)
    out = {"ms_per_step": round(replay(g, steps), 4)}
    del g
    try:
        g, evs = capture(True)
    except TypeError:  # this torch cannot record timing events as graph nodes
        return out
    n = min(steps, 200)
    per = [0.0] * len(parts)
    for _ in range(n):
        g.replay()
        torch.cuda.synchronize()
        for i in range(len(parts)):
            per[i] += evs[i].elapsed_time(evs[i + 1])
    out["parts_us"] = {p.name: round(per[i] * 1e3 / n, 2) for i, p in enumerate(parts)}
    return out


def host_link_peak(dev, nbytes=1 << 30, reps=5):
    """Plain copies between pinned host memory and the device, best of
    `reps`: one `nbytes` buffer host->device, device->host, and both at once
    on two streams.  GB/s of bytes moved (both directions for the last)."""
    h_in = torch.ones(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.ones(nbytes, dtype=torch.uint8, device=dev)
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(h2d, d2h):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            s_in.wait_stream(cur)
            s_out.wait_stream(cur)
            if h2d:
                with torch.cuda.stream(s_in):
                    d_in.copy_(h_in, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    h_out.copy_(d_out, non_blocking=True)
            cur.wait_stream(s_in)
            cur.wait_stream(s_out)
            b.record(cur)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) / 1e3)
        return (int(h2d) + int(d2h)) * nbytes / best / 1e9

    out = {"h2d_gbs": round(timed(True, False), 1), "d2h_gbs": round(timed(False, True), 1),
           "both_gbs": round(timed(True, True), 1), "buffer_bytes": nbytes}
    del h_in, h_out, d_in, d_out
    return out


def back_to_back_us(part, calls=50):
    """us per call of `calls` launches of one part back to back (events
    around the whole loop), so each launch may overlap the previous one's
    tail.  Meaningful L2-cold only for parts whose data exceed L2."""
    for _ in range(3):
        part.fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    a.record(stream)
    for _ in range(calls):
        part.fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / calls


def launch_floor_us(dev, calls=100):
    """The cost of any launch as the parts and the extras are timed: a
    one-element torch kernel, us per call one at a time after an L2 flush
    (events around each call, the flush outside them), and back to back from
    a CUDA graph of `calls` such launches (so the host's launch cost does not
    count), means of many calls."""
    tiny = torch.zeros(1, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    for _ in range(10):
        tiny.add_(1.0)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(calls)]
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        tiny.add_(1.0)
        e1.record(stream)
    torch.cuda.synchronize()
    single = sum(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs) / calls
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(calls):
            tiny.add_(1.0)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(10):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    graphed = a.elapsed_time(b) * 1e3 / (10 * calls)
    return {"single_after_flush": round(single, 2), "back_to_back_graph": round(graphed, 2),
            "kernel": "one-element torch add"}


def copy_same_size_timing(x, calls=50):
    """A torch copy of the prefill input into a second buffer of the same
    size (the same bytes read and written as a prefill launch moves, minus
    the states and weights): us per copy back to back, and one at a time
    with events around each copy as the parts loop times its parts.  Both
    L2-cold: the two buffers exceed L2."""
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        y.copy_(x)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(calls):
        y.copy_(x)
    b.record(stream)
    torch.cuda.synchronize()
    b2b = a.elapsed_time(b) * 1e3 / calls
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(calls)]
    for e0, e1 in evs:
        e0.record(stream)
        y.copy_(x)
        e1.record(stream)
    torch.cuda.synchronize()
    single = sum(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs) / calls
    nbytes = 2 * x.numel() * x.element_size()
    del y
    return {"bytes": nbytes, "us_back_to_back": round(b2b, 2),
            "gbs_back_to_back": round(nbytes / (b2b * 1e-6) / 1e9, 1),
            "us_event_bracketed": round(single, 2),
            "gbs_event_bracketed": round(nbytes / (single * 1e-6) / 1e9, 1)}


def marginal_timing(parts, steps, stream):
    """What each part adds to the headline loop: the loop of K steps with every
    part, and with each part left out in turn (the rest in step order, nothing
    between the launches), timed with events around each loop.  A part's
    marginal time is the step's time minus the time without it, so it counts
    only what does not overlap its neighbours' launches and tails."""
    def loop_us(keep):
        for _ in range(5):
            for p in keep:
                p.fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            for p in keep:
                p.fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / steps

    full = loop_us(parts)
    out = {}
    for p in parts:
        out[p.name] = round(full - loop_us([q for q in parts if q is not p]), 2)
    full_again = loop_us(parts)
    return {"step_us": round((full + full_again) / 2, 2), "marginal_us": out,
            "steps": steps}


def concurrent_streams_timing(parts, steps):
    """The step's parts on two streams at once: the prefill parts on one,
    decode and paged on another (they share no buffer), as an engine would
    overlap a prefill batch with a decode batch.  Each stream keeps its own
    parts in step order; the two are joined at the end.  ms per step and
    algorithmic GB/s of the step (not the headline, which runs the parts one
    after another)."""
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    pre = [p for p in parts if p.name.startswith("prefill")]
    rest = [p for p in parts if not p.name.startswith("prefill")]

    def run(n):
        side.wait_stream(main)
        for _ in range(n):
            for p in pre:
                p.fn_on(main.cuda_stream)
            for p in rest:
                p.fn_on(side.cuda_stream)
        main.wait_stream(side)

    run(5)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    run(steps)
    b.record(main)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nbytes = sum(p.nbytes for p in parts)
    return {"ms_per_step": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "streams": "prefill parts on one stream, decode and paged on another"}


def run_ours(args):
    import causal_depthwise_conv1d_fwd_gb300 as ccv  # noqa: F401
    from causal_depthwise_conv1d_fwd_gb300 import _lib

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    _lib.load()
    parts, cases, dev_args = make_parts(dev, rank)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        for p in parts:
            p.fn()
    torch.cuda.synchronize()

    # The headline: K steps back to back with nothing between the launches,
    # so each kernel's launch may overlap the previous one's tail (every
    # kernel of the library is launched with programmatic serialization).
    sampler = ClockSampler(dev)
    if rank == 0:
        sampler.start()
    barrier(dev)
    torch.cuda.synchronize()
    sampler.mark("start")
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        for p in parts:
            p.fn()
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark("end")
    barrier(dev)
    seconds = t_start.elapsed_time(t_end) / 1e3
    clocks = sampler.stop() if rank == 0 else None
    max_seconds = max_over_ranks(seconds, dev)

    # The parts: the same K steps again with an event between parts (an
    # event between two launches also serialises them).
    parts_s = time_parts(parts, args.steps, stream)
    graph = graph_step_timing(parts, args.steps)
    b2b = {p.name: back_to_back_us(p) for p in parts if p.name.startswith("prefill")}
    concurrent = concurrent_streams_timing(parts, args.steps)
    marginal = marginal_timing(parts, min(args.steps, 2000), stream)

    step_bytes = sum(p.nbytes for p in parts)
    value = whole_job_rate(step_bytes, args.steps, world, max_seconds) / 1e9
    pre = [p for p in parts if p.name.startswith("prefill")]
    pre_s = sum(p.ms for p in pre) / 1e3
    mtok = whole_job_rate(sum(p.tokens for p in pre), args.steps, world,
                          max_over_ranks(pre_s, dev)) / 1e6
    dominant = max(parts, key=lambda p: p.ms)
    peak, peak_kind = measured_peak_hbm()
    dom_us = dominant.ms * 1e3 / (args.steps * dominant.launches)
    achieved = dominant.nbytes / dominant.launches / (dom_us * 1e-6) / 1e9
    traffic = recorded_traffic(dominant.kernel)

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    e2e_s, h2d, d2h, e2e_windows = run_e2e(dev, cases, dev_args, e2e_steps)
    e2e_s = max_over_ranks(e2e_s, dev)
    e2e_value = whole_job_rate(step_bytes, e2e_steps, world, e2e_s) / 1e9
    link = host_link_peak(dev)
    link_gbs = (h2d + d2h) * e2e_steps / e2e_s / 1e9
    graph_us = decode_graph_us(dev_args)
    spec = spec_verify_timing(dev, rank)
    atrex = atrex_shapes_timing(dev)
    paged_streams = paged_streams_timing(dev)
    paged_single = paged_single_launch_timing(dev)
    widths = width_variants_timing(dev)
    short_seqs = short_sequences_timing(dev)
    small = small_configs_timing(dev)
    floor = launch_floor_us(dev)
    copy_ref = copy_same_size_timing(dev_args["prefill_tokens_dim"][0]["x"])

    if rank != 0:
        return
    cpu = cpu_baseline(cases, budget_s=args.cpu_seconds) if world == 1 else None
    cpu_all = cpu_baseline_all_cores(cases, budget_s=min(5.0, args.cpu_seconds)) if world == 1 else None
    parts_out = {}
    for p in parts:
        us = p.ms * 1e3 / args.steps
        # What one launch moving these bytes at the copy rate would take when
        # timed the same way: the launch floor plus bytes / peak.
        ref_us = floor["single_after_flush"] + p.nbytes / (peak * 1e3)
        entry = {"kernel": p.kernel, "us": round(us, 2), "bytes": p.nbytes,
                 "gbs": round(p.nbytes / (us * 1e-6) / 1e9, 1),
                 "frac_of_peak": round(p.nbytes / (us * 1e-6) / 1e9 / peak, 4),
                 "launch_floor_plus_copy_us": round(ref_us, 2),
                 "frac_of_launch_floor_plus_copy": round(ref_us / us, 4)}
        if p.name.startswith("prefill"):
            entry["mtok_s"] = round(p.tokens / (us * 1e-6) / 1e6, 1)
            # launches of this part alone, back to back (inputs exceed L2)
            entry["us_back_to_back"] = round(b2b[p.name], 2)
            entry["gbs_back_to_back"] = round(p.nbytes / (b2b[p.name] * 1e-6) / 1e9, 1)
            # against a torch copy of x (same size), each timed the same way
            entry["frac_of_same_size_copy_back_to_back"] = round(copy_ref["us_back_to_back"] / b2b[p.name], 4)
            entry["frac_of_same_size_copy_event_bracketed"] = round(copy_ref["us_event_bracketed"] / us, 4)
        if p.name == "decode":
            entry["us_per_call_l2_cold"] = round(us, 2)
            entry["us_per_call_graph_warm"] = round(graph_us, 2)
        if "parts_us" in graph:
            entry["us_in_graph_step"] = graph["parts_us"][p.name]
        parts_out[p.name] = entry
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_seconds * 1e3 / args.steps, 4),
        "graph_step": graph,
        "concurrent_step": concurrent,
        "parts_loop_ms_per_step": round(parts_s * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "width": 4, "dim": 8192, "storage": "bf16",
                   "prefill_tokens": sum(p.tokens for p in pre) // 2,
                   "bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2: each step streams 1.07 GB of prefill traffic, "
                         "so every part starts L2-cold; no explicit flush",
                   "parallelism": f"{world} independent replica(s), no collective"},
        "mtok_per_s_prefill": round(mtok, 1),
        "decode_us_per_call": parts_out["decode"]["us_per_call_l2_cold"],
        "decode_us_per_call_graph_warm": round(graph_us, 2),
        "spec_verify": spec,
        "atrex_shapes": atrex,
        "paged_streams": paged_streams,
        "paged_single_launch": paged_single,
        "width_variants": widths,
        "short_sequences": short_seqs,
        "marginal_in_step": marginal,
        "small_configs": small,
        "launch_floor_us": floor,
        "copy_same_size": copy_ref,
        "parts": parts_out,
        "roofline": {"bound": "hbm", "kernel": dominant.kernel, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": dominant.nbytes // dominant.launches,
                     "avg_launch_us": round(dom_us, 2)},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "steps": e2e_steps,
                "windows": 3, "window_gbs": [round(step_bytes * e2e_steps / w / 1e9, 1)
                                              for w in e2e_windows],
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "link_gbs": round(link_gbs, 1), "link_peak_gbs": link["both_gbs"],
                "frac_of_link": round(link_gbs / link["both_gbs"], 4), "link_peak": link},
        "gpu_launches": sum(p.launches for p in parts) * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
    }
    print(json.dumps(line))


# ------------------------------------------------------ CPU / reference ----

def _channel_slice_prefill(case, c):
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    return wl.PrefillCase(case.name, case.x[:c], case.weight[:c],
                          None if case.bias is None else case.bias[:c],
                          None if case.conv_states is None else case.conv_states[:, :c].clone(),
                          case.query_start_loc, case.cache_indices, case.has_initial_state,
                          case.activation, case.pad_slot_id, case.lengths)


def oracle_sample_step(cases, frac):
    """Run the oracle once over a `frac` channel sample of every part of the
    step; return (bytes of the sample, seconds)."""
    import oracle
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    total_bytes, total_s = 0, 0.0
    for name in ("prefill_tokens_dim", "prefill_dim_tokens"):
        c = cases[name]
        nc = max(1, int(round(c.dim * frac)))
        s = _channel_slice_prefill(c, nc)
        out = torch.empty_strided(s.x.shape, s.x.stride(), dtype=torch.bfloat16)
        t0 = time.perf_counter()
        oracle.ccv_fwd(s.x, s.weight, s.bias, s.conv_states, s.query_start_loc, s.cache_indices,
                       s.has_initial_state, s.activation, s.pad_slot_id, out=out)
        total_s += time.perf_counter() - t0
        total_bytes += prefill_bytes(s)
    c = cases["decode"]
    nc = max(1, int(round(c.x.shape[1] * frac)))
    x = c.x[:, :nc].clone()
    st = c.conv_state[:, :nc].clone()
    t0 = time.perf_counter()
    oracle.ccv_update(x, st, c.weight[:nc], c.bias[:nc], c.activation, c.conv_state_indices,
                      c.pad_slot_id)
    total_s += time.perf_counter() - t0
    total_bytes += decode_bytes(wl.DecodeCase(c.name, x, c.weight[:nc], c.bias[:nc], st,
                                              c.conv_state_indices, c.activation))
    c = cases["paged"]
    H = c.cache.shape[1]
    C_full = c.x.shape[1]
    W = c.weight.shape[1]
    c_sub = max(1, int(round(C_full * frac)))
    if c_sub >= c.ws:
        nh, ws_sub = min(H, -(-c_sub // c.ws)), c.ws
    else:
        nh, ws_sub = 1, c_sub
    C = nh * ws_sub
    x = c.x.view(c.T, H, c.ws)[:, :nh, :ws_sub].reshape(c.T, C).contiguous()
    w = c.weight.view(H, c.ws, W)[:nh, :ws_sub].reshape(C, W).contiguous()
    cache = c.cache[:, :nh].clone()
    seq = torch.empty(c.T, dtype=torch.int32)
    qs = torch.empty(c.T, dtype=torch.int32)
    t0 = time.perf_counter()
    oracle.paged_sconv_seq_metadata(c.query_start_loc, len(c.req_lengths), c.num_actual_tokens,
                                    seq, qs, c.T)
    oracle.paged_sconv_fwd(x, w, cache, c.positions, c.block_table, seq, c.slot_mapping, qs,
                           c.off_s, ws_sub, c.block_size, c.activation, c.use_residual)
    total_s += time.perf_counter() - t0
    total_bytes += int(paged_bytes(c) * C / C_full)
    return total_bytes, total_s


def cpu_baseline(cases, budget_s=15.0):
    """The oracle, single-threaded, on a channel sample sized to ~budget_s."""
    b, s = oracle_sample_step(cases, 1.0 / 512)
    frac = min(1.0, (1.0 / 512) * max(1.0, budget_s / max(s, 1e-6)))
    b, s = oracle_sample_step(cases, frac)
    return {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{frac:.4f} of the channels of every part of one step "
                      f"({b / 1e6:.1f} MB algorithmic, {s:.1f} s), single-threaded C oracle"}


def cpu_baseline_all_cores(cases, budget_s=5.0):
    """The same oracle on every host core: one thread per core, each running a
    channel sample of the step on its own copies (the C calls release the
    interpreter lock, and each writes only buffers it owns)."""
    import concurrent.futures

    n = len(os.sched_getaffinity(0))
    _, s1 = oracle_sample_step(cases, 1.0 / 512)
    frac = min(1.0, (1.0 / 512) * max(1.0, budget_s / max(s1, 1e-6)))
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(n) as ex:
        res = list(ex.map(lambda _: oracle_sample_step(cases, frac), range(n)))
    wall = time.perf_counter() - t0
    nbytes = sum(b for b, _ in res)
    return {"value": round(nbytes / wall / 1e9, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{n} threads, each {frac:.4f} of the channels of every part of one step "
                      f"({nbytes / 1e6:.1f} MB algorithmic in {wall:.1f} s wall)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

    cases = {
        "prefill_tokens_dim": wl.config_large_prefill(1003, layout="tokens_dim"),
        "prefill_dim_tokens": wl.config_large_prefill(1003, layout="dim_tokens"),
        "decode": wl.config_decode(1002),
        "paged": wl.config_paged(1004),
    }
    # size one step so that warmup + steps take about args.ref_seconds in total
    b, s = oracle_sample_step(cases, 1.0 / 2048)
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    frac = min(1.0, (1.0 / 2048) * max(0.05, per_step / max(s, 1e-6)))
    for _ in range(args.warmup):
        oracle_sample_step(cases, frac)
    tb, ts = 0, 0.0
    for _ in range(args.steps):
        b, s = oracle_sample_step(cases, frac)
        tb += b
        ts += s
    value = tb / ts / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ts * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "width": 4, "dim": 8192, "storage": "bf16",
                   "sample": f"{frac:.5f} of the channels of every part per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{frac:.5f} of the channels of every part per step, "
                                   "single-threaded C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
