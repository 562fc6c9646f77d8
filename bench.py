"""Benchmark of the MLA latent-cache decode step on GB300.

One step = the cache-write of this step's new row (row end_pos-1 of every
sequence) followed by the absorbed decode over positions 0..end_pos-1, in one
call (mla_decode_append; the sparse workload: mla_decode_sparse with its new
rows; multi-token workloads: their new rows appended, then mla_decode_mtp).  Inputs are
seeded synthetic tensors of the workload's shapes, resident in HBM before the
timed region.  The timed region is one CUDA-graph launch holding exactly K
steps; successive steps rotate over cache copies (or top-k lists) so that each
step's working set is not served from L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..8]
    python bench.py --impl reference ...     # the CPU oracle, same metric

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica on its own GPU (independent sequences, no data-path collective);
the timing is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_latent_kv_07_gb300 as mla  # noqa: E402
from mla_latent_kv_07_gb300 import inputs, layout  # noqa: E402

# the long-context FP8 decode: the largest configuration and the one whose
# target is a fraction of the HBM bandwidth
DEFAULT_WORKLOAD = 4
SOAK_SECONDS = 3.0     # graph replays under load before the timed steps (clock samples)
CEILING_BYTES = 2 << 30  # one buffer far larger than L2 for the streaming-read ceiling
METRIC = "MLA decode: cache HBM TB/s (algorithmic cache bytes / step time)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers

def peaks(path: str | None = None):
    """Roofline denominators: each one the measured figure from
    MEASURED_PEAKS.json when the file gives it (a number, or an object with a
    "value"), else the fallback.  Returns (peaks, "measured" | "fallback" |
    "measured and fallback")."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
    except (OSError, ValueError):
        p = {}
    out, got = {}, set()
    for k, fb in FALLBACK_PEAKS.items():
        v = p.get(k) if isinstance(p, dict) else None
        if isinstance(v, dict):
            v = v.get("value")
        try:
            v = float(v)
        except (TypeError, ValueError):
            v = None
        if v is not None and v > 0 and math.isfinite(v):
            out[k] = v
            got.add(k)
        else:
            out[k] = fb
    src = "measured" if len(got) == len(FALLBACK_PEAKS) else ("fallback" if not got else "measured and fallback")
    return out, src


def decode_path(H: int) -> str:
    """Which decode kernel the library runs for H heads (mirrors its choice)."""
    if H == 128 and os.environ.get("MLA_DECODE_PATH", "") != "mma":
        return "decode_tc_kernel"
    return "decode_mma_kernel"


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    src = "decode_tc.cu" if kernel == "decode_tc_kernel" else "decode_mma.cu"
    for name in (src, "common.cuh", "tc_ptx.cuh", "append_row.cuh", "schedule.cuh"):
        with open(os.path.join(ROOT, "mla_latent_kv_07_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_kernel_traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = re.search(r"^kernel_source_sha256_16:\s*(\S+)", text, re.M)
    if not src or src.group(1) != kernel_source_hash(kernel):
        return None
    m = re.search(rf"^{re.escape(workload)}:\s*([0-9.eE+]+)", text, re.M)
    return float(m.group(1)) if m else None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 20 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for ln in out.strip().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:   # timestamp + the 9 queried fields
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10], parts[5]))
            except (ValueError, IndexError):
                continue
        window = [r for r in rows if self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        where = "load soak + timed region"
        if not window:
            window, where = rows, "around the timed region (region shorter than the sampling period)"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in window for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in window), "sm_max_mhz": max(r[2] for r in window),
                "reasons": reasons, "samples": len(window), "window": where}


def slowest(ms: float, device) -> float:
    """Largest time over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, slowest_s: float) -> float:
    """Units all ranks processed / the slowest rank's time (weak scaling)."""
    return world * units_per_rank / slowest_s


# ------------------------------------------------------------ workload set-up

class Setup:
    """Device-resident inputs of one workload, with rotation for L2."""

    def __init__(self, w: inputs.Workload, device, seed_offset: int = 0):
        self.w = w
        self.device = device
        g = lambda shape, tid: inputs.randn_bf16(shape, 1000 * w.index + tid + seed_offset, device)
        self.ends = inputs.end_positions(w).to(device)
        self.ends_host = self.ends.cpu().tolist()
        self.tokens = sum(min(t, w.topk) if w.topk else t for t in self.ends_host)
        lead = (w.B, w.H) if w.mtp == 1 else (w.B, w.mtp, w.H)
        self.ql, self.qp = g(lead + (512,), inputs.T_QL), g(lead + (64,), inputs.T_QP)
        self.kv_new, self.pe_new = g((w.B, 512), inputs.T_KVNEW), g((w.B, 64), inputs.T_PENEW)
        step_bytes = layout.step_bytes(self.tokens, w.B, w.H, w.fmt)
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.rot = max(1, math.ceil(2 * l2 / step_bytes))
        base = self._make_cache(g)
        if w.topk:
            # rotate the top-k lists (different gathered rows each step), one cache
            self.caches = [base]
            self.topks = [inputs.topk_indices(w.B, w.topk, self.ends_host,
                                              1000 * w.index + inputs.T_TOPK + 17 * r).to(device)
                          for r in range(self.rot)]
            self.rotation = f"{self.rot} top-k lists ({self.rot * step_bytes / 1e6:.0f} MB gathered)"
        else:
            self.caches = [base] + [self._clone(base) for _ in range(self.rot - 1)]
            self.topks = None
            self.rotation = f"{self.rot} cache copies ({self.rot * step_bytes / 1e6:.0f} MB read)"
        self.l2_bytes = l2
        self.out = torch.empty(lead + (512,), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(lead, dtype=torch.float32, device=device)
        self.ws = mla.alloc_workspace(w.B * w.mtp, w.H, w.S, w.topk, device)
        if w.absorb:
            self.q_nope, self.wkv_b = (t.to(device) for t in inputs.absorb_inputs(w))
            self.o = torch.empty((w.B, w.H, 128), dtype=torch.bfloat16, device=device)
        # the step's new rows: positions end_pos - mtp .. end_pos - 1 (a prefill
        # chunk's rows are taken as already written)
        self.start_pos = ([] if w.mtp > PREFILL_MTP else
                          [[t - w.mtp + j for t in self.ends_host] for j in range(w.mtp)])

    def _make_cache(self, g):
        w = self.w
        kv = g((w.B, w.S, 512), inputs.T_KV)
        pe = g((w.B, w.S, 64), inputs.T_PE)
        if w.fmt == 0:
            return mla.Cache(w.B, w.S, 0, kv=kv, pe=pe, device=self.device)
        cache = mla.Cache(w.B, w.S, 1, pe=pe, device=self.device)
        # quantise every row with the library's cache-write kernel: view the
        # [B, S] rows as B*S one-row slots and append them in chunks
        flat = mla.Cache(w.B * w.S, 1, 1, kv=cache.kv.view(w.B * w.S, 1, 512),
                         kv_scale=cache.kv_scale.view(w.B * w.S, 1, 4),
                         pe=cache.pe.view(w.B * w.S, 1, 64))
        rows = kv.view(w.B * w.S, 512)
        pe_rows = pe.view(w.B * w.S, 64)
        zeros = [0] * 2048
        for r0 in range(0, w.B * w.S, 2048):
            n = min(2048, w.B * w.S - r0)
            sub = mla.Cache(n, 1, 1, kv=flat.kv[r0:r0 + n], kv_scale=flat.kv_scale[r0:r0 + n],
                            pe=flat.pe[r0:r0 + n])
            mla.cache_append(sub, rows[r0:r0 + n], pe_rows[r0:r0 + n], zeros[:n])
        torch.cuda.synchronize()
        del kv
        return cache

    def _clone(self, c):
        return mla.Cache(c.max_batch, c.max_seq_len, c.fmt, kv=c.kv.clone(),
                         kv_scale=None if c.kv_scale is None else c.kv_scale.clone(), pe=c.pe.clone())

    def step(self, i: int):
        w = self.w
        if w.topk:
            mla.decode_sparse(self.caches[0], self.ql, self.qp, self.ends, w.S, w.softmax_scale,
                              self.topks[i % self.rot], kv_new=self.kv_new, pe_new=self.pe_new,
                              out=self.out, lse=self.lse, workspace=self.ws)
        else:
            c = self.caches[i % self.rot]
            if w.absorb:
                mla.absorb_q(self.q_nope, self.wkv_b, out=self.ql)
            if w.mtp > 1:
                for sp in self.start_pos:
                    mla.cache_append(c, self.kv_new, self.pe_new, sp)
                mla.decode_mtp(c, self.ql, self.qp, self.ends, w.S, w.softmax_scale, out=self.out,
                               lse=self.lse, workspace=self.ws)
            else:   # the new row (position end_pos - 1) is written by the decode call itself
                mla.decode_append(c, self.kv_new, self.pe_new, self.ql, self.qp, self.ends, w.S,
                                  w.softmax_scale, out=self.out, lse=self.lse, workspace=self.ws)
            if w.absorb:
                mla.project_out(self.out, self.wkv_b, out=self.o)


# --------------------------------------------------------------- GPU arm

PREFILL_MTP = 16     # more new tokens than this: a prefill chunk (no per-step appends)
PREFILL_SAMPLE = 8   # the oracle times this many of a chunk's tokens and scales to the chunk

def _time_graph(build, stream):
    """Capture `build()` in a CUDA graph, replay it once to warm up, then time
    one replay with CUDA events on `stream` (seconds)."""
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        build()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def read_ceiling_gbs(st, stream, passes: int = 8):
    """HBM read rate of the library's streaming read kernel over one buffer of
    CEILING_BYTES (far larger than L2, so every pass reads from HBM), one launch
    per pass, `passes` launches in a CUDA graph: the device's achievable
    streaming read rate, in GB/s.  Also returned: the same kernel over the
    step's own rotated cache tensors (one launch per tensor), a size-limited
    rate that includes the launch and ramp of short reads."""
    sink = torch.zeros(1, dtype=torch.int32, device=st.device)
    big = torch.empty(CEILING_BYTES, dtype=torch.uint8, device=st.device)
    big.fill_(1)
    with torch.cuda.stream(stream):
        mla.read_ceiling(big, sink, stream=stream)
    torch.cuda.synchronize()
    t = _time_graph(lambda: [mla.read_ceiling(big, sink, stream=stream) for _ in range(passes)], stream)
    ceiling = CEILING_BYTES * passes / t / 1e9
    del big
    tensors = [[x for x in (c.kv, c.pe, c.kv_scale) if x is not None] for c in st.caches]
    reps = 24
    nbytes = sum(x.numel() * x.element_size() for i in range(reps) for x in tensors[i % len(tensors)])
    t = _time_graph(lambda: [mla.read_ceiling(x, sink, stream=stream)
                             for i in range(reps) for x in tensors[i % len(tensors)]], stream)
    return ceiling, nbytes / t / 1e9, nbytes / reps


def run_warm(st, stream, steps: int = 200):
    """The same step with one cache (or one top-k list) every time, so the
    cache stays in L2: (step us, decode-kernel us).  None when one copy of
    the step's bytes does not fit in L2."""
    w = st.w
    if layout.step_bytes(st.tokens, w.B, w.H, w.fmt) * 1.2 > st.l2_bytes:
        return None
    for _ in range(3):
        st.step(0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(steps):
            st.step(0)
    kgraph = torch.cuda.CUDAGraph()
    mla.trace_begin(steps)
    with torch.cuda.graph(kgraph, stream=stream):
        for _ in range(steps):
            st.step(0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()          # warms L2 with the one cache
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        kgraph.replay()
    kern_ms, timed, _ = mla.trace_end()
    return {"step_us": round(e0.elapsed_time(e1) * 1e3 / steps, 3),
            "kernel_us": round(kern_ms * 1e3 / max(timed, 1), 3),
            "note": "one cache resident in L2 (warm); the headline is the cold, rotated number"}


def run_select(st, stream, reps: int = 200):
    """The top-k position selection timed on its own, at the sparse
    workload's shape: seeded N(0,1) fp32 scores for every position of every
    sequence, K of them selected per sequence; `reps` launches in a CUDA graph,
    cycling through score buffers that together exceed twice the L2.
    Algorithmic bytes: the scores read once and the lists written."""
    w = st.w
    pk, src = peaks()
    one = w.B * w.S * 4
    n = max(1, math.ceil(2 * st.l2_bytes / one))
    scores = [inputs.randn_bf16((w.B, w.S), 1000 * w.index + 97 + k, st.device).float() for k in range(n)]
    ends = st.ends
    out = torch.empty((w.B, w.topk), dtype=torch.int32, device=st.device)
    call = lambda k: mla.topk_select(scores[k % n], ends, w.topk, out=out, stream=stream)
    with torch.cuda.stream(stream):
        for k in range(3):
            call(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(reps):
            call(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / reps
    nbytes = sum(int(e) for e in st.ends_host) * 4 + w.B * w.topk * 4
    return {"kernel": "topk_select_kernel", "us": round(t * 1e6, 3), "bytes": nbytes,
            "gbs": round(nbytes / t / 1e9, 1), "frac": round(nbytes / t / 1e9 / pk["hbm_gbs"], 4),
            "peak_source": f"of {src}",
            "sample": f"{w.B} x {w.S} fp32 scores, top {w.topk} each; {n} rotating score buffers "
                      f"({n * one / 1e6:.0f} MB), cold in L2"}


def run_gemms(st, stream, reps: int = 200):
    """The query absorption and value projection timed on their own: `reps`
    launches of each captured in a CUDA graph (launches back to back), CUDA
    events around the replay, cycling through copies of wkv_b that together
    exceed twice the L2 (every launch reads its weights from HBM).
    Algorithmic bytes: one head-half of wkv_b (H x 128 x 512 bf16) plus the
    activations in and out."""
    w = st.w
    pk, src = peaks()
    nw = max(1, math.ceil(2 * st.l2_bytes / (st.wkv_b.numel() * 2)))
    wcopies = [st.wkv_b] + [st.wkv_b.clone() for _ in range(nw - 1)]
    res = {}
    for name, call, act in (
            ("absorb_q", lambda wk: mla.absorb_q(st.q_nope, wk, out=st.ql, stream=stream),
             w.B * w.H * (128 + 512) * 2),
            ("project_out", lambda wk: mla.project_out(st.out, wk, out=st.o, stream=stream),
             w.B * w.H * (512 + 128) * 2)):
        with torch.cuda.stream(stream):
            for i in range(3):
                call(wcopies[i % nw])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                call(wcopies[i % nw])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / reps
        nbytes = w.H * 128 * 512 * 2 + act
        res[name] = {"us": round(t * 1e6, 3), "bytes": nbytes, "gbs": round(nbytes / t / 1e9, 1),
                     "frac": round(nbytes / t / 1e9 / pk["hbm_gbs"], 4), "peak_source": f"of {src}",
                     "bound": "hbm (weights; N = batch is far below the MMA's M)"}
    res["weights"] = f"{nw} rotating copies of wkv_b ({nw * st.wkv_b.numel() * 2 / 1e6:.0f} MB), cold in L2"
    return res


def run_gpu(args, rank, world, local_rank):
    import torch.distributed as dist
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    mla.lib()
    w = inputs.WORKLOADS[args.workload]
    st = Setup(w, device, seed_offset=0)
    K, W = args.steps, args.warmup
    for i in range(W):
        st.step(i)
    torch.cuda.synchronize()

    # the timed graph: exactly K steps with nothing between their kernels (an
    # event node would end the programmatic launch overlap of its neighbours);
    # the library counts the kernels it launches
    stream = torch.cuda.Stream(device)
    graph = torch.cuda.CUDAGraph()
    mla.trace_begin(0)
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            st.step(W + i)
    _, _, launches = mla.trace_end()
    # a second graph times the decode kernel itself: events around each decode
    # kernel of KK further steps
    KK = min(K, 500)
    kgraph = torch.cuda.CUDAGraph()
    mla.trace_begin(KK)
    with torch.cuda.graph(kgraph, stream=stream):
        for i in range(KK):
            st.step(W + K + i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Load soak: the same K-step graph replayed back to back for about
    # SOAK_SECONDS right before the timed steps, so the clocks are sampled
    # under sustained load and the timed steps run in that state.  Its mean
    # per step is reported as "sustained"; `value` is the timed K steps.
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    one = max(e0.elapsed_time(e1) / 1e3, 1e-6)
    soak_reps = max(1, min(100000, math.ceil(args.soak / one))) if args.soak > 0 else 1
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(soak_reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    soak_s = e0.elapsed_time(e1) / 1e3
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if sampler:
        sampler.mark(False)
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    with torch.cuda.stream(stream):
        kgraph.replay()
    kern_ms, timed, _ = mla.trace_end()
    clocks = sampler.stop() if sampler else None
    ceil_gbs, same_gbs, same_bytes = read_ceiling_gbs(st, stream)
    ms = slowest(ms, device)
    step_s = ms / 1e3 / K
    cache_bytes = st.tokens * layout.cache_bytes_per_token(w.fmt)
    value = whole_job_rate(cache_bytes, world, step_s) / 1e12
    tokens_per_s = whole_job_rate(w.B * w.mtp, world, step_s)

    # dominant kernel: the decode kernel, timed by its own events
    kern_s = kern_ms / 1e3 / max(timed, 1)
    pk, pk_src = peaks()
    # token j of s attends end_pos - (s - 1 - j) positions
    attended = w.mtp * st.tokens - w.B * w.mtp * (w.mtp - 1) // 2
    flops = layout.step_flops(attended, w.H)
    t_hbm = cache_bytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved, peak, unit, bound = cache_bytes / kern_s / 1e9, pk["hbm_gbs"], "GB/s", "hbm"
    else:
        achieved, peak, unit, bound = flops / kern_s / 1e12, pk["bf16_tflops"], "TFLOP/s", "tensor"
    kernel = decode_path(w.H)
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(w.name, kernel),
                "peak_source": f"of {pk_src}", "kernel": kernel,
                "kernel_us": round(kern_s * 1e6, 3),
                "hbm_frac_of_step": round(cache_bytes / step_s / 1e9 / pk["hbm_gbs"], 4),
                "cache_read_frac_of_read_ceiling": round(cache_bytes / kern_s / 1e9 / ceil_gbs, 4),
                "roofline_time_us": round(max(t_hbm, t_tc) * 1e6, 3)}

    warm = run_warm(st, stream)
    gemms = run_gemms(st, stream) if w.absorb else None
    select = run_select(st, stream) if w.topk else None
    e2e = run_e2e(st, K, W) if not args.no_e2e else None
    cpu = run_cpu_baseline(w) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms / K, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.fmt == 0 else "fp8-e4m3 cache, bf16 MMA",
        "data": "synthetic (seeded N(0,1) bf16; FP8 cache quantised by the library's append)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "end_pos": w.T or f"U[{w.T_lo},{w.T_hi}]",
                   "attended_positions": st.tokens, "cache": "bf16" if w.fmt == 0 else "fp8-e4m3/128",
                   "topk": w.topk or None, "mtp": w.mtp,
                   "step": ("fused append + top-k gather decode" if w.topk else
                            "append new row + query absorption + decode + value projection" if w.absorb else
                            f"prefill chunk of {w.mtp} tokens over the {w.T}-position prefix (rows already "
                            "in the cache; causal among the chunk)" if w.mtp > PREFILL_MTP else
                            "append new row + decode (one call: the decode writes the row)" if w.mtp == 1 else
                            f"append {w.mtp} new rows + multi-token decode (each cache position counted once)"),
                   "l2": f"inputs larger than L2: rotating {st.rotation}; L2 {st.l2_bytes / 1e6:.0f} MB",
                   "timing": "CUDA graph of exactly K steps, CUDA events on its stream, right after a "
                          f"{args.soak:g} s load soak of the same graph",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": round(tokens_per_s, 1),
        "wall_ms_per_step": round(t_wall * 1e3 / K, 6),
        "roofline": roofline,
        "warm": warm,
        "gemms": gemms,
        "select": select,
        "read_ceiling": {"gbs": round(ceil_gbs, 1), "kernel": "read_ceiling_kernel",
                         "bytes_per_pass": CEILING_BYTES, "frac_of_measured_hbm": round(ceil_gbs / pk["hbm_gbs"], 4),
                         "sample": f"one {CEILING_BYTES >> 30} GiB buffer (cold in L2) per launch, 8 launches "
                                   "in a CUDA graph, 16-byte loads",
                         "same_size_gbs": round(same_gbs, 1), "same_size_bytes_per_pass": int(same_bytes),
                         "same_size_sample": "the step's own rotated cache tensors, one launch per tensor "
                                             "(size-limited: includes launch and ramp)"},
        "sustained": {"seconds": round(soak_s, 3), "steps": soak_reps * K,
                      "ms_per_step": round(soak_s * 1e3 / (soak_reps * K), 6),
                      "value": round(whole_job_rate(cache_bytes, world, soak_s / (soak_reps * K)) / 1e12, 4),
                      "note": "the K-step graph replayed back to back right before the timed steps (clock "
                              "samples under load); value is the timed K steps"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def _pack(named, align=256):
    """Byte offsets of the named tensors laid end to end, each `align`-aligned."""
    offs, total = {}, 0
    for k, t in named.items():
        offs[k] = total
        total += -(-t.numel() * t.element_size() // align) * align
    return offs, total


def _views(buf, offs, like):
    return {k: buf.narrow(0, offs[k], t.numel() * t.element_size()).view(t.dtype).view(t.shape)
            for k, t in like.items()}


def run_e2e(st: Setup, K: int, W: int):
    """Public API per step with host buffers: the step's inputs leave pinned
    host memory in one copy (laid end to end) and its results come back in
    one copy, all inside the timing; the steps' calls and copies are captured
    in one CUDA graph, as a serving loop replays them.  Two device slots and
    three streams let the copies of one step overlap the kernels of the
    previous one (the pipelined number); the serial number runs copy,
    kernels, copy on one stream."""
    w = st.w
    src = {("qn" if w.absorb else "ql"): (st.q_nope if w.absorb else st.ql), "qp": st.qp, "ends": st.ends}
    if w.topk or st.start_pos:   # the step's new cache rows
        src["kv_new"], src["pe_new"] = st.kv_new, st.pe_new
    if w.topk:
        src["topk"] = st.topks[0]
    res = {"res": st.o if w.absorb else st.out, "lse": st.lse}   # the step's results
    in_offs, in_total = _pack(src)
    out_offs, out_total = _pack(res)
    host_in = torch.empty(in_total, dtype=torch.uint8).pin_memory()
    for k, v in _views(host_in, in_offs, src).items():
        v.copy_(src[k].cpu())
    host_out = torch.empty(out_total, dtype=torch.uint8).pin_memory()
    dev_in = [torch.empty(in_total, dtype=torch.uint8, device=st.device) for _ in range(2)]
    dev_out = [torch.empty(out_total, dtype=torch.uint8, device=st.device) for _ in range(2)]
    vin = [_views(b, in_offs, src) for b in dev_in]
    vout = [_views(b, out_offs, res) for b in dev_out]
    h2d = sum(v.numel() * v.element_size() for v in src.values())
    d2h = sum(v.numel() * v.element_size() for v in res.values())
    n = min(K, 2000)

    def kernels(i, d, o):
        if w.topk:
            mla.decode_sparse(st.caches[0], d["ql"], d["qp"], d["ends"], w.S, w.softmax_scale, d["topk"],
                              kv_new=d["kv_new"], pe_new=d["pe_new"], out=o["res"], lse=o["lse"],
                              workspace=st.ws)
            return
        c = st.caches[i % st.rot]
        ql = mla.absorb_q(d["qn"], st.wkv_b, out=st.ql) if w.absorb else d["ql"]
        x = st.out if w.absorb else o["res"]
        if w.mtp > 1:
            for sp in st.start_pos:
                mla.cache_append(c, d["kv_new"], d["pe_new"], sp)
            mla.decode_mtp(c, ql, d["qp"], d["ends"], w.S, w.softmax_scale, out=x, lse=o["lse"],
                           workspace=st.ws)
        else:
            mla.decode_append(c, d["kv_new"], d["pe_new"], ql, d["qp"], d["ends"], w.S, w.softmax_scale,
                              out=x, lse=o["lse"], workspace=st.ws)
        if w.absorb:
            mla.project_out(x, st.wkv_b, out=o["res"])

    comp, up, down = torch.cuda.Stream(st.device), torch.cuda.Stream(st.device), torch.cuda.Stream(st.device)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free, out_ready, out_free = ([ev() for _ in range(2)] for _ in range(4))
    used = [False, False]

    def pipelined(i):
        k = i % 2
        if used[k]:
            up.wait_event(in_free[k])       # the kernels of step i-2 are done with slot k's inputs
            comp.wait_event(out_free[k])    # and its results are home
        with torch.cuda.stream(up):
            dev_in[k].copy_(host_in, non_blocking=True)
            in_ready[k].record(up)
        comp.wait_event(in_ready[k])
        with torch.cuda.stream(comp):
            kernels(i, vin[k], vout[k])
            in_free[k].record(comp)
            out_ready[k].record(comp)
        down.wait_event(out_ready[k])
        with torch.cuda.stream(down):
            host_out.copy_(dev_out[k], non_blocking=True)
            out_free[k].record(down)
        used[k] = True

    def serial(i):
        dev_in[0].copy_(host_in, non_blocking=True)
        kernels(i, vin[0], vout[0])
        host_out.copy_(dev_out[0], non_blocking=True)

    def graph_of(body):
        # n steps, each with its own upload and read-back, in one CUDA graph
        # (the other streams fork from and join the capturing one)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=comp):
            fork = ev()
            fork.record(comp)
            up.wait_event(fork)
            down.wait_event(fork)
            for i in range(n):
                body(i)
            for s_ in (up, down):
                j = ev()
                j.record(s_)
                comp.wait_event(j)
        return g

    def timed(g):
        with torch.cuda.stream(comp):
            g.replay()   # warm-up
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(comp):
            e0.record(comp)
            g.replay()
            e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    for i in range(min(W, 10)):   # eager warm-up of every call on the path
        with torch.cuda.stream(comp):
            serial(i)
    torch.cuda.synchronize()
    g_pipe = graph_of(pipelined)
    step_s = timed(g_pipe)
    del g_pipe
    g_serial = graph_of(serial)
    serial_s = timed(g_serial)
    del g_serial
    cache_bytes = st.tokens * layout.cache_bytes_per_token(w.fmt)
    return {"value": round(cache_bytes / step_s / 1e12, 4), "unit": "TB/s", "steps": n,
            "ms_per_step": round(step_s * 1e3, 6), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "serial_value": round(cache_bytes / serial_s / 1e12, 4),
            "serial_ms_per_step": round(serial_s * 1e3, 6),
            "path": "python binding -> C ABI, captured with the copies in one CUDA graph of the steps; per "
                    "step one H2D of the step's inputs (pinned, laid end to end) and one D2H of its out "
                    "and lse; two device slots, so the copies of a step overlap the kernels of the "
                    "previous one (serial_*: copy, kernels, copy in one stream)"}


# ------------------------------------------------------------ CPU oracle

def oracle_sample(w: inputs.Workload, budget_s: float):
    """Bounded sample of the workload for the CPU oracle: whole sequences (all
    heads), drawn with the same recipe on the CPU, until the time budget."""
    from oracle import oracle as orc
    ends = inputs.end_positions(w)
    S = int(ends.max())
    kv = inputs.randn_bf16((1, S, 512), 1000 * w.index + inputs.T_KV)
    pe = inputs.randn_bf16((1, S, 64), 1000 * w.index + inputs.T_PE)
    cache = {"fmt": w.fmt, "pe": inputs.bf16_bits(pe)}
    if w.fmt == 0:
        cache["kv"] = inputs.bf16_bits(kv)
    else:
        cache["kv"], cache["kv_scale"] = orc.quantize_rows(inputs.bf16_bits(kv))
    lead = (1, w.H) if w.mtp == 1 else (1, w.mtp, w.H)
    ql = inputs.randn_bf16(lead + (512,), 1000 * w.index + inputs.T_QL)
    qp = inputs.randn_bf16(lead + (64,), 1000 * w.index + inputs.T_QP)
    if w.mtp > PREFILL_MTP:   # a prefill chunk: its last PREFILL_SAMPLE tokens (time scaled up)
        ql, qp = ql[:, -PREFILL_SAMPLE:].contiguous(), qp[:, -PREFILL_SAMPLE:].contiguous()
    topk = None
    if w.topk:
        topk = inputs.topk_indices(1, w.topk, [int(ends[0])], 1000 * w.index + inputs.T_TOPK).numpy()
    T = int(ends[0])
    tokens = min(T, w.topk) if w.topk else T
    absorb = None
    if w.absorb:
        qn, wkv = inputs.absorb_inputs(w)
        absorb = (inputs.bf16_bits(qn[:1]), inputs.bf16_bits(wkv))
    return orc, cache, inputs.bf16_bits(ql), inputs.bf16_bits(qp), T, topk, tokens, absorb


def time_oracle_step(sample, w):
    orc, cache, ql, qp, T, topk, tokens, absorb = sample
    t0 = time.perf_counter()
    if absorb is not None:
        q_lat = orc.absorb_q(absorb[0], absorb[1])
        out, _ = orc.decode_absorbed(cache, q_lat, qp, [T], w.softmax_scale)
        orc.project_out(out.reshape(1, w.H, 512), absorb[1])
    elif w.mtp > 1:
        orc.decode_absorbed_mtp(cache, ql, qp, [T], w.softmax_scale)
    else:
        orc.decode_absorbed(cache, ql, qp, [T], w.softmax_scale, topk=topk)
    dt = time.perf_counter() - t0
    if w.mtp > PREFILL_MTP:   # the chunk's last tokens attend the most positions: an upper bound
        dt *= w.mtp / PREFILL_SAMPLE
    return dt, tokens


def sample_note(w):
    return (f"; the last {PREFILL_SAMPLE} of the chunk's {w.mtp} tokens timed, the time scaled by "
            f"{w.mtp // PREFILL_SAMPLE}" if w.mtp > PREFILL_MTP else "")


def run_cpu_baseline(w, min_seconds: float = 1.0):
    """The oracle on one sequence of the workload, repeated until about
    `min_seconds` of wall time (x the cores it uses: ~10-30 s of CPU work)."""
    from oracle import oracle as orc
    sample = oracle_sample(w, 10.0)
    total, reps, tokens = 0.0, 0, 0
    while total < min_seconds or reps == 0:
        dt, tokens = time_oracle_step(sample, w)
        total += dt
        reps += 1
    bytes_ = reps * tokens * layout.cache_bytes_per_token(w.fmt)
    out = {"value": round(bytes_ / total / 1e12, 8), "unit": "TB/s", "cores": orc.num_threads(),
           "kind": "oracle", "seconds": round(total, 3),
           "sample": f"{reps} x one sequence of the workload (end_pos {sample[4]}, all {w.H} heads, "
                     f"{tokens} attended positions{sample_note(w)}), fp64 oracle, OpenMP over heads"}
    if w.index == 1:   # the tiny workload: the same sample on one thread as well
        cores = orc.num_threads()
        orc.set_num_threads(1)
        try:
            t1, r1 = 0.0, 0
            while t1 < min_seconds / 2 or r1 == 0:
                dt, _ = time_oracle_step(sample, w)
                t1 += dt
                r1 += 1
        finally:
            orc.set_num_threads(cores)
        out["one_thread"] = {"value": round(r1 * tokens * layout.cache_bytes_per_token(w.fmt) / t1 / 1e12, 8),
                             "unit": "TB/s", "seconds": round(t1, 3), "reps": r1}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    from oracle import oracle as orc
    w = inputs.WORKLOADS[args.workload]
    sample = oracle_sample(w, 10.0)
    for _ in range(min(args.warmup, 1)):
        time_oracle_step(sample, w)
    K = args.steps if args.steps <= 5 else 5
    dt = 0.0
    for _ in range(K):
        d, tokens = time_oracle_step(sample, w)
        dt += d / K
    value = tokens * layout.cache_bytes_per_token(w.fmt) / dt / 1e12
    desc = (f"one sequence of {w.name} per step (end_pos {sample[4]}, all {w.H} heads, "
            f"{tokens} attended positions{sample_note(w)})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "TB/s",
        "n_gpus": world, "steps": K, "warmup": min(args.warmup, 1), "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "sample": desc},
        "cpu_baseline": {"value": round(value, 8), "unit": "TB/s", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 8), "unit": "TB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--soak", type=float, default=SOAK_SECONDS,
                    help="seconds of back-to-back graph replays before the timed steps (0: one replay)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
