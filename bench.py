#!/usr/bin/env python3
"""Benchmark of the softmax / LayerNorm reduce path on GB300.

One step = one pass of the whole hot path of a Transformer-big encoder layer
(attention softmax [32,16,512,512] bf16 with a padding mask, two LayerNorms
[16384,1024] bf16; forward and backward; ten kernel launches) through the C
ABI of libls_reduce.so, inputs resident in HBM.  The metric is whole-job
algorithmic HBM GB/s (bytes the method must move / time), with rows/s and the
roofline fraction of the dominant kernel beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs its own
replica of the pass on its own GPU (the rows are independent; there is no
data-path collective); the job time is the maximum over ranks.

Besides the headline the line carries, each measured over at least
--kernel-seconds of device time whatever --steps is: the per-kernel times of
the pass (``kernels``); every kernel alone with a cold L2 on the large
configurations -- softmax [8,16,T,T] bf16 for T in {768, 1024, 2048} and
LayerNorm [16384, N] bf16 for N in {4096, 8192} -- and on the encoder shapes
(``large_configs``, ``encoder_cold``); the widened kernels (``next_rows``);
the same layer with the fused LayerNorm backward and the masked softmax
backward (``fused_pass``); the pass replayed from a CUDA graph
(``graph_pass``); and the end-to-end pass fed from pinned host memory
(``e2e``).

--impl reference times the CPU oracle (fp64 C, on all host cores) on a
bounded row sample of the same workload; it is a deliberately slow baseline.
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
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "softmax & LayerNorm fwd+bwd HBM GB/s (% of GB300 peak) and rows/s"
WORKLOAD = ("encoder_big: attention softmax fwd+bwd [B=32,H=16,T=512,T=512] bf16, padding "
            "mask (valid length U[256,512]), no causal; two LayerNorm fwd+bwd (dinp, "
            "dgamma/dbeta) [16384,1024] bf16, eps=1e-8; one stream, pre-LN layer order")
FALLBACK_HBM_GBS = 6800.0
DOMINANT = "softmax_bw"
# ncu summary with the dominant kernel's DRAM bytes per launch (see profiles/)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "softmax_bw_encoder_big.txt")


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; only a barrier and a max)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """The largest value any rank holds (the job time is the slowest rank's)."""
    if world <= 1:
        return value
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# The sources that define the dominant kernel and its launch: a change to any
# of them makes the committed ncu traffic figure stale.
DOMINANT_SOURCES = ("ls_device.cuh", "softmax.cuh", "dispatch.cuh")


def csrc_digest() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "transformer_reduce_gb300", "csrc")
    for fn in DOMINANT_SOURCES:
        with open(os.path.join(d, fn), "rb") as f:
            h.update(fn.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when missing or taken on different kernel sources."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    m = re.search(r"^traffic_bytes_per_launch:\s*(\d+)\s+csrc_sha=(\w+)", text, re.M)
    if not m or m.group(2) != csrc_digest():
        return None
    return int(m.group(1))


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded row sample of the same workload)
# ---------------------------------------------------------------------------

class OracleSample:
    """Row sample of the encoder pass, staged as float64 host arrays.

    sm_case / sm_inputs: the softmax case and its tensors (scores, mask, dout,
    lengths); ln: list of (LayerNormCase, inputs dict with x, gamma, beta, dy).
    """

    def __init__(self, sm_case, sm_inputs, ln, softmax_frac=32, ln_frac=4):
        import oracle
        from transformer_reduce_gb300 import traffic
        oracle.build()
        self.oracle = oracle
        s = sm_case
        rows = np.arange(0, s.rows, softmax_frac, dtype=np.int64)
        flat = sm_inputs["scores"].reshape(-1, s.T)
        idx = torch.from_numpy(rows).to(flat.device)
        self.x = flat.index_select(0, idx).double().cpu().numpy()
        self.dy = sm_inputs["dout"].reshape(-1, s.T).index_select(0, idx).double().cpu().numpy()
        mask = sm_inputs["mask"]
        self.mask = None if mask is None else mask.double().cpu().numpy()
        self.batch = rows // (s.H * s.T)
        self.query = rows % s.T
        self.causal = s.causal
        frac_s = len(rows) / s.rows
        self.bytes = (traffic.softmax_fw_bytes(s.B, s.H, s.T, sm_inputs["lengths"], s.causal,
                                               s.dtype, mask is not None)
                      + traffic.softmax_bw_bytes(s.B, s.H, s.T, s.dtype)) * frac_s
        self.ln = []
        for c, li in ln:
            n = c.rows // ln_frac
            self.ln.append((li["x"][:n].double().cpu().numpy(), li["gamma"].double().cpu().numpy(),
                            li["beta"].double().cpu().numpy(), li["dy"][:n].double().cpu().numpy(),
                            c))
            self.bytes += (traffic.layernorm_fw_bytes(n, c.hidden, c.dtype)
                           + traffic.layernorm_dinp_bytes(n, c.hidden, c.dtype)
                           + traffic.layernorm_dgdb_bytes(n, c.hidden, c.dtype))
        self.description = (f"every {softmax_frac}th softmax row ({len(rows)} of {s.rows}) fw+bw, "
                            f"first 1/{ln_frac} of each LayerNorm's rows fw+dinp+dgamma/dbeta; "
                            "inputs pre-staged as float64 host arrays")
        self.pool = None

    @classmethod
    def from_path(cls, path, **kw):
        sm_inputs = {"scores": path.scores, "dout": path.dprobs, "mask": path.mask,
                     "lengths": path.lengths}
        ln = [(b.case, {"x": b.x, "gamma": b.gamma, "beta": b.beta, "dy": b.dy}) for b in path.ln]
        return cls(path.sm, sm_inputs, ln, **kw)

    def _shard(self, i, k):
        """The oracle calls on the i-th of k contiguous row blocks of the sample
        (the unmodified oracle functions; the gamma/beta column sums of the
        blocks are added at the end)."""
        o = self.oracle
        sl = slice(i * len(self.x) // k, (i + 1) * len(self.x) // k)
        y = o.softmax_fw(self.x[sl], self.mask, batch=self.batch[sl], query=self.query[sl],
                         causal=self.causal)
        o.softmax_bw(self.dy[sl], y)
        sums = []
        for x, g, b, dy, c in self.ln:
            r0, r1 = i * len(x) // k, (i + 1) * len(x) // k
            _, m, r = o.layernorm_fw(x[r0:r1], g, b, c.eps)
            o.layernorm_bw_dinp(dy[r0:r1], x[r0:r1], g, m, r)
            sums.append(o.layernorm_bw_dgamma_dbeta(dy[r0:r1], x[r0:r1], m, r))
        return sums

    def run(self, threads=1):
        """One pass over the sample on `threads` host threads (the C oracle
        releases the interpreter lock, so row blocks run in parallel)."""
        if threads <= 1:
            parts = [self._shard(0, 1)]
        else:
            if self.pool is None or self.pool._max_workers != threads:
                import concurrent.futures
                self.pool = concurrent.futures.ThreadPoolExecutor(threads)
            parts = list(self.pool.map(lambda i: self._shard(i, threads), range(threads)))
        for j in range(len(self.ln)):
            np.sum([p[j][0] for p in parts], axis=0)
            np.sum([p[j][1] for p in parts], axis=0)

    def time(self, min_seconds=10.0, max_passes=1000, threads=1):
        self.run(threads)  # first touch of the output buffers is not timed
        n, t0 = 0, time.perf_counter()
        while True:
            self.run(threads)
            n += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or n >= max_passes:
                return el / n


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def host_link(dev, nbytes: int = 256 << 20, reps: int = 3) -> dict:
    """Copy-engine bandwidth between pinned host memory and this GPU: each
    direction alone, then both at once on two streams (GB/s each way).  The
    end-to-end pass cannot move its host bytes faster than this."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(up: bool, down: bool) -> float:
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        s_up.wait_event(e0)
        s_down.wait_event(e0)
        for _ in range(reps):
            if up:
                with torch.cuda.stream(s_up):
                    d_in.copy_(h_in, non_blocking=True)
            if down:
                with torch.cuda.stream(s_down):
                    h_out.copy_(d_out, non_blocking=True)
        for s in (s_up, s_down):
            torch.cuda.current_stream(dev).wait_stream(s)
        e1.record()
        torch.cuda.synchronize(dev)
        return reps * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9

    timed(True, True)  # warm-up
    return {"h2d_gbs": round(timed(True, False), 1), "d2h_gbs": round(timed(False, True), 1),
            "both_gbs_each_way": round(timed(True, True), 1)}


# Kernels launched per call of each pass entry (ln_dgdb and the fused
# LayerNorm backward are a partial-sum kernel plus the fixed-order final sum).
KERNELS_PER_CALL = {"ln_dgdb": 2, "ln_bw": 2}

# Cold-L2 single-kernel measurements: (kernel, workload) pairs.
LARGE_CONFIGS = ([(k, f"softmax_T{T}") for T in (768, 1024, 2048)
                  for k in ("softmax_fw", "softmax_bw")]
                 + [(k, f"layernorm_N{N}") for N in (4096, 8192)
                    for k in ("ln_fw", "ln_dinp", "ln_dgdb")])
ENCODER_COLD = [("softmax_fw", "encoder_big"), ("softmax_bw", "encoder_big"),
                ("ln_fw", "encoder_big"), ("ln_dinp", "encoder_big"),
                ("ln_dgdb", "encoder_big")]
NEXT_ROWS = [("softmax_bw_masked", "encoder_big"), ("softmax_bw_masked", "softmax_T1024"),
             ("ln_bw", "encoder_big"), ("ln_bw", "layernorm_N4096"),
             ("ln_bw", "layernorm_N8192"), ("rms_fw", "layernorm_N8192"),
             ("rms_dinp", "layernorm_N8192"), ("ce_fw", "ce_gpt2"), ("ce_bw", "ce_gpt2")]


def cold_table(jobs, dev, peak, min_seconds):
    """Each (kernel, workload) launched alone after an L2 read-flush, timed
    with CUDA events on its stream over at least `min_seconds` of device time;
    only that kernel's buffers are allocated."""
    from transformer_reduce_gb300 import profile_kernel as pk
    from transformer_reduce_gb300 import workloads
    out = {}
    for kernel, wname in jobs:
        if kernel.startswith("ce"):
            case = pk.CE_CASES[wname]
        elif wname == "encoder_big":
            case = workloads.ENCODER_BIG["softmax"] if kernel.startswith("softmax") \
                else workloads.ENCODER_BIG["layernorm"][0]
        else:
            case = (pk.SOFTMAX_CASES if kernel.startswith("softmax") else pk.LN_CASES)[wname]
        call, nbytes, keep = pk.prepare(kernel, case, dev)
        ms = pk.time_kernel(call, 20, dev, min_seconds=min_seconds)
        mean_ms = sum(ms) / len(ms)
        gbs = nbytes / (mean_ms / 1e3) / 1e9
        out[f"{kernel}@{case.name}"] = {
            "kernel": kernel, "workload": case.name, "dtype": case.dtype,
            "launches": len(ms), "mean_us": round(mean_ms * 1e3, 2),
            "median_us": round(statistics.median(ms) * 1e3, 2),
            "bytes": nbytes, "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
        del keep, call
        torch.cuda.empty_cache()
    return out


def event_floor_us(stream, dev, reps=200):
    """Mean time of a CUDA event pair around a library call that does almost
    nothing (a LayerNorm forward of one row of eight features): the launch
    latency that every per-kernel event time of the one-stream pass carries."""
    from transformer_reduce_gb300 import _lib
    x = torch.ones(1, 8, device=dev, dtype=torch.bfloat16)
    g = torch.ones(8, device=dev, dtype=torch.bfloat16)
    y = torch.empty_like(x)
    st = torch.empty(2, device=dev)
    pairs = []
    for i in range(reps + 10):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s = _lib.ls_layernorm_fw(y.data_ptr(), st.data_ptr(), st.data_ptr() + 4, x.data_ptr(),
                                 g.data_ptr(), g.data_ptr(), 1, 8, 1e-8, _lib.LS_BF16,
                                 stream.cuda_stream)
        if s != _lib.LS_OK:
            raise _lib.LsError(s, "ls_layernorm_fw")
        e1.record(stream)
        if i >= 10:
            pairs.append((e0, e1))
    torch.cuda.synchronize(dev)
    return round(sum(a.elapsed_time(b) for a, b in pairs) / len(pairs) * 1e3, 2)


def kernel_stats(timers, kbytes, peak):
    kernels = {}
    for name, pairs in timers.items():
        ms = [a.elapsed_time(b) for a, b in pairs]
        per_launch = kbytes[name]
        calls_per_step = len(per_launch)
        avg_ms = sum(ms) / len(ms)
        bytes_per_call = sum(per_launch) / calls_per_step
        gbs = bytes_per_call / (avg_ms / 1e3) / 1e9
        kernels[name] = {"calls_per_step": calls_per_step, "calls_timed": len(ms),
                         "avg_ms": round(avg_ms, 5), "bytes_per_call": int(bytes_per_call),
                         "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
    return kernels


def run_ours(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    from transformer_reduce_gb300 import build, workloads
    build.build()
    from transformer_reduce_gb300.layer_path import LayerReducePath, PipelinedPasses
    dev = torch.device("cuda", local)
    path = LayerReducePath(workloads.ENCODER_BIG["softmax"], workloads.ENCODER_BIG["layernorm"],
                           device=dev)
    stream = torch.cuda.Stream(dev)
    side = torch.cuda.Stream(dev)  # the gamma/beta gradients beside the backward
    step_bytes = path.step_bytes()
    kbytes = path.kernel_bytes()
    launches_per_step = sum(KERNELS_PER_CALL.get(n, 1) for n, _ in path.sequence())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    min_s = args.kernel_seconds

    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        path.run(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    # timed region 1 (the headline): K passes back to back on one stream, as
    # one layer's forward and backward issue them, no event between kernels
    # (it would break the programmatic overlap of neighbouring launches)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        path.run(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    elapsed_s = t0.elapsed_time(t1) / 1e3
    pass_s = elapsed_s / args.steps
    # timed region 2: the same calls one after the other on one stream with an
    # event pair around every call, for each kernel's own launch duration
    # (the roofline's denominator); at least min_s of passes
    timers = {}
    kernel_steps = max(args.steps, int(min_s / pass_s) + 1)
    for _ in range(kernel_steps):
        path.run(stream, timers=timers)
    torch.cuda.synchronize(dev)
    barrier(world)
    job_s = max_over_ranks(elapsed_s, world)
    total_bytes = sum_over_ranks(step_bytes * args.steps, world)
    value = total_bytes / job_s / 1e9

    peak, peak_src = hbm_peak()
    kernels = kernel_stats(timers, kbytes, peak)
    dom = kernels[DOMINANT]
    traffic = ncu_traffic()
    roofline = {"bound": "hbm", "kernel": "softmax_bw_vec<bf16,32,2>", "achieved": dom["gbs"],
                "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                "frac": round(dom["gbs"] / peak, 4), "traffic": traffic,
                "algorithmic_bytes": dom["bytes_per_call"]}

    # the same calls with each LayerNorm's dgamma/dbeta on a second stream,
    # issued as early as a real layer could (LN2's once the forward statistics
    # exist, LN1's once the softmax backward has produced its dy)
    for _ in range(args.warmup):
        path.run_overlapped(stream, side)
    torch.cuda.synchronize(dev)
    o0 = torch.cuda.Event(enable_timing=True)
    o1 = torch.cuda.Event(enable_timing=True)
    over_steps = max(args.steps, int(min_s / pass_s) + 1)
    o0.record(stream)
    for _ in range(over_steps):
        path.run_overlapped(stream, side)
    o1.record(stream)
    torch.cuda.synchronize(dev)
    over_s = max_over_ranks(o0.elapsed_time(o1) / 1e3, world)
    overlapped = {
        "steps": over_steps, "ms_per_step": round(over_s / over_steps * 1e3, 5),
        "gbs": round(sum_over_ranks(step_bytes * over_steps, world) / over_s / 1e9, 1),
        "note": "same calls and outputs as the headline pass; each LayerNorm's dgamma/dbeta on "
                "a second stream, LN2's once the forward statistics exist, LN1's once the "
                "softmax backward is done (when its dy would exist)"}
    floor_us = event_floor_us(stream, dev)

    # the same one-stream pass captured in a CUDA graph (ten passes per graph,
    # the library calls recorded once and replayed): the launch boundaries
    # cost less when the GPU front end replays a graph
    graph_pass = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        per_graph = 10
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g, stream=stream):
            for _ in range(per_graph):
                path.run(stream)
        torch.cuda.synchronize(dev)
        for _ in range(max(1, args.warmup // per_graph + 1)):
            g.replay()
        reps = max(args.steps // per_graph, int(min_s / (pass_s * per_graph)) + 1)
        cs = torch.cuda.current_stream(dev)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(cs)
        for _ in range(reps):
            g.replay()
        g1.record(cs)
        torch.cuda.synchronize(dev)
        graph_s = max_over_ranks(g0.elapsed_time(g1) / 1e3, world)
        graph_pass = {
            "steps": reps * per_graph, "passes_per_graph": per_graph,
            "ms_per_step": round(graph_s / (reps * per_graph) * 1e3, 5),
            "gbs": round(sum_over_ranks(step_bytes * reps * per_graph, world) / graph_s / 1e9, 1),
            "note": "the headline's calls captured once in a CUDA graph and replayed"}
        del g

    # the same layer with the fused LayerNorm backward and the masked softmax
    # backward, one stream, at least min_s of passes
    fused_bytes = path.fused_step_bytes()
    for _ in range(args.warmup):
        path.run_fused(stream)
    torch.cuda.synchronize(dev)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    fused_steps = max(args.steps, int(min_s / pass_s) + 1)
    f0.record(stream)
    for _ in range(fused_steps):
        path.run_fused(stream)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    fused_s = max_over_ranks(f0.elapsed_time(f1) / 1e3, world)
    ftimers = {}
    for _ in range(kernel_steps):
        path.run_fused(stream, timers=ftimers)
    torch.cuda.synchronize(dev)
    barrier(world)
    fused_pass = {
        "calls": [n for n, _ in path.fused_sequence()],
        "steps": fused_steps, "ms_per_step": round(fused_s / fused_steps * 1e3, 5),
        "bytes_per_step": fused_bytes,
        "gbs": round(sum_over_ranks(fused_bytes * fused_steps, world) / fused_s / 1e9, 1),
        "rows_per_s": {k: round(world * v * fused_steps / fused_s)
                       for k, v in path.rows().items()},
        "kernels": kernel_stats(ftimers, path.fused_kernel_bytes(), peak),
        "note": "one stream; the same outputs as the headline pass up to the fused "
                "kernels' own summation order"}

    # end to end: every input copied from pinned host memory to the device,
    # the pass, every output copied back, each step; copies overlapped with
    # the kernels of neighbouring steps on their own streams (two device
    # buffer sets)
    link = host_link(dev)
    # lower bound of an end-to-end step: its larger copy direction at the
    # both-directions rate (the copies of a step overlap each other)
    link["floor_ms_per_step"] = round(
        max(path.h2d_bytes(), path.d2h_bytes()) / (link["both_gbs_each_way"] * 1e9) * 1e3, 4)
    e2e_steps = max(30, int(min_s / (link["floor_ms_per_step"] / 1e3)) + 1)
    twin = LayerReducePath(workloads.ENCODER_BIG["softmax"], workloads.ENCODER_BIG["layernorm"],
                           device=dev)
    pipe = PipelinedPasses([path, twin])
    pipe.run(4)  # warm-up: both buffer sets, copy engines
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = pipe.run(e2e_steps)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = sum_over_ranks(step_bytes * e2e_steps, world) / e2e_s / 1e9
    del twin, pipe
    torch.cuda.empty_cache()

    # every kernel alone with a cold L2: the large configurations, the
    # encoder shapes and the widened kernels (only that kernel's buffers are
    # allocated; the pass's buffers stay)
    large = cold_table(LARGE_CONFIGS, dev, peak, min_s) if not args.no_cold else None
    enc_cold = cold_table(ENCODER_COLD, dev, peak, min_s) if not args.no_cold else None
    nxt = cold_table(NEXT_ROWS, dev, peak, min_s) if not args.no_cold else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample.from_path(path)
        cores = host_cores()
        per_pass_1 = sample.time(min_seconds=args.cpu_seconds / 2)
        per_pass = sample.time(min_seconds=args.cpu_seconds / 2, threads=cores)
        cpu = {"value": round(sample.bytes / per_pass / 1e9, 4), "unit": "GB/s", "cores": cores,
               "kind": "oracle",
               "sample": sample.description + f"; row blocks on {cores} host threads",
               "seconds_per_sample_pass": round(per_pass, 4),
               "single_core_value": round(sample.bytes / per_pass_1 / 1e9, 4)}

    rows = path.rows()
    ln_mb = path.ln[0].x.numel() * path.ln[0].x.element_size() / 1e6
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(job_s / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "compute": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "storage": "bf16", "parallelism": "replicas",
                       "schedule": "the ten kernels back to back on one stream (programmatic "
                                   "dependent launch, no event between them); per-kernel times "
                                   "from the same pass with an event pair around every call",
                       "l2": f"inputs larger than L2 (pass moves {step_bytes / 1e9:.2f} GB; "
                             f"L2 {l2 / 1e6:.0f} MB); no flush; each LayerNorm tensor "
                             f"({ln_mb:.1f} MB) fits in L2, so the LayerNorm calls may find "
                             f"their inputs warm from the call before; the cold tables flush"},
            "pct_of_peak": round(100 * value / world / peak, 2),
            "rows_per_s": {k: round(world * v * args.steps / job_s) for k, v in rows.items()},
            "bytes_per_step": step_bytes,
            "dense_equivalent": {
                "bytes_per_step": path.dense_step_bytes(),
                "gbs": round(world * path.dense_step_bytes() * args.steps / job_s / 1e9, 1),
                "note": "as if the softmax forward read masked keys too"},
            "overlapped": overlapped,
            "graph_pass": graph_pass,
            "kernels": kernels,
            "kernels_note": (f"in-pass, one stream, {kernel_steps} passes, a CUDA event pair "
                             f"around every call; such a pair around a call that does almost "
                             f"nothing measures {floor_us} us (launch latency that the "
                             "headline pass overlaps), so short kernels read slower here than "
                             f"inside the pass; each LayerNorm tensor ({ln_mb:.1f} MB) fits in "
                             "L2, so ln_dinp and ln_dgdb may find x and dy that the call before "
                             "them read still in L2; encoder_cold has every kernel alone after "
                             "an L2 flush"),
            "event_floor_us": floor_us,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": path.h2d_bytes(), "d2h_bytes_per_step": path.d2h_bytes(),
                    "steps": e2e_steps, "ms_per_step": round(e2e_s / e2e_steps * 1e3, 4),
                    "host_link": link},
            "fused_pass": fused_pass,
            "large_configs": large,
            "encoder_cold": enc_cold,
            "next_rows": nxt,
            "cold_note": (f"each kernel alone after a read of 2x L2, CUDA events on its stream, "
                          f"at least {min_s} s of device time per entry; frac_of_peak uses the "
                          "mean launch time"),
            "clocks": clk,
            "gpu_launches": launches_per_step * args.steps,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return  # rank 0 alone runs the CPU reference
    from transformer_reduce_gb300 import workloads
    # inputs are drawn by torch's generator (on the GPU when there is one, for
    # speed); no kernel of this repository runs in this arm
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    sm_case = workloads.ENCODER_BIG["softmax"]
    ln_cases = workloads.ENCODER_BIG["layernorm"]
    sm_inputs = workloads.softmax_inputs(sm_case, device=dev)
    ln = [(c, workloads.layernorm_inputs(c, device=dev)) for c in ln_cases]
    sample = OracleSample(sm_case, sm_inputs, ln, softmax_frac=64, ln_frac=8)
    del sm_inputs, ln
    cores = host_cores()
    sample.run(cores)
    for _ in range(args.warmup):
        sample.run(cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.run(cores)
    el = time.perf_counter() - t0
    value = sample.bytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "storage": "bf16",
                   "parallelism": f"{cores} host threads over row blocks",
                   "sample": sample.description},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": sample.description + f"; row blocks on {cores} host threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum host time spent timing the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-seconds", type=float, default=0.3,
                    help="minimum device time of each per-kernel, fused-pass, end-to-end and "
                         "cold-L2 measurement")
    ap.add_argument("--no-cold", action="store_true",
                    help="skip the cold-L2 single-kernel tables")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay of the pass")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
