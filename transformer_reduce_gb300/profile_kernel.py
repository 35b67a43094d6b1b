"""Launch (and optionally time) single kernels of the library on one workload.

    python -m transformer_reduce_gb300.profile_kernel KERNEL [--workload W] [--launches N]
    python -m transformer_reduce_gb300.profile_kernel --sweep [--launches N]

KERNEL is softmax_fw, softmax_bw, softmax_bw_masked, ln_fw, ln_dinp, ln_dgdb, ln_bw
(the fused backward), rms_fw, rms_dinp, ce_fw or ce_bw (cross entropy; its
workloads are the ce_* cases, ce_gpt2 by default), or pass: --launches whole
passes of the encoder layer (the benchmark's ten calls on one stream), or
pass_fused: the same layer with the fused LayerNorm backward and the masked
softmax backward (the benchmark's fused_pass).  Only the
buffers that kernel touches are allocated (for the encoder workload at most
~0.8 GB), so a multi-pass ncu capture, which saves and restores device memory
between passes, stays small while the tensors still exceed L2.

--sweep times every kernel on every workload of ``workloads`` (softmax: the
tiny, GPT-2-small, length-sweep and encoder cases; LayerNorm: the tiny,
GPT-2-small, width-sweep and encoder cases).  Each launch is timed alone with
CUDA events on its stream, after an L2 flush (a read of 2x the L2 size: it
evicts the kernel's inputs and leaves no dirty lines whose write-back would
run during the timed launch); one
JSON line per (kernel, workload) gives the median time and the algorithmic
GB/s (``traffic``).  These are per-kernel context numbers; the benchmark
proper is bench.py.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import _lib, build, traffic, workloads

_DT = {"f32": _lib.LS_F32, "f16": _lib.LS_F16, "bf16": _lib.LS_BF16}

SOFTMAX_CASES = {c.name: c for c in
                 [workloads.TINY["softmax"], workloads.GPT2_SMALL["softmax"],
                  *workloads.SOFTMAX_SWEEP, workloads.ENCODER_BIG["softmax"]]}
CE_CASES = {c.name: c for c in workloads.CE_CASES}
LN_CASES = {c.name: c for c in
            [workloads.TINY["layernorm"], workloads.GPT2_SMALL["layernorm"],
             *workloads.LAYERNORM_SWEEP, workloads.ENCODER_BIG["layernorm"][0]]}


def _ok(s, where):
    if s != _lib.LS_OK:
        raise _lib.LsError(s, where)


def prepare(kernel: str, case, dev):
    """(call, algorithmic bytes) for one kernel on one case; call() enqueues it."""
    st = torch.cuda.current_stream(dev).cuda_stream
    if kernel.startswith("ce"):
        ci = workloads.cross_entropy_inputs(case, device=dev)
        z, t = ci["logits"], ci["target"]
        valid = int((t >= 0).sum())
        f32 = dict(device=dev, dtype=torch.float32)
        loss = torch.empty(case.rows, **f32)
        lse = torch.full((case.rows,), 12.0, **f32)
        if kernel == "ce_fw":
            keep = (z, t, loss, lse)
            return (lambda: _lib.ls_cross_entropy_fw(
                loss.data_ptr(), lse.data_ptr(), z.data_ptr(), t.data_ptr(), case.rows,
                case.vocab, _DT[case.dtype], st)), \
                traffic.cross_entropy_fw_bytes(case.rows, valid, case.vocab, case.dtype), keep
        dz = torch.empty_like(z)
        keep = (z, t, lse, dz, ci)
        return (lambda: _lib.ls_cross_entropy_bw(
            dz.data_ptr(), z.data_ptr(), t.data_ptr(), lse.data_ptr(), ci["dloss"].data_ptr(),
            case.rows, case.vocab, _DT[case.dtype], st)), \
            traffic.cross_entropy_bw_bytes(case.rows, valid, case.vocab, case.dtype), keep
    if kernel.startswith("softmax"):
        s = case
        inp = workloads.softmax_inputs(s, device=dev)
        x, mask, dout = inp["scores"], inp["mask"], inp["dout"]
        m = 0 if mask is None else mask.data_ptr()
        if kernel == "softmax_fw":
            y = torch.empty_like(x)
            nbytes = traffic.softmax_fw_bytes(s.B, s.H, s.T, inp["lengths"], s.causal, s.dtype,
                                              mask is not None)
            keep = (x, mask, y)
            return (lambda: _lib.ls_softmax_fw(y.data_ptr(), x.data_ptr(), m, s.B, s.H, s.T, s.T,
                                               s.causal, _DT[s.dtype], st)), nbytes, keep
        yf = workloads.softmax_probability_like(s, inp["lengths"], device=dev)
        dx = torch.empty_like(x)
        keep = (dout, yf, dx, mask)
        if kernel == "softmax_bw_masked":
            nbytes = traffic.softmax_bw_masked_bytes(s.B, s.H, s.T, inp["lengths"], s.causal,
                                                     s.dtype, mask is not None)
            return (lambda: _lib.ls_softmax_bw_masked(dx.data_ptr(), dout.data_ptr(),
                                                      yf.data_ptr(), m, s.B, s.H, s.T, s.T,
                                                      s.causal, _DT[s.dtype], st)), nbytes, keep
        return (lambda: _lib.ls_softmax_bw(dx.data_ptr(), dout.data_ptr(), yf.data_ptr(), s.B,
                                           s.H, s.T, s.T, _DT[s.dtype], st)), \
            traffic.softmax_bw_bytes(s.B, s.H, s.T, s.dtype), keep
    c = case
    li = workloads.layernorm_inputs(c, device=dev)
    f32 = dict(device=dev, dtype=torch.float32)
    mean = torch.full((c.rows,), c.x_mean, **f32)
    rstd = torch.full((c.rows,), 1.0 / c.x_std, **f32)
    if kernel == "ln_fw":
        y = torch.empty_like(li["x"])
        keep = (li, y, mean, rstd)
        return (lambda: _lib.ls_layernorm_fw(
            y.data_ptr(), mean.data_ptr(), rstd.data_ptr(), li["x"].data_ptr(),
            li["gamma"].data_ptr(), li["beta"].data_ptr(), c.rows, c.hidden, c.eps,
            _DT[c.dtype], st)), traffic.layernorm_fw_bytes(c.rows, c.hidden, c.dtype), keep
    if kernel == "rms_fw":
        y = torch.empty_like(li["x"])
        keep = (li, y, rstd)
        return (lambda: _lib.ls_rmsnorm_fw(
            y.data_ptr(), rstd.data_ptr(), li["x"].data_ptr(), li["gamma"].data_ptr(), c.rows,
            c.hidden, 1e-6, _DT[c.dtype], st)), traffic.rmsnorm_fw_bytes(c.rows, c.hidden, c.dtype), keep
    if kernel == "rms_dinp":
        dx = torch.empty_like(li["x"])
        keep = (li, dx, rstd)
        return (lambda: _lib.ls_rmsnorm_bw_dinp(
            dx.data_ptr(), li["dy"].data_ptr(), li["x"].data_ptr(), li["gamma"].data_ptr(),
            rstd.data_ptr(), c.rows, c.hidden, _DT[c.dtype], st)), \
            traffic.rmsnorm_dinp_bytes(c.rows, c.hidden, c.dtype), keep
    if kernel == "ln_dinp":
        dx = torch.empty_like(li["x"])
        keep = (li, dx, mean, rstd)
        return (lambda: _lib.ls_layernorm_bw_dinp(
            dx.data_ptr(), li["dy"].data_ptr(), li["x"].data_ptr(), li["gamma"].data_ptr(),
            mean.data_ptr(), rstd.data_ptr(), c.rows, c.hidden, _DT[c.dtype], st)), \
            traffic.layernorm_dinp_bytes(c.rows, c.hidden, c.dtype), keep
    if kernel == "ln_bw":
        n = _lib.ls_layernorm_bw_workspace_size(c.rows, c.hidden)
        ws = torch.empty(max(n, 16) // 4, **f32)
        dx = torch.empty_like(li["x"])
        dg = torch.empty(c.hidden, **f32)
        db = torch.empty(c.hidden, **f32)
        keep = (li, ws, dx, dg, db, mean, rstd)
        return (lambda: _lib.ls_layernorm_bw(
            dx.data_ptr(), dg.data_ptr(), db.data_ptr(), li["dy"].data_ptr(), li["x"].data_ptr(),
            li["gamma"].data_ptr(), mean.data_ptr(), rstd.data_ptr(), c.rows, c.hidden,
            ws.data_ptr(), ws.numel() * 4, _DT[c.dtype], st)), \
            traffic.layernorm_bw_fused_bytes(c.rows, c.hidden, c.dtype), keep
    n = _lib.ls_layernorm_bw_dgamma_dbeta_workspace_size(c.rows, c.hidden)
    ws = torch.empty(max(n, 16) // 4, **f32)
    dg = torch.empty(c.hidden, **f32)
    db = torch.empty(c.hidden, **f32)
    keep = (li, ws, dg, db, mean, rstd)
    return (lambda: _lib.ls_layernorm_bw_dgamma_dbeta(
        dg.data_ptr(), db.data_ptr(), li["dy"].data_ptr(), li["x"].data_ptr(), mean.data_ptr(),
        rstd.data_ptr(), c.rows, c.hidden, ws.data_ptr(), ws.numel() * 4, _DT[c.dtype], st)), \
        traffic.layernorm_dgdb_bytes(c.rows, c.hidden, c.dtype), keep


def time_kernel(call, launches: int, dev, min_seconds: float = 0.0, warmup: int = 3,
                max_launches: int = 100_000) -> list:
    """Per-launch device times (ms), each launch timed alone after an L2 flush.

    At least `launches` launches are timed, and more until their device time
    adds up to `min_seconds` (capped at `max_launches`), after `warmup`
    untimed launches.  The flush reads a buffer of twice the L2 size and
    writes 4 bytes: it evicts the kernel's inputs and leaves no dirty lines
    whose write-back would run during the timed launch.  Stream order puts it
    before the start event and the launch is queued while it runs, so there
    is no idle gap inside the timed interval."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(2 * l2 // 4 + 1024, device=dev, dtype=torch.float32)
    sink = torch.empty((), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)

    def batch(n):
        ev = []
        for _ in range(n):
            torch.sum(flush, dim=0, out=sink)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            _ok(call(), "kernel")
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]

    batch(max(warmup, 1))
    out = batch(max(launches, 1))
    while sum(out) < min_seconds * 1e3 and len(out) < max_launches:
        est = max(sum(out) / len(out), 1e-3)
        need = int((min_seconds * 1e3 - sum(out)) / est) + 1
        out += batch(min(max(need, 1), max_launches - len(out), 2000))
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", nargs="?",
                    choices=["softmax_fw", "softmax_bw", "softmax_bw_masked", "ln_fw", "ln_dinp",
                             "ln_dgdb", "ln_bw", "rms_fw", "rms_dinp", "ce_fw", "ce_bw", "pass",
                             "pass_fused"])
    ap.add_argument("--workload", default="encoder_big",
                    help="softmax or LayerNorm case name (encoder_big picks the encoder's case)")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--only", default="", help="comma-separated kernels for --sweep")
    a = ap.parse_args(argv)
    build.build()
    dev = torch.device("cuda", 0)
    if a.sweep:
        peak = None
        try:
            import os
            root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
            peak = json.load(open(os.path.join(root, "MEASURED_PEAKS.json")))["hbm_gbs"]
        except Exception:
            pass
        jobs = [(k, c) for k in ("softmax_fw", "softmax_bw", "softmax_bw_masked")
                for c in SOFTMAX_CASES.values()]
        jobs += [(k, c) for k in ("ln_fw", "ln_dinp", "ln_dgdb", "ln_bw", "rms_fw", "rms_dinp")
                 for c in LN_CASES.values()]
        jobs += [(k, c) for k in ("ce_fw", "ce_bw") for c in CE_CASES.values()]
        if a.only:
            keep_k = set(a.only.split(","))
            jobs = [(k, c) for k, c in jobs if k in keep_k]
        for kernel, case in jobs:
            call, nbytes, keep = prepare(kernel, case, dev)
            ms = time_kernel(call, max(a.launches, 5), dev)
            med = statistics.median(ms)
            gbs = nbytes / (med / 1e3) / 1e9
            print(json.dumps({"kernel": kernel, "workload": case.name, "dtype": case.dtype,
                              "median_us": round(med * 1e3, 2), "min_us": round(min(ms) * 1e3, 2),
                              "bytes": nbytes, "gbs": round(gbs, 1),
                              "frac_of_peak": round(gbs / peak, 4) if peak else None}),
                  flush=True)
            del keep, call
            torch.cuda.empty_cache()
        return
    if a.kernel is None:
        ap.error("KERNEL or --sweep is required")
    if a.kernel in ("pass", "pass_fused"):
        from .layer_path import LayerReducePath
        path = LayerReducePath(workloads.ENCODER_BIG["softmax"],
                               workloads.ENCODER_BIG["layernorm"], device=dev)
        torch.cuda.synchronize(dev)
        for _ in range(a.launches):
            path.run() if a.kernel == "pass" else path.run_fused()
        torch.cuda.synchronize(dev)
        print(f"profile_kernel: {a.launches} encoder passes ({a.kernel})")
        return
    if a.kernel.startswith("ce"):
        case = CE_CASES[a.workload if a.workload in CE_CASES else "ce_gpt2"]
    elif a.workload == "encoder_big":
        case = workloads.ENCODER_BIG["softmax"] if a.kernel.startswith("softmax") \
            else workloads.ENCODER_BIG["layernorm"][0]
    else:
        case = (SOFTMAX_CASES if a.kernel.startswith("softmax") else LN_CASES)[a.workload]
    call, _, keep = prepare(a.kernel, case, dev)
    torch.cuda.synchronize(dev)
    for _ in range(a.launches):
        _ok(call(), a.kernel)
    torch.cuda.synchronize(dev)
    del keep
    print(f"profile_kernel: {a.kernel} x{a.launches} on {case.name}")


if __name__ == "__main__":
    main()
