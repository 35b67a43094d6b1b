"""Launch one kernel of the library a few times on one workload, for ncu.

    python -m transformer_reduce_gb300.profile_kernel KERNEL [--workload W] [--launches N]

KERNEL is softmax_fw, softmax_bw, ln_fw, ln_dinp or ln_dgdb.  Only the
buffers that kernel touches are allocated (for the encoder workload at most
~0.8 GB), so a multi-pass ncu capture (which saves and restores device memory
between passes) stays small, while the tensors still exceed L2 and the DRAM
counters mean what they say.  This is a profiling driver, not a benchmark: it
prints nothing but a line naming what it launched.
"""
from __future__ import annotations

import argparse

import torch

from . import _lib, build, workloads

_DT = {"f32": _lib.LS_F32, "f16": _lib.LS_F16, "bf16": _lib.LS_BF16}

WORKLOADS = {
    "encoder_big": (workloads.ENCODER_BIG["softmax"], workloads.ENCODER_BIG["layernorm"][0]),
    "gpt2_small": (workloads.GPT2_SMALL["softmax"], workloads.GPT2_SMALL["layernorm"]),
    "softmax_T2048": (workloads.SOFTMAX_SWEEP[-1], None),
    "layernorm_N8192": (None, workloads.LAYERNORM_SWEEP[-1]),
}


def _ok(s, where):
    if s != _lib.LS_OK:
        raise _lib.LsError(s, where)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["softmax_fw", "softmax_bw", "ln_fw", "ln_dinp", "ln_dgdb"])
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="encoder_big")
    ap.add_argument("--launches", type=int, default=3)
    a = ap.parse_args(argv)
    build.build()
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream(dev).cuda_stream
    sm_case, ln_case = WORKLOADS[a.workload]
    calls = []
    if a.kernel.startswith("softmax"):
        s = sm_case
        inp = workloads.softmax_inputs(s, device=dev)
        x, mask, dout = inp["scores"], inp["mask"], inp["dout"]
        m = 0 if mask is None else mask.data_ptr()
        if a.kernel == "softmax_fw":
            y = torch.empty_like(x)
            del dout
            calls.append(lambda: _lib.ls_softmax_fw(y.data_ptr(), x.data_ptr(), m, s.B, s.H, s.T,
                                                    s.T, s.causal, _DT[s.dtype], st))
        else:
            yf = workloads.softmax_probability_like(s, inp["lengths"], device=dev)
            dx = torch.empty_like(x)
            del x
            calls.append(lambda: _lib.ls_softmax_bw(dx.data_ptr(), dout.data_ptr(), yf.data_ptr(),
                                                    s.B, s.H, s.T, s.T, _DT[s.dtype], st))
    else:
        c = ln_case
        li = workloads.layernorm_inputs(c, device=dev)
        f32 = dict(device=dev, dtype=torch.float32)
        mean = torch.full((c.rows,), c.x_mean, **f32)
        rstd = torch.full((c.rows,), 1.0 / c.x_std, **f32)
        if a.kernel == "ln_fw":
            y = torch.empty_like(li["x"])
            calls.append(lambda: _lib.ls_layernorm_fw(
                y.data_ptr(), mean.data_ptr(), rstd.data_ptr(), li["x"].data_ptr(),
                li["gamma"].data_ptr(), li["beta"].data_ptr(), c.rows, c.hidden, c.eps,
                _DT[c.dtype], st))
        elif a.kernel == "ln_dinp":
            dx = torch.empty_like(li["x"])
            calls.append(lambda: _lib.ls_layernorm_bw_dinp(
                dx.data_ptr(), li["dy"].data_ptr(), li["x"].data_ptr(), li["gamma"].data_ptr(),
                mean.data_ptr(), rstd.data_ptr(), c.rows, c.hidden, _DT[c.dtype], st))
        else:
            n = _lib.ls_layernorm_bw_dgamma_dbeta_workspace_size(c.rows, c.hidden)
            ws = torch.empty(max(n, 16) // 4, **f32)
            dg = torch.empty(c.hidden, **f32)
            db = torch.empty(c.hidden, **f32)
            calls.append(lambda: _lib.ls_layernorm_bw_dgamma_dbeta(
                dg.data_ptr(), db.data_ptr(), li["dy"].data_ptr(), li["x"].data_ptr(),
                mean.data_ptr(), rstd.data_ptr(), c.rows, c.hidden, ws.data_ptr(),
                ws.numel() * 4, _DT[c.dtype], st))
    torch.cuda.synchronize(dev)
    for _ in range(a.launches):
        for call in calls:
            _ok(call(), a.kernel)
    torch.cuda.synchronize(dev)
    print(f"profile_kernel: {a.kernel} x{a.launches} on {a.workload}")


if __name__ == "__main__":
    main()
