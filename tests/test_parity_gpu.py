"""GPU parity: libls_reduce.so (through its C ABI) against the fp64 CPU oracle.

Same seeded inputs on both sides; the tolerance rule is in ``_parity.py``.
Small configurations are compared element by element on every row; the
full-size configurations on sampled rows (first, last, batch edges, seeded
random rows) and, for the column-sum kernel, sampled columns over all rows.
Backward inputs never come from the GPU: the softmax forward output fed to
the backward is the oracle's (small sizes) or a seeded probability-like
tensor (full sizes), and the LayerNorm statistics are the oracle's.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from _parity import (compare, oracle_ln_stats, oracle_softmax_all, oracle_softmax_rows,
                     sample_rows, take_rows)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_reduce_gb300 import build
    build.build()
    import transformer_reduce_gb300 as L
    L.load()
    oracle.build()
    return L


def _L():
    import transformer_reduce_gb300 as L
    return L


def _dt(name):
    from transformer_reduce_gb300.workloads import DTYPES
    return DTYPES[name]


# ----------------------------------------------------------------------------
# generic checkers
# ----------------------------------------------------------------------------

def check_softmax(case, full=True, seed=0):
    """fw and bw of one SoftmaxCase; returns the stats list."""
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    inp = W.softmax_inputs(case, device=DEV)
    x, mask, dout = inp["scores"], inp["mask"], inp["dout"]
    y = L.softmax_fw(x, mask, causal=case.causal)
    torch.cuda.synchronize()
    B, H, T, _ = case.shape
    stats = []
    if full:
        ref = oracle_softmax_all(x, mask, case.causal)
        stats.append(compare(y, ref, case.dtype, f"{case.name} softmax_fw"))
        # backward input: the oracle's forward output, stored in the storage dtype
        y_in = torch.from_numpy(ref).to(_dt(case.dtype)).to(DEV)
        dx = L.softmax_bw(dout, y_in)
        torch.cuda.synchronize()
        refb = oracle.softmax_bw(dout.reshape(-1, T).cpu(), y_in.reshape(-1, T).cpu())
        stats.append(compare(dx.reshape(-1, T), refb, case.dtype, f"{case.name} softmax_bw"))
        y_host = y.reshape(-1, T).cpu().float().numpy()
        ref_zero = ref.reshape(-1, T) == 0.0
    else:
        rows = sample_rows(B * H * T, boundaries=[b * H * T for b in range(1, B)], seed=seed)
        ref = oracle_softmax_rows(x, mask, rows, case.causal)
        stats.append(compare(take_rows(y, rows), ref, case.dtype, f"{case.name} softmax_fw"))
        y_in = W.softmax_probability_like(case, inp["lengths"], device=DEV)
        dx = L.softmax_bw(dout, y_in)
        torch.cuda.synchronize()
        refb = oracle.softmax_bw(take_rows(dout, rows), take_rows(y_in, rows))
        stats.append(compare(take_rows(dx, rows), refb, case.dtype, f"{case.name} softmax_bw"))
        y_host = take_rows(y, rows).float().numpy()
        ref_zero = ref == 0.0
    # masked and future keys are exactly zero on the GPU as in the oracle
    assert np.all(y_host[ref_zero] == 0.0), "masked/future probabilities must be exactly 0"
    return stats


def check_layernorm(case, full=True, seed=0):
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    inp = W.layernorm_inputs(case, device=DEV)
    x, g, b, dy = inp["x"], inp["gamma"], inp["beta"], inp["dy"]
    y, mean, rstd = L.layernorm_fw(x, g, b, case.eps)
    torch.cuda.synchronize()
    stats = []
    R, N = x.shape
    rows = np.arange(R) if full else sample_rows(R, seed=seed)
    yr, mr, rr = oracle.layernorm_fw(take_rows(x, rows), g.cpu(), b.cpu(), case.eps)
    stats.append(compare(take_rows(y, rows), yr, case.dtype, f"{case.name} ln_fw y"))
    stats.append(compare(mean.cpu()[rows], mr, case.dtype, f"{case.name} ln_fw mean"))
    stats.append(compare(rstd.cpu()[rows], rr, case.dtype, f"{case.name} ln_fw rstd"))
    # backward inputs: the oracle's statistics of every row, stored as fp32
    m_all, r_all = oracle_ln_stats(x, g, b, case.eps)
    mean_in = torch.from_numpy(m_all).float().to(DEV)
    rstd_in = torch.from_numpy(r_all).float().to(DEV)
    dx = L.layernorm_bw_dinp(dy, x, g, mean_in, rstd_in)
    dgm, dbt = L.layernorm_bw_dgamma_dbeta(dy, x, mean_in, rstd_in)
    torch.cuda.synchronize()
    refdx = oracle.layernorm_bw_dinp(take_rows(dy, rows), take_rows(x, rows), g.cpu(),
                                     mean_in.cpu()[rows], rstd_in.cpu()[rows])
    stats.append(compare(take_rows(dx, rows), refdx, case.dtype, f"{case.name} ln_dinp"))
    cols = np.arange(N) if full else np.unique(np.concatenate(
        [np.arange(min(8, N)), np.arange(max(0, N - 8), N),
         np.random.default_rng(seed).integers(0, N, size=48)]))
    ci = torch.from_numpy(cols).to(DEV)
    rg, rb = oracle.layernorm_bw_dgamma_dbeta(dy.index_select(1, ci).cpu(),
                                              x.index_select(1, ci).cpu(),
                                              mean_in.cpu(), rstd_in.cpu())
    stats.append(compare(dgm.cpu()[cols], rg, case.dtype, f"{case.name} ln_dgamma"))
    stats.append(compare(dbt.cpu()[cols], rb, case.dtype, f"{case.name} ln_dbeta"))
    return stats


# ----------------------------------------------------------------------------
# the five configurations
# ----------------------------------------------------------------------------

def test_tiny_layer_fp32():
    from transformer_reduce_gb300 import workloads as W
    check_softmax(W.TINY["softmax"], full=True)
    check_layernorm(W.TINY["layernorm"], full=True)


def test_gpt2_small_fp16():
    from transformer_reduce_gb300 import workloads as W
    check_softmax(W.GPT2_SMALL["softmax"], full=True)
    check_layernorm(W.GPT2_SMALL["layernorm"], full=True)


@pytest.mark.parametrize("T", [32, 64, 128, 256, 384, 512, 768, 1024, 2048])
def test_softmax_length_sweep_bf16(T):
    from transformer_reduce_gb300 import workloads as W
    case = [c for c in W.SOFTMAX_SWEEP if c.T == T][0]
    check_softmax(case, full=case.rows * T <= (1 << 22), seed=T)


@pytest.mark.parametrize("N", [768, 1024, 2048, 4096, 8192])
def test_layernorm_width_sweep_bf16(N):
    from transformer_reduce_gb300 import workloads as W
    case = [c for c in W.LAYERNORM_SWEEP if c.hidden == N][0]
    check_layernorm(case, full=False, seed=N)


def test_encoder_big_layer_pass_bf16():
    """The pass the benchmark times (same calls, shapes and launches), checked
    on sampled rows of every output.  The forward outputs are checked as the
    pass leaves them; the backward calls are then re-issued by the same pass
    object on backward inputs that come from the seeded generator (softmax)
    and from the oracle (LayerNorm statistics), never from the GPU."""
    from transformer_reduce_gb300 import workloads as W
    from transformer_reduce_gb300.layer_path import LayerReducePath
    p = LayerReducePath(W.ENCODER_BIG["softmax"], W.ENCODER_BIG["layernorm"], device=DEV)
    p.run()
    p.run()
    torch.cuda.synchronize()
    s = p.sm
    rows = sample_rows(s.rows, boundaries=[b * s.H * s.T for b in range(1, s.B)], seed=5)
    ref = oracle_softmax_rows(p.scores, p.mask, rows, s.causal)
    compare(take_rows(p.probs, rows), ref, s.dtype, "encoder softmax_fw")
    lr = {}
    for b in p.ln:
        c = b.case
        r = sample_rows(c.rows, seed=7)
        yr, mr, rr = oracle.layernorm_fw(take_rows(b.x, r), b.gamma.cpu(), b.beta.cpu(), c.eps)
        compare(take_rows(b.y, r), yr, c.dtype, f"{c.name} y")
        compare(b.mean.cpu()[r], mr, c.dtype, f"{c.name} mean")
        compare(b.rstd.cpu()[r], rr, c.dtype, f"{c.name} rstd")
        lr[c.name] = r

    # backward on generator / oracle inputs, through the pass's own calls
    p.probs.copy_(W.softmax_probability_like(s, p.lengths, device=DEV))
    for b in p.ln:
        m, r = oracle_ln_stats(b.x, b.gamma, b.beta, b.case.eps)
        b.mean.copy_(torch.from_numpy(m).float())
        b.rstd.copy_(torch.from_numpy(r).float())
    st = torch.cuda.current_stream().cuda_stream
    for name, call in p.sequence():
        if name in ("softmax_bw", "ln_dinp", "ln_dgdb"):
            call(st)
    torch.cuda.synchronize()
    refb = oracle.softmax_bw(take_rows(p.dprobs, rows), take_rows(p.probs, rows))
    compare(take_rows(p.dscores, rows), refb, s.dtype, "encoder softmax_bw")
    for b in p.ln:
        c = b.case
        r = lr[c.name]
        refdx = oracle.layernorm_bw_dinp(take_rows(b.dy, r), take_rows(b.x, r), b.gamma.cpu(),
                                         b.mean.cpu()[r], b.rstd.cpu()[r])
        compare(take_rows(b.dx, r), refdx, c.dtype, f"{c.name} dx")
        cols = np.array([0, 1, 7, 8, 255, 256, 511, 512, 777, c.hidden - 1])
        ci = torch.from_numpy(cols).to(DEV)
        rg, rb = oracle.layernorm_bw_dgamma_dbeta(b.dy.index_select(1, ci).cpu(),
                                                  b.x.index_select(1, ci).cpu(),
                                                  b.mean.cpu(), b.rstd.cpu())
        compare(b.dgamma.cpu()[cols], rg, c.dtype, f"{c.name} dgamma")
        compare(b.dbeta.cpu()[cols], rb, c.dtype, f"{c.name} dbeta")


def test_overlapped_pass_matches_the_serial_pass():
    """dgamma/dbeta on a side stream (the benchmark's schedule) gives exactly
    the outputs of the one-stream pass, over several passes in a row."""
    from transformer_reduce_gb300 import workloads as W
    from transformer_reduce_gb300.layer_path import LayerReducePath
    mk = lambda: LayerReducePath(W.GPT2_SMALL["softmax"],  # noqa: E731
                                 [W.GPT2_SMALL["layernorm"], W.TINY["layernorm"]], device=DEV)
    a, b = mk(), mk()
    st = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    for _ in range(3):
        a.run(st)
        b.run_overlapped(st, side)
    torch.cuda.synchronize()
    for x, y in zip(a._outputs(), b._outputs()):
        assert torch.equal(x, y)


def test_pass_replayed_from_a_cuda_graph_matches_the_eager_pass():
    """The library's calls can be captured in a CUDA graph (they allocate and
    synchronise nothing); the replay writes exactly the eager pass's outputs."""
    from transformer_reduce_gb300 import workloads as W
    from transformer_reduce_gb300.layer_path import LayerReducePath
    mk = lambda: LayerReducePath(W.GPT2_SMALL["softmax"],  # noqa: E731
                                 [W.GPT2_SMALL["layernorm"], W.TINY["layernorm"]], device=DEV)
    a, b = mk(), mk()
    st = torch.cuda.Stream()
    a.run(st)
    b.run(st)  # first calls (occupancy queries, attributes) outside the capture
    torch.cuda.synchronize()
    for t in b._outputs():
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        b.run(st)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for x, y in zip(a._outputs(), b._outputs()):
        assert torch.equal(x, y)


def test_fused_pass_matches_the_serial_pass():
    """The layer with the fused LayerNorm backward and the masked softmax
    backward (the benchmark's fused_pass) gives the outputs of the plain pass
    within the tolerance rule; only summation orders differ."""
    from transformer_reduce_gb300 import workloads as W
    from transformer_reduce_gb300.layer_path import LayerReducePath
    mk = lambda: LayerReducePath(W.ENCODER_BIG["softmax"],  # noqa: E731
                                 W.ENCODER_BIG["layernorm"], device=DEV)
    a = mk()
    a.run()
    torch.cuda.synchronize()
    want = [t.clone() for t in a._outputs()]
    for t in a._outputs():
        t.fill_(float("nan"))
    a.run_fused()
    a.run_fused()
    torch.cuda.synchronize()
    names = ["probs", "dscores"] + [f"ln{i} {n}" for i in (1, 2)
                                     for n in ("y", "mean", "rstd", "dx", "dgamma", "dbeta")]
    rows = sample_rows(a.sm.rows, k=256, seed=3)
    for name, got, ref in zip(names, a._outputs(), want):
        if got.dim() == 4:
            got, ref = take_rows(got, rows), take_rows(ref, rows)
        compare(got, ref.double().cpu().numpy(), "bf16", f"fused pass {name}")


def test_pipelined_passes_deliver_the_plain_pass_outputs():
    """The end-to-end schedule (two device buffer sets, copies on their own
    streams) brings back exactly what one plain pass computes."""
    from transformer_reduce_gb300 import workloads as W
    from transformer_reduce_gb300.layer_path import LayerReducePath, PipelinedPasses
    mk = lambda: LayerReducePath(W.GPT2_SMALL["softmax"],  # noqa: E731
                                 [W.GPT2_SMALL["layernorm"], W.TINY["layernorm"]], device=DEV)
    a, b = mk(), mk()
    pipe = PipelinedPasses([a, b])
    for h in pipe.hout:
        h.fill_(float("nan"))
    pipe.run(3)  # the last step runs on buffer set a
    torch.cuda.synchronize()
    ref = mk()
    ref.run()
    torch.cuda.synchronize()
    for h, d in zip(pipe.hout, ref._outputs()):
        assert torch.equal(h, d.cpu())


# ----------------------------------------------------------------------------
# edge cases
# ----------------------------------------------------------------------------

def _softmax_case(B, H, T, causal, pad, dtype, seed=9, std=3.0):
    from transformer_reduce_gb300.workloads import SoftmaxCase
    return SoftmaxCase(f"edge_{dtype}_{B}x{H}x{T}", B, H, T, causal, pad, std, dtype, seed)


def _ln_case(rows, hidden, dtype, seed=9, mean=1.0, std=2.0):
    from transformer_reduce_gb300.workloads import LayerNormCase
    return LayerNormCase(f"edge_{dtype}_{rows}x{hidden}", rows, hidden, mean, std, dtype, seed)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("T", [1, 3, 8, 37, 100, 264, 1000])
def test_softmax_ragged_lengths(dtype, T):
    # lengths that are not a multiple of the 16-byte vector take the looped path
    check_softmax(_softmax_case(2, 3, T, True, (max(1, T // 2), T), dtype), full=True)
    check_softmax(_softmax_case(2, 3, T, False, (max(1, T // 2), T), dtype), full=True)


@pytest.mark.parametrize("dtype,Tk", [("bf16", 4096), ("bf16", 16384), ("f32", 8192),
                                      ("f16", 20000), ("f32", 3000), ("bf16", 16392)])
def test_softmax_long_rows(dtype, Tk):
    """Rows beyond one warp: multi-warp register buckets and the looped path."""
    L = _L()
    dt = _dt(dtype)
    g = torch.Generator(device=DEV).manual_seed(Tk)
    B, H, Tq = 2, 2, 6
    x = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).mul(3).to(dt)
    mask = torch.zeros(B, Tk, device=DEV)
    mask[0, Tk // 3:] = -math.inf
    mask = mask.to(dt)
    dout = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).to(dt)
    y = L.softmax_fw(x, mask)
    torch.cuda.synchronize()
    ref = oracle.softmax_fw_tensor(x.cpu(), mask.cpu())
    compare(y, ref, dtype, f"long fw {Tk}")
    assert np.all(y.cpu().float().numpy()[ref == 0.0] == 0.0)
    y_in = torch.from_numpy(ref).to(dt).to(DEV)
    dx = L.softmax_bw(dout, y_in)
    torch.cuda.synchronize()
    refb = oracle.softmax_bw(dout.reshape(-1, Tk).cpu(), y_in.reshape(-1, Tk).cpu())
    compare(dx.reshape(-1, Tk), refb, dtype, f"long bw {Tk}")
    # causal needs Tq == Tk; a square long case on a few rows of the batch
    if Tk <= 4096:
        xc = torch.randn(1, 1, Tk, Tk, generator=g, device=DEV).to(dt)
        yc = L.softmax_fw(xc, causal=True)
        torch.cuda.synchronize()
        rows = sample_rows(Tk, k=24, seed=1)
        compare(take_rows(yc, rows), oracle_softmax_rows(xc, None, rows, True), dtype,
                f"long causal {Tk}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 5, 8, 24, 32, 64, 100, 770, 1000, 1536, 12288, 20000])
def test_layernorm_odd_widths(dtype, N):
    # 8-32 features: rows of one to four 16-byte chunks, held by one or two
    # threads (the row's shift and statistics pass through one-lane shuffles)
    check_layernorm(_ln_case(33, N, dtype), full=True)


def test_layernorm_single_row_and_constant_rows():
    L = _L()
    for dtype in ("f32", "bf16"):
        dt = _dt(dtype)
        x = torch.full((3, 256), 0.375, device=DEV, dtype=dt)
        x[1] = -3.0
        x[2, :] = torch.linspace(-1, 1, 256, device=DEV).to(dt)
        g = torch.linspace(0.5, 1.5, 256, device=DEV).to(dt)
        b = torch.linspace(-0.2, 0.2, 256, device=DEV).to(dt)
        y, mean, rstd = L.layernorm_fw(x, g, b, 1e-8)
        yr, mr, rr = oracle.layernorm_fw(x.cpu(), g.cpu(), b.cpu(), 1e-8)
        compare(y, yr, dtype, "constant rows y")
        compare(mean, mr, dtype, "constant rows mean")
        compare(rstd, rr, dtype, "constant rows rstd")
        # a constant row normalises to beta exactly
        assert torch.equal(y[0], b) and torch.equal(y[1], b)
        y1, m1, r1 = L.layernorm_fw(x[2:3].contiguous(), g, b, 1e-8)
        compare(y1, yr[2:3], dtype, "single row")


def test_softmax_fully_masked_rows_and_nonbinary_mask():
    L = _L()
    for dtype in ("f32", "f16", "bf16"):
        dt = _dt(dtype)
        g = torch.Generator(device=DEV).manual_seed(3)
        x = torch.randn(3, 2, 5, 40, generator=g, device=DEV).mul(3).to(dt)
        mask = torch.randn(3, 40, generator=g, device=DEV).to(dt)  # finite additive bias
        mask[1] = -math.inf                                          # batch 1: nothing visible
        mask[2, ::3] = -math.inf
        y = L.softmax_fw(x, mask)
        torch.cuda.synchronize()
        ref = oracle.softmax_fw_tensor(x.cpu(), mask.cpu())
        compare(y, ref, dtype, "mask edge fw")
        assert torch.all(y[1] == 0)
        y_in = torch.from_numpy(ref).to(dt).to(DEV)
        dx = L.softmax_bw(torch.randn(x.shape, generator=g, device=DEV).to(dt), y_in)
        torch.cuda.synchronize()
        assert torch.all(dx[1] == 0)


def test_in_place_calls():
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    case = _softmax_case(2, 2, 256, True, (100, 256), "bf16")
    inp = W.softmax_inputs(case, device=DEV)
    x = inp["scores"].clone()
    ref = oracle_softmax_all(x, inp["mask"], True)
    L.softmax_fw(x, inp["mask"], causal=True, out=x)
    torch.cuda.synchronize()
    compare(x, ref, "bf16", "in-place softmax_fw")
    yf = W.softmax_probability_like(case, inp["lengths"], device=DEV)
    d = inp["dout"].clone()
    refb = oracle.softmax_bw(d.reshape(-1, 256).cpu(), yf.reshape(-1, 256).cpu())
    L.softmax_bw(d, yf, dinp=d)
    torch.cuda.synchronize()
    compare(d.reshape(-1, 256), refb, "bf16", "in-place softmax_bw")
    lc = _ln_case(64, 1024, "bf16")
    li = W.layernorm_inputs(lc, device=DEV)
    m, r = oracle_ln_stats(li["x"], li["gamma"], li["beta"], lc.eps)
    mt, rt = torch.from_numpy(m).float().to(DEV), torch.from_numpy(r).float().to(DEV)
    dy = li["dy"].clone()
    refdx = oracle.layernorm_bw_dinp(dy.cpu(), li["x"].cpu(), li["gamma"].cpu(), mt.cpu(), rt.cpu())
    L.layernorm_bw_dinp(dy, li["x"], li["gamma"], mt, rt, dx=dy)
    torch.cuda.synchronize()
    compare(dy, refdx, "bf16", "in-place ln_dinp")


def test_misaligned_pointers_take_the_scalar_path():
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    case = _softmax_case(1, 2, 128, False, (64, 128), "bf16")
    inp = W.softmax_inputs(case, device=DEV)
    n = inp["scores"].numel()
    buf = torch.empty(n + 1, device=DEV, dtype=torch.bfloat16)
    xs = buf[1:].view(case.shape)          # 2-byte aligned, not 16-byte aligned
    xs.copy_(inp["scores"])
    y = L.softmax_fw(xs, inp["mask"])
    torch.cuda.synchronize()
    compare(y, oracle_softmax_all(inp["scores"], inp["mask"], False), "bf16", "misaligned fw")
    lc = _ln_case(16, 512, "bf16")
    li = W.layernorm_inputs(lc, device=DEV)
    xb = torch.empty(li["x"].numel() + 3, device=DEV, dtype=torch.bfloat16)
    xm = xb[3:].view(16, 512)
    xm.copy_(li["x"])
    y, mean, rstd = L.layernorm_fw(xm, li["gamma"], li["beta"], 1e-8)
    yr, mr, rr = oracle.layernorm_fw(li["x"].cpu(), li["gamma"].cpu(), li["beta"].cpu(), 1e-8)
    compare(y, yr, "bf16", "misaligned ln y")


def test_empty_problems():
    L = _L()
    x = torch.empty(0, 4, 8, 8, device=DEV)
    assert L.softmax_fw(x).shape == x.shape
    assert L.softmax_bw(x, x).shape == x.shape
    xe = torch.empty(0, 64, device=DEV, dtype=torch.bfloat16)
    g = torch.ones(64, device=DEV, dtype=torch.bfloat16)
    y, m, r = L.layernorm_fw(xe, g, g, 1e-8)
    assert y.shape == (0, 64)
    dg, db = L.layernorm_bw_dgamma_dbeta(xe, xe, m, r,
                                         dgamma=torch.full((64,), 7.0, device=DEV),
                                         dbeta=torch.full((64,), 7.0, device=DEV))
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)   # a sum over no rows is zero


def test_dgamma_dbeta_is_bitwise_reproducible():
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    case = W.LAYERNORM_SWEEP[1]
    li = W.layernorm_inputs(case, device=DEV)
    _, mean, rstd = L.layernorm_fw(li["x"], li["gamma"], li["beta"], case.eps)
    outs = [L.layernorm_bw_dgamma_dbeta(li["dy"], li["x"], mean, rstd) for _ in range(3)]
    torch.cuda.synchronize()
    for dg, db in outs[1:]:
        assert torch.equal(dg, outs[0][0]) and torch.equal(db, outs[0][1])


def test_outputs_stay_inside_their_buffers():
    """Guard bands of a sentinel pattern around every output are left untouched."""
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    G = 4096
    for case, ln in [(_softmax_case(2, 3, 100, True, (50, 100), "bf16"), _ln_case(7, 100, "bf16")),
                     (_softmax_case(2, 3, 512, False, (300, 512), "bf16"), _ln_case(9, 1024, "bf16")),
                     (_softmax_case(1, 2, 64, True, None, "f32"), _ln_case(5, 4096, "f32"))]:
        dt = _dt(case.dtype)
        inp = W.softmax_inputs(case, device=DEV)
        n = inp["scores"].numel()

        def guarded(numel, dtype):
            buf = torch.full((numel + 2 * G,), -12345.0, device=DEV, dtype=dtype)
            return buf, buf[G:G + numel]

        ybuf, y = guarded(n, dt)
        L.softmax_fw(inp["scores"], inp["mask"], case.causal, out=y.view(case.shape))
        dbuf, d = guarded(n, dt)
        L.softmax_bw(inp["dout"], y.view(case.shape), dinp=d.view(case.shape))
        li = W.layernorm_inputs(ln, device=DEV)
        R, N = ln.rows, ln.hidden
        lybuf, ly = guarded(R * N, dt)
        mbuf, m = guarded(R, torch.float32)
        rbuf, r = guarded(R, torch.float32)
        L.layernorm_fw(li["x"], li["gamma"], li["beta"], 1e-8, y=ly.view(R, N), mean=m, rstd=r)
        dxbuf, dx = guarded(R * N, dt)
        L.layernorm_bw_dinp(li["dy"], li["x"], li["gamma"], m, r, dx=dx.view(R, N))
        gbuf, gg = guarded(N, torch.float32)
        bbuf, bb = guarded(N, torch.float32)
        L.layernorm_bw_dgamma_dbeta(li["dy"], li["x"], m, r, dgamma=gg, dbeta=bb)
        torch.cuda.synchronize()
        for buf in (ybuf, dbuf, lybuf, mbuf, rbuf, dxbuf, gbuf, bbuf):
            assert torch.all(buf[:G] == -12345.0) and torch.all(buf[-G:] == -12345.0)


def test_widened_outputs_stay_inside_their_buffers():
    """Guard bands around the outputs and workspaces of the widened entry
    points (masked and scaled softmax, fused LayerNorm backward, RMSNorm,
    cross entropy) are left untouched."""
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    G = 4096
    SENT = -12345.0

    def guarded(numel, dtype):
        buf = torch.full((numel + 2 * G,), SENT, device=DEV, dtype=dtype)
        return buf, buf[G:G + numel]

    bufs = []
    for case, ln, vocab in [(_softmax_case(2, 3, 100, True, (50, 100), "bf16"), _ln_case(7, 100, "bf16"), 1001),
                            (_softmax_case(2, 3, 512, False, (300, 512), "bf16"), _ln_case(309, 1024, "bf16"), 50257),
                            (_softmax_case(1, 2, 64, True, None, "f32"), _ln_case(5, 4096, "f32"), 77)]:
        dt = _dt(case.dtype)
        inp = W.softmax_inputs(case, device=DEV)
        n = inp["scores"].numel()
        ybuf, y = guarded(n, dt)
        L.softmax_fw(inp["scores"], inp["mask"], case.causal, out=y.view(case.shape), scale=0.25)
        dbuf, d = guarded(n, dt)
        L.softmax_bw_masked(inp["dout"], y.view(case.shape), inp["mask"], case.causal,
                            dinp=d.view(case.shape), scale=0.25)
        bufs += [ybuf, dbuf]
        li = W.layernorm_inputs(ln, device=DEV)
        R, N = ln.rows, ln.hidden
        _, m, r = L.layernorm_fw(li["x"], li["gamma"], li["beta"], 1e-8)
        n_ws = L.ls_layernorm_bw_workspace_size(R, N)
        wsbuf, ws = guarded(max(n_ws, 16) // 4, torch.float32)
        dxbuf, dx = guarded(R * N, dt)
        gbuf, gg = guarded(N, torch.float32)
        bbuf, bb = guarded(N, torch.float32)
        L.layernorm_bw(li["dy"], li["x"], li["gamma"], m, r, workspace=ws, dx=dx.view(R, N),
                       dgamma=gg, dbeta=bb)
        rybuf, ry = guarded(R * N, dt)
        rrbuf, rr = guarded(R, torch.float32)
        L.rmsnorm_fw(li["x"], li["gamma"], 1e-6, y=ry.view(R, N), rstd=rr)
        rdxbuf, rdx = guarded(R * N, dt)
        L.rmsnorm_bw_dinp(li["dy"], li["x"], li["gamma"], rr, dx=rdx.view(R, N))
        rgbuf, rg = guarded(N, torch.float32)
        L.rmsnorm_bw_dgamma(li["dy"], li["x"], rr, dgamma=rg)
        bufs += [wsbuf, dxbuf, gbuf, bbuf, rybuf, rrbuf, rdxbuf, rgbuf]
        ce = W.CrossEntropyCase("guard", 1, 13, vocab, (10, 12), 3.0, case.dtype, 3)
        ci = W.cross_entropy_inputs(ce, device=DEV)
        lbuf, lo = guarded(13, torch.float32)
        sbuf, ls = guarded(13, torch.float32)
        L.cross_entropy_fw(ci["logits"], ci["target"], loss=lo, lse=ls)
        zbuf, dz = guarded(13 * vocab, dt)
        L.cross_entropy_bw(ci["logits"], ci["target"], ls, ci["dloss"], dlogits=dz.view(13, vocab))
        bufs += [lbuf, sbuf, zbuf]
    torch.cuda.synchronize()
    for buf in bufs:
        assert torch.all(buf[:G] == SENT) and torch.all(buf[-G:] == SENT)


# ----------------------------------------------------------------------------
# causal with Tq < Tk, and the masked backward
# ----------------------------------------------------------------------------

def _rand_problem(B, H, Tq, Tk, dtype, seed, lengths=None):
    g = torch.Generator(device=DEV).manual_seed(seed)
    dt = _dt(dtype)
    x = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).mul(3).to(dt)
    dout = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).to(dt)
    mask = None
    if lengths is not None:
        m = torch.zeros(B, Tk, device=DEV)
        for b, n in enumerate(lengths):
            m[b, n:] = -math.inf
        mask = m.to(dt)
    return x, dout, mask


@pytest.mark.parametrize("dtype,shape", [("f32", (2, 3, 5, 9)), ("bf16", (1, 2, 64, 256)),
                                         ("f16", (2, 2, 7, 37)), ("bf16", (1, 1, 40, 4096))])
def test_softmax_fw_causal_with_fewer_queries(dtype, shape):
    L = _L()
    B, H, Tq, Tk = shape
    x, _, mask = _rand_problem(B, H, Tq, Tk, dtype, 61, lengths=[Tk - 1] * B)
    y = L.softmax_fw(x, mask, causal=True)
    torch.cuda.synchronize()
    ref = oracle.softmax_fw_tensor_offset(x.cpu(), mask.cpu(), causal=True)
    compare(y, ref, dtype, f"causal Tq<Tk fw {shape}")
    assert np.all(y.cpu().float().numpy()[ref == 0.0] == 0.0)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape,lengths,causal", [
    ((2, 3, 16, 16), [9, 16], True),
    ((2, 3, 16, 256), [200, 77], False),
    ((2, 2, 40, 64), [64, 33], True),
    ((1, 2, 8, 100), [61], True),        # ragged: looped path
    ((1, 2, 4, 2048), [1500], False),
    ((1, 1, 3, 5000), [4000], True),     # beyond the register buckets
])
def test_softmax_bw_masked_ignores_invisible_keys(dtype, shape, lengths, causal):
    """The masked backward equals the oracle's masked backward, is exactly 0 on
    invisible keys, and is unaffected by garbage there in out_fw and dout."""
    L = _L()
    B, H, Tq, Tk = shape
    x, dout, mask = _rand_problem(B, H, Tq, Tk, dtype, 62, lengths)
    yref = oracle.softmax_fw_tensor_offset(x.cpu(), mask.cpu(), causal=causal)
    invisible = torch.from_numpy(yref == 0.0).to(DEV)
    y = torch.from_numpy(yref).to(_dt(dtype)).to(DEV)
    y_dirty = torch.where(invisible, torch.full_like(y, 7.0), y)
    d_dirty = torch.where(invisible, torch.full_like(dout, -3.0), dout)
    dx = L.softmax_bw_masked(d_dirty, y_dirty, mask, causal=causal)
    torch.cuda.synchronize()
    want = oracle.softmax_bw_masked_tensor(d_dirty.cpu(), y_dirty.cpu(), mask.cpu(), causal=causal)
    compare(dx, want, dtype, f"masked bw {shape} causal={causal}")
    assert torch.all(dx[invisible] == 0)
    # with the forward's own zeros it is the plain backward
    dx_plain = L.softmax_bw(dout, y)
    torch.cuda.synchronize()
    compare(dx_plain, oracle.softmax_bw(dout.reshape(-1, Tk).cpu(), y.reshape(-1, Tk).cpu()),
            dtype, "plain bw on the same forward")


def test_softmax_bw_masked_encoder_big_sampled():
    """The Transformer-big encoder shape (padding mask), sampled rows."""
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    s = W.ENCODER_BIG["softmax"]
    inp = W.softmax_inputs(s, device=DEV)
    y = W.softmax_probability_like(s, inp["lengths"], device=DEV)
    dx = L.softmax_bw_masked(inp["dout"], y, inp["mask"], causal=False)
    torch.cuda.synchronize()
    rows = sample_rows(s.rows, boundaries=[b * s.H * s.T for b in range(1, s.B)], seed=8)
    want = oracle.softmax_bw_masked(take_rows(inp["dout"], rows), take_rows(y, rows),
                                    inp["mask"].cpu(), batch=rows // (s.H * s.T))
    compare(take_rows(dx, rows), want, s.dtype, "encoder masked bw")


# ----------------------------------------------------------------------------
# scaled softmax: softmax(scale * scores + mask) and its masked backward
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape,lengths,causal,scale", [
    ((2, 3, 16, 16), [9, 16], True, 0.125),
    ((2, 3, 16, 256), [200, 77], False, 1 / math.sqrt(64)),
    ((2, 2, 40, 64), [64, 33], True, 0.3),       # bottom-right causal, Tq < Tk
    ((1, 2, 8, 100), [61], True, 0.125),         # ragged: looped path
    ((1, 1, 3, 5000), [4000], False, 0.05),      # beyond the register buckets
])
def test_scaled_softmax_forward_and_masked_backward(dtype, shape, lengths, causal, scale):
    L = _L()
    B, H, Tq, Tk = shape
    x, dout, mask = _rand_problem(B, H, Tq, Tk, dtype, 71, lengths)
    # a non-binary additive bias on the valid keys, -inf on the padding
    g = torch.Generator(device=DEV).manual_seed(72)
    bias = torch.randn(B, Tk, generator=g, device=DEV).to(mask.dtype)
    mask = torch.where(torch.isinf(mask.float()), mask, bias)
    y = L.softmax_fw(x, mask, causal=causal, scale=scale)
    torch.cuda.synchronize()
    ref = oracle.softmax_fw_tensor_scaled(x.cpu(), mask.cpu(), causal=causal, scale=scale)
    compare(y, ref, dtype, f"scaled fw {shape}")
    assert np.all(y.cpu().float().numpy()[ref == 0.0] == 0.0)
    yin = torch.from_numpy(ref).to(_dt(dtype)).to(DEV)
    dx = L.softmax_bw_masked(dout, yin, mask, causal=causal, scale=scale)
    torch.cuda.synchronize()
    want = oracle.softmax_bw_masked_scaled_tensor(dout.cpu(), yin.cpu(), mask.cpu(),
                                                  causal=causal, scale=scale)
    compare(dx, want, dtype, f"scaled masked bw {shape}")
    # scale 1 is the unscaled entry point, bit for bit
    assert torch.equal(L.softmax_fw(x, mask, causal=causal, scale=1.0),
                       L.softmax_fw(x, mask, causal=causal))
    assert torch.equal(L.softmax_bw_masked(dout, yin, mask, causal=causal, scale=1.0),
                       L.softmax_bw_masked(dout, yin, mask, causal=causal))


def test_scaled_softmax_encoder_big_sampled():
    """The Transformer-big encoder shape with the 1/sqrt(64) score scale."""
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    s = W.ENCODER_BIG["softmax"]
    inp = W.softmax_inputs(s, device=DEV)
    scale = 0.125
    y = L.softmax_fw(inp["scores"], inp["mask"], scale=scale)
    torch.cuda.synchronize()
    rows = sample_rows(s.rows, boundaries=[b * s.H * s.T for b in range(1, s.B)], seed=9)
    xr = take_rows(inp["scores"], rows)
    ref = oracle.softmax_fw_scaled(xr, inp["mask"].cpu(), batch=rows // (s.H * s.T), scale=scale)
    compare(take_rows(y, rows), ref, s.dtype, "encoder scaled fw")


# ----------------------------------------------------------------------------
# RMSNorm (FastTransformer page, section 5.4)
# ----------------------------------------------------------------------------

def check_rmsnorm(case, full=True, seed=0, eps=1e-6):
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    inp = W.layernorm_inputs(case, device=DEV)
    x, g, dy = inp["x"], inp["gamma"], inp["dy"]
    y, rstd = L.rmsnorm_fw(x, g, eps)
    torch.cuda.synchronize()
    R, N = x.shape
    rows = np.arange(R) if full else sample_rows(R, seed=seed)
    yr, rr = oracle.rmsnorm_fw(take_rows(x, rows), g.cpu(), eps)
    compare(take_rows(y, rows), yr, case.dtype, f"{case.name} rms y")
    compare(rstd.cpu()[rows], rr, case.dtype, f"{case.name} rms rstd")
    # backward inputs: the oracle's rstd of every row, stored as fp32
    r_all = np.concatenate([oracle.rmsnorm_fw(x[r0:r0 + 2048].cpu(), g.cpu(), eps)[1]
                            for r0 in range(0, R, 2048)])
    rstd_in = torch.from_numpy(r_all).float().to(DEV)
    dx = L.rmsnorm_bw_dinp(dy, x, g, rstd_in)
    dg = L.rmsnorm_bw_dgamma(dy, x, rstd_in)
    torch.cuda.synchronize()
    compare(take_rows(dx, rows), oracle.rmsnorm_bw_dinp(take_rows(dy, rows), take_rows(x, rows),
                                                        g.cpu(), rstd_in.cpu()[rows]),
            case.dtype, f"{case.name} rms dx")
    cols = np.arange(N) if full else np.unique(np.concatenate(
        [np.arange(min(8, N)), np.arange(max(0, N - 8), N),
         np.random.default_rng(seed).integers(0, N, size=48)]))
    ci = torch.from_numpy(cols).to(DEV)
    want = oracle.rmsnorm_bw_dgamma(dy.index_select(1, ci).cpu(), x.index_select(1, ci).cpu(),
                                    rstd_in.cpu())
    compare(dg.cpu()[cols], want, case.dtype, f"{case.name} rms dgamma")


@pytest.mark.parametrize("N", [768, 1024, 4096, 8192])
def test_rmsnorm_width_sweep_bf16(N):
    from transformer_reduce_gb300 import workloads as W
    case = [c for c in W.LAYERNORM_SWEEP if c.hidden == N][0]
    check_rmsnorm(case, full=False, seed=N)


def test_rmsnorm_small_configs():
    from transformer_reduce_gb300 import workloads as W
    check_rmsnorm(W.TINY["layernorm"], full=True)
    check_rmsnorm(W.GPT2_SMALL["layernorm"], full=True)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [1, 7, 8, 24, 32, 100, 770, 1536, 20000])
def test_rmsnorm_odd_widths(dtype, N):
    check_rmsnorm(_ln_case(21, N, dtype), full=True)


def test_rmsnorm_in_place_gradient_and_zero_rows():
    L = _L()
    from transformer_reduce_gb300 import workloads as W
    lc = _ln_case(40, 1024, "bf16")
    li = W.layernorm_inputs(lc, device=DEV)
    _, r = oracle.rmsnorm_fw(li["x"].cpu(), li["gamma"].cpu(), 1e-6)
    rt = torch.from_numpy(r).float().to(DEV)
    dy = li["dy"].clone()
    want = oracle.rmsnorm_bw_dinp(dy.cpu(), li["x"].cpu(), li["gamma"].cpu(), rt.cpu())
    L.rmsnorm_bw_dinp(dy, li["x"], li["gamma"], rt, dx=dy)
    torch.cuda.synchronize()
    compare(dy, want, "bf16", "in-place rms dx")
    xe = torch.empty(0, 64, device=DEV, dtype=torch.bfloat16)
    dg = L.rmsnorm_bw_dgamma(xe, xe, torch.empty(0, device=DEV),
                             dgamma=torch.full((64,), 5.0, device=DEV))
    torch.cuda.synchronize()
    assert torch.all(dg == 0)


# ----------------------------------------------------------------------------
# fused LayerNorm backward: dx, dgamma, dbeta from one read of dy and x
# ----------------------------------------------------------------------------

def check_ln_bw_fused(case, full=True, seed=0):
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    inp = W.layernorm_inputs(case, device=DEV)
    x, g, b, dy = inp["x"], inp["gamma"], inp["beta"], inp["dy"]
    R, N = x.shape
    m_all, r_all = oracle_ln_stats(x, g, b, case.eps)
    mean_in = torch.from_numpy(m_all).float().to(DEV)
    rstd_in = torch.from_numpy(r_all).float().to(DEV)
    dx, dgm, dbt = L.layernorm_bw(dy, x, g, mean_in, rstd_in)
    torch.cuda.synchronize()
    rows = np.arange(R) if full else sample_rows(R, seed=seed)
    refdx = oracle.layernorm_bw_dinp(take_rows(dy, rows), take_rows(x, rows), g.cpu(),
                                     mean_in.cpu()[rows], rstd_in.cpu()[rows])
    compare(take_rows(dx, rows), refdx, case.dtype, f"{case.name} fused dx")
    cols = np.arange(N) if full else np.unique(np.concatenate(
        [np.arange(min(8, N)), np.arange(max(0, N - 8), N),
         np.random.default_rng(seed).integers(0, N, size=48)]))
    ci = torch.from_numpy(cols).to(DEV)
    rg, rb = oracle.layernorm_bw_dgamma_dbeta(dy.index_select(1, ci).cpu(),
                                              x.index_select(1, ci).cpu(),
                                              mean_in.cpu(), rstd_in.cpu())
    compare(dgm.cpu()[cols], rg, case.dtype, f"{case.name} fused dgamma")
    compare(dbt.cpu()[cols], rb, case.dtype, f"{case.name} fused dbeta")
    return dy, x, g, mean_in, rstd_in, (dx, dgm, dbt)


@pytest.mark.parametrize("N", [768, 1024, 4096, 8192])
def test_ln_bw_fused_width_sweep_bf16(N):
    from transformer_reduce_gb300 import workloads as W
    case = [c for c in W.LAYERNORM_SWEEP if c.hidden == N][0]
    check_ln_bw_fused(case, full=False, seed=N)


def test_ln_bw_fused_small_configs_and_encoder():
    from transformer_reduce_gb300 import workloads as W
    check_ln_bw_fused(W.TINY["layernorm"], full=True)
    check_ln_bw_fused(W.GPT2_SMALL["layernorm"], full=True)
    check_ln_bw_fused(W.ENCODER_BIG["layernorm"][1], full=False, seed=5)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("rows,N", [(1, 64), (7, 1024), (303, 256), (304, 512), (305, 768),
                                    (1000, 2048), (333, 8192), (9, 16384), (21, 7), (21, 770),
                                    (21, 20000), (77, 8), (77, 24), (77, 32)])
def test_ln_bw_fused_ragged_chunks_and_widths(dtype, rows, N):
    # row counts around the 304-chunk cut (one row per chunk, a ragged last
    # chunk) and widths that take the scalar two-kernel path
    check_ln_bw_fused(_ln_case(rows, N, dtype), full=True)


def test_ln_bw_fused_is_bitwise_reproducible_and_in_place():
    L = _L()
    case = _ln_case(4099, 1024, "bf16")
    dy, x, g, m, r, (dx0, dg0, db0) = check_ln_bw_fused(case, full=False, seed=3)
    for _ in range(2):
        dx1, dg1, db1 = L.layernorm_bw(dy, x, g, m, r)
        torch.cuda.synchronize()
        assert torch.equal(dx0, dx1) and torch.equal(dg0, dg1) and torch.equal(db0, db1)
    # dx written over dy
    d = dy.clone()
    L.layernorm_bw(d, x, g, m, r, dx=d)
    torch.cuda.synchronize()
    assert torch.equal(d, dx0)


def test_ln_bw_fused_zero_rows_and_workspace_rejection():
    L = _L()
    xe = torch.empty(0, 64, device=DEV, dtype=torch.bfloat16)
    _, dg, db = L.layernorm_bw(xe, xe, torch.ones(64, device=DEV, dtype=torch.bfloat16),
                               torch.empty(0, device=DEV), torch.empty(0, device=DEV),
                               dgamma=torch.full((64,), 7.0, device=DEV),
                               dbeta=torch.full((64,), 7.0, device=DEV))
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)
    case = _ln_case(4096, 1024, "bf16")
    from transformer_reduce_gb300 import workloads as W
    li = W.layernorm_inputs(case, device=DEV)
    m = torch.zeros(4096, device=DEV)
    need = L.ls_layernorm_bw_workspace_size(4096, 1024)
    small = torch.empty(need // 4 - 1, device=DEV)
    with pytest.raises(L.LsError):
        L.layernorm_bw(li["dy"], li["x"], li["gamma"], m, m, workspace=small)


# ----------------------------------------------------------------------------
# mask forms: the kernels classify each batch entry's mask row as a window of
# visible keys or as "general"; every form must give the oracle's result
# ----------------------------------------------------------------------------

def _mask_forms(B, Tk, dt, seed):
    """[B, Tk] additive masks cycling through the forms the kernels tell
    apart: right padding (with -0.0 among the visible keys), left padding, a
    window in the middle, -inf holes inside the visible keys, finite biases
    with right padding, nothing visible, and no padding at all."""
    g = torch.Generator().manual_seed(seed)
    m = torch.zeros(B, Tk)
    for b in range(B):
        form = b % 7
        lo = int(torch.randint(1, max(2, Tk // 3), (1,), generator=g))
        hi = int(torch.randint(max(lo + 1, Tk // 2), Tk, (1,), generator=g))
        if form == 0:
            m[b, hi:] = -math.inf
            m[b, 1:hi:5] = -0.0
        elif form == 1:
            m[b, :lo] = -math.inf
        elif form == 2:
            m[b, :lo] = -math.inf
            m[b, hi:] = -math.inf
        elif form == 3:
            m[b, hi:] = -math.inf
            m[b, lo:lo + 3] = -math.inf
        elif form == 4:
            m[b] = torch.randn(Tk, generator=g)
            m[b, hi:] = -math.inf
        elif form == 5:
            m[b] = -math.inf
    return m.to(dt).to(DEV)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("H,Tq,Tk,causal", [
    (2, 16, 256, False), (2, 64, 64, True), (1, 40, 512, True),   # Tq < Tk: bottom-right
    (2, 8, 1000, False),                                          # ragged chunk count
    (2, 8, 100, True),                                            # 16-bit: looped path
])
def test_softmax_mask_forms(dtype, H, Tq, Tk, causal):
    """Forward, scaled forward and masked backward (with garbage at invisible
    keys) on every mask form, each against the oracle."""
    L = _L()
    dt = _dt(dtype)
    B = 14
    g = torch.Generator(device=DEV).manual_seed(Tk + Tq)
    x = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).mul(3).to(dt)
    dout = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).to(dt)
    mask = _mask_forms(B, Tk, dt, seed=Tk)
    y = L.softmax_fw(x, mask, causal=causal)
    ys = L.softmax_fw(x, mask, causal=causal, scale=0.3)
    torch.cuda.synchronize()
    ref = oracle.softmax_fw_tensor_offset(x.cpu(), mask.cpu(), causal=causal)
    compare(y, ref, dtype, f"mask forms fw {Tq}x{Tk}")
    assert np.all(y.cpu().float().numpy()[ref == 0.0] == 0.0)
    refs = oracle.softmax_fw_tensor_scaled(x.cpu(), mask.cpu(), causal=causal, scale=0.3)
    compare(ys, refs, dtype, f"mask forms scaled fw {Tq}x{Tk}")
    invisible = torch.from_numpy(ref == 0.0).to(DEV)
    y_in = torch.from_numpy(ref).to(dt).to(DEV)
    y_dirty = torch.where(invisible, torch.full_like(y_in, 5.0), y_in)
    d_dirty = torch.where(invisible, torch.full_like(dout, float("nan")), dout)
    dx = L.softmax_bw_masked(d_dirty, y_dirty, mask, causal=causal)
    torch.cuda.synchronize()
    want = oracle.softmax_bw_masked_tensor(torch.nan_to_num(d_dirty, nan=0.0).cpu(),
                                           y_dirty.cpu(), mask.cpu(), causal=causal)
    compare(dx, want, dtype, f"mask forms masked bw {Tq}x{Tk}")
    assert torch.all(dx[invisible] == 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("H,Tq", [(1, 1), (1, 2), (2, 3)])
def test_softmax_many_batch_entries_per_block(dtype, H, Tq):
    """A block whose rows span more batch entries than it classifies (one or
    two rows per entry) treats every mask row as general; results as the
    oracle's for every form."""
    L = _L()
    dt = _dt(dtype)
    B, Tk = 700, 64
    g = torch.Generator(device=DEV).manual_seed(B + H + Tq)
    x = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).mul(3).to(dt)
    dout = torch.randn(B, H, Tq, Tk, generator=g, device=DEV).to(dt)
    mask = _mask_forms(B, Tk, dt, seed=B + Tq)
    y = L.softmax_fw(x, mask, causal=False)
    torch.cuda.synchronize()
    ref = oracle.softmax_fw_tensor(x.cpu(), mask.cpu())
    compare(y, ref, dtype, f"many entries fw H={H} Tq={Tq}")
    y_in = torch.from_numpy(ref).to(dt).to(DEV)
    dx = L.softmax_bw_masked(dout, y_in, mask)
    torch.cuda.synchronize()
    compare(dx, oracle.softmax_bw_masked_tensor(dout.cpu(), y_in.cpu(), mask.cpu()), dtype,
            f"many entries masked bw H={H} Tq={Tq}")
