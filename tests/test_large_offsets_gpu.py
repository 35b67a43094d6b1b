"""GPU parity at sizes past 32-bit offsets: more than 2^32 elements in one
tensor, and more than 2^31 rows.

Row and element offsets are 64-bit throughout the library; the register
pipelines of the softmax forward and the masked backward use 32-bit row
cursors and hand problems of more than 2^31 - 1 rows to the looped kernels.
These cases check rows whose element offsets lie past 2^31 and 2^32 (and rows
past index 2^31) against the fp64 oracle, on sampled rows, and the column
sums over every row on sampled columns.  Inputs are seeded and synthetic;
backward inputs never come from the GPU.  The largest case holds about
103 GB on the device.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import compare, oracle_softmax_rows, sample_rows, take_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

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
    torch.cuda.empty_cache()
    yield L
    torch.cuda.empty_cache()


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _need(nbytes):
    free, _ = torch.cuda.mem_get_info(0)
    if free < nbytes:
        pytest.skip(f"needs {nbytes / 1e9:.0f} GB free on the device, {free / 1e9:.0f} GB are")


def test_softmax_past_2_pow_32_elements(lib):
    """[65, 16, 2048, 2048] bf16 (4.36e9 elements) with a padding mask: the
    register pipelines, rows at element offsets 2^31 and 2^32 and the last."""
    L = lib
    B, H, T = 65, 16, 2048
    _need(64 << 30)
    rows_n = B * H * T
    g = _gen(101)
    lengths = torch.randint(T // 2, T + 1, (B,), generator=torch.Generator().manual_seed(102))
    mask = torch.zeros(B, T)
    for b, n in enumerate(lengths.tolist()):
        mask[b, n:] = -float("inf")
    mask = mask.to(torch.bfloat16).to(DEV)
    x = torch.randn(B, H, T, T, generator=g, device=DEV, dtype=torch.bfloat16).mul_(3.0)
    y = L.softmax_fw(x, mask)
    torch.cuda.synchronize()
    edges = [b * H * T for b in range(1, B)] + [(1 << 31) // T, (1 << 32) // T]
    rows = sample_rows(rows_n, boundaries=edges, k=128, seed=103)
    assert rows.max() * T >= (1 << 32)
    compare(take_rows(y, rows), oracle_softmax_rows(x, mask, rows, False), "bf16",
            "past-2^32 softmax_fw")
    del x, y
    torch.cuda.empty_cache()

    # backward inputs: probability-like y (0 on masked keys), dout ~ N(0, 1)
    yin = torch.rand(B, H, T, T, generator=g, device=DEV, dtype=torch.bfloat16).mul_(2.0 / T)
    yin.mul_((mask == 0).to(torch.bfloat16).view(B, 1, 1, T))
    dout = torch.randn(B, H, T, T, generator=g, device=DEV, dtype=torch.bfloat16)
    dx = L.softmax_bw(dout, yin)
    torch.cuda.synchronize()
    compare(take_rows(dx, rows), oracle.softmax_bw(take_rows(dout, rows), take_rows(yin, rows)),
            "bf16", "past-2^32 softmax_bw")
    L.softmax_bw_masked(dout, yin, mask, dinp=dx)
    torch.cuda.synchronize()
    want = oracle.softmax_bw_masked(take_rows(dout, rows), take_rows(yin, rows), mask.cpu(),
                                    batch=rows // (H * T))
    compare(take_rows(dx, rows), want, "bf16", "past-2^32 masked bw")


def test_softmax_past_2_pow_31_rows(lib):
    """[1, 1, 2^31 + 40, 8] bf16: more rows than a 32-bit row cursor holds, so
    the forward and the masked backward take their looped kernels and the
    plain backward its register kernel with 64-bit rows."""
    L = lib
    Tq, Tk = (1 << 31) + 40, 8
    _need(110 << 30)
    g = _gen(111)
    mask = torch.tensor([[0.0] * 6 + [-float("inf")] * 2], dtype=torch.bfloat16, device=DEV)
    x = torch.randn(1, 1, Tq, Tk, generator=g, device=DEV, dtype=torch.bfloat16).mul_(3.0)
    y = L.softmax_fw(x, mask)
    torch.cuda.synchronize()
    rows = sample_rows(Tq, boundaries=[(1 << 31) - 1, 1 << 31], k=64, seed=112)
    assert rows.max() > (1 << 31)
    compare(take_rows(y, rows), oracle_softmax_rows(x, mask, rows, False), "bf16",
            "past-2^31-rows softmax_fw")
    del x, y
    torch.cuda.empty_cache()

    yin = torch.rand(1, 1, Tq, Tk, generator=g, device=DEV, dtype=torch.bfloat16).mul_(1.0 / 3)
    yin[..., 6:] = 0
    dout = torch.randn(1, 1, Tq, Tk, generator=g, device=DEV, dtype=torch.bfloat16)
    dx = L.softmax_bw_masked(dout, yin, mask)
    torch.cuda.synchronize()
    want = oracle.softmax_bw_masked(take_rows(dout, rows), take_rows(yin, rows), mask.cpu(),
                                    batch=np.zeros_like(rows))
    compare(take_rows(dx, rows), want, "bf16", "past-2^31-rows masked bw")
    L.softmax_bw(dout, yin, dinp=dx)
    torch.cuda.synchronize()
    compare(take_rows(dx, rows), oracle.softmax_bw(take_rows(dout, rows), take_rows(yin, rows)),
            "bf16", "past-2^31-rows softmax_bw")


def test_layernorm_past_2_pow_32_elements(lib):
    """[2^22 + 3, 1024] bf16 (4.3e9 elements): forward and input gradient on
    sampled rows (element offsets past 2^31 and 2^32 and the last rows), the
    dgamma / dbeta column sums over every row on sampled columns, and the
    fused backward.  dy has mean 0.5 and the backward's saved statistics are
    seeded inputs (mean 1.0, rstd 0.5 +- 0.05) while x has mean 1.5, so the
    column sums stay far from zero and the relative rule applies to them."""
    L = lib
    R, N = (1 << 22) + 3, 1024
    _need(48 << 30)
    g = _gen(121)
    x = torch.randn(R, N, generator=g, device=DEV, dtype=torch.bfloat16).mul_(2.0).add_(1.5)
    gamma = torch.rand(N, generator=g, device=DEV, dtype=torch.bfloat16).add_(0.5)
    beta = torch.randn(N, generator=g, device=DEV, dtype=torch.bfloat16).mul_(0.1)
    eps = 1e-8
    y, mean, rstd = L.layernorm_fw(x, gamma, beta, eps)
    torch.cuda.synchronize()
    rows = sample_rows(R, boundaries=[(1 << 31) // N, (1 << 32) // N], k=128, seed=122)
    assert rows.max() * N >= (1 << 32)
    yr, mr, rr = oracle.layernorm_fw(take_rows(x, rows), gamma.cpu(), beta.cpu(), eps)
    compare(take_rows(y, rows), yr, "bf16", "past-2^32 ln_fw y")
    compare(mean.cpu()[rows], mr, "bf16", "past-2^32 ln_fw mean")
    compare(rstd.cpu()[rows], rr, "bf16", "past-2^32 ln_fw rstd")
    del y, mean, rstd
    torch.cuda.empty_cache()

    dy = torch.randn(R, N, generator=g, device=DEV, dtype=torch.bfloat16).add_(0.5)
    mean_in = torch.randn(R, generator=g, device=DEV).mul_(0.05).add_(1.0)
    rstd_in = torch.rand(R, generator=g, device=DEV).mul_(0.1).add_(0.45)
    mean_h, rstd_h = mean_in.cpu(), rstd_in.cpu()
    cols = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N),
                                     np.random.default_rng(123).integers(0, N, size=48)]))
    ci = torch.from_numpy(cols).to(DEV)
    want_g, want_b = oracle.layernorm_bw_dgamma_dbeta(dy.index_select(1, ci).cpu(),
                                                      x.index_select(1, ci).cpu(), mean_h, rstd_h)
    assert np.abs(want_g).min() > 1e4 and np.abs(want_b).min() > 1e4
    want_dx = oracle.layernorm_bw_dinp(take_rows(dy, rows), take_rows(x, rows), gamma.cpu(),
                                       mean_h[rows], rstd_h[rows])

    dx = L.layernorm_bw_dinp(dy, x, gamma, mean_in, rstd_in)
    dgm, dbt = L.layernorm_bw_dgamma_dbeta(dy, x, mean_in, rstd_in)
    torch.cuda.synchronize()
    compare(take_rows(dx, rows), want_dx, "bf16", "past-2^32 ln_dinp")
    compare(dgm.cpu()[cols], want_g, "bf16", "past-2^32 ln_dgamma")
    compare(dbt.cpu()[cols], want_b, "bf16", "past-2^32 ln_dbeta")

    dx.zero_()
    dx, dgm, dbt = L.layernorm_bw(dy, x, gamma, mean_in, rstd_in, dx=dx)
    torch.cuda.synchronize()
    compare(take_rows(dx, rows), want_dx, "bf16", "past-2^32 fused ln bw dx")
    compare(dgm.cpu()[cols], want_g, "bf16", "past-2^32 fused ln bw dgamma")
    compare(dbt.cpu()[cols], want_b, "bf16", "past-2^32 fused ln bw dbeta")
