"""Helpers of the GPU parity tests: the tolerance rule, row sampling, and
oracle calls on row blocks (so full-size problems never need the whole tensor
in float64 on the host).

Tolerance rule (|gpu - ref| <= atol + rtol * |ref|, ref = the fp64 oracle):
  * atol = rtol = 1e-5 when the configuration stores fp32, 1e-3 when it stores
    fp16 or bf16 (the HW4 page's kernel-test tolerance).  fp32 outputs of a
    16-bit configuration (mean, rstd, dgamma, dbeta) take the configuration's
    tolerance.
  * bf16 outputs may instead be within one bf16 step of the oracle's value
    rounded to bf16: the storage step alone (2^-8 relative) exceeds 1e-3 for
    |ref| above ~0.34, so a correctly rounded result can miss the literal rule.
    Both counts are reported.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle


def tolerance(cfg_dtype: str) -> float:
    return 1e-5 if cfg_dtype == "f32" else 1e-3


def _key16(t: torch.Tensor) -> torch.Tensor:
    bits = t.contiguous().view(torch.int16).to(torch.int32) & 0xFFFF
    return torch.where((bits & 0x8000) != 0, -(bits & 0x7FFF), bits)


# Error statistics of every comparison of the session, written out as JSON
# lines by conftest.py when LS_PARITY_REPORT names a file.
REPORT = []


def compare(gpu: torch.Tensor, ref: np.ndarray, cfg_dtype: str, what: str) -> dict:
    """Assert the tolerance rule element by element; return error statistics."""
    gpu = gpu.detach().cpu()
    ref = np.asarray(ref, dtype=np.float64).reshape(tuple(gpu.shape))
    g = gpu.to(torch.float64).numpy()
    tol = tolerance(cfg_dtype)
    err = np.abs(g - ref)
    strict = err <= tol + tol * np.abs(ref)
    ok = strict.copy()
    max_ulp = 0
    if gpu.dtype == torch.bfloat16:
        r16 = torch.from_numpy(ref).to(torch.bfloat16)
        d = (_key16(gpu) - _key16(r16)).abs().numpy()
        # reported over the values the absolute tolerance does not cover
        # (near zero a bf16 step is tiny and the step count meaningless)
        big = np.abs(ref) >= tol
        max_ulp = int(d[big].max()) if np.any(big) else 0
        ok |= d <= 1
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    n_bad = int((~ok).sum())
    if n_bad:
        idx = np.argwhere(~ok)[:5]
        detail = [(tuple(int(v) for v in i), float(g[tuple(i)]), float(ref[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {n_bad}/{ok.size} elements out of tolerance, e.g. {detail}")
    rel = err / np.maximum(np.abs(ref), np.finfo(np.float64).tiny)
    stats = {"what": what, "cfg_dtype": cfg_dtype, "out_dtype": str(gpu.dtype).replace("torch.", ""),
             "n": int(ok.size), "strict_frac": float(strict.mean()) if ok.size else 1.0,
             "max_abs": float(err.max()) if err.size else 0.0,
             "max_rel_where_ref_ge_1e-3": float(rel[np.abs(ref) >= 1e-3].max())
             if np.any(np.abs(ref) >= 1e-3) else 0.0,
             "max_bf16_steps": max_ulp, "tol": tol}
    REPORT.append(stats)
    return stats


def sample_rows(nrows: int, boundaries=(), k: int = 192, seed: int = 0) -> np.ndarray:
    """Sorted unique row indices: the first and last rows, rows around the
    given boundaries (e.g. batch edges), and k seeded random rows."""
    rng = np.random.default_rng(seed)
    pick = set(range(min(8, nrows))) | set(range(max(0, nrows - 8), nrows))
    for b in boundaries:
        pick |= {r for r in (b - 2, b - 1, b, b + 1) if 0 <= r < nrows}
    pick |= set(rng.integers(0, nrows, size=min(k, nrows)).tolist())
    return np.array(sorted(pick), dtype=np.int64)


def oracle_softmax_rows(x4: torch.Tensor, mask, rows: np.ndarray, causal: bool) -> np.ndarray:
    """Oracle softmax forward of the listed rows of a [B,H,Tq,Tk] tensor."""
    B, H, Tq, Tk = x4.shape
    flat = x4.reshape(-1, Tk)
    idx = torch.from_numpy(rows).to(flat.device)
    xr = flat.index_select(0, idx).cpu()
    return oracle.softmax_fw(xr, None if mask is None else mask.cpu(),
                             batch=rows // (H * Tq), query=rows % Tq, causal=causal)


def oracle_softmax_all(x4: torch.Tensor, mask, causal: bool, block: int = 8192) -> np.ndarray:
    """Oracle softmax forward of every row (row blocks of `block`)."""
    B, H, Tq, Tk = x4.shape
    n = B * H * Tq
    out = np.empty((n, Tk))
    for r0 in range(0, n, block):
        rows = np.arange(r0, min(n, r0 + block), dtype=np.int64)
        out[r0:r0 + len(rows)] = oracle_softmax_rows(x4, mask, rows, causal)
    return out.reshape(B, H, Tq, Tk)


def take_rows(t: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    flat = t.reshape(-1, t.shape[-1])
    return flat.index_select(0, torch.from_numpy(rows).to(flat.device)).cpu()


def oracle_ln_stats(x: torch.Tensor, gamma, beta, eps: float, block: int = 1024):
    """Oracle LayerNorm mean / rstd of every row, computed in row blocks."""
    rows = x.shape[0]
    mean = np.empty(rows)
    rstd = np.empty(rows)
    g, b = gamma.cpu(), beta.cpu()
    for r0 in range(0, rows, block):
        xr = x[r0:r0 + block].cpu()
        _, m, r = oracle.layernorm_fw(xr, g, b, eps)
        mean[r0:r0 + len(m)] = m
        rstd[r0:r0 + len(r)] = r
    return mean, rstd
