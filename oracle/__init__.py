"""CPU oracle for the softmax / LayerNorm reduce path (TEST INFRASTRUCTURE).

This package is the checker, not the product.  Only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it; the library ``transformer_reduce_gb300`` never does, and the two
share no code.  The arithmetic lives in ``ref_reduce.c`` (plain C, double
precision, the textbook definitions); this module compiles it with gcc and
marshals numpy arrays in and out.  Every value that reaches the C code is
converted exactly to float64 (fp32, fp16 and bf16 values are all doubles),
so both sides of a parity test see the same numbers.

Sources are cited in ``ref_reduce.c``: the pages "CMU 11-868 L10:
Accelerating Transformers on GPUs, and Where LightSeq Finds the Time"
(section "Technique 2", slides 21-24) and "CMU 11-868 HW4：把 Softmax 與
LayerNorm 寫成 CUDA 融合 kernel" (Problems 1.1-2.2 and the test baseline
softmax(inp + mask)); the L10 page's "Technique 1" (slide 12) for the cross
entropy reduce kernel, and the FastTransformer page's section 5.4 for RMSNorm.

Every function here is pinned by ``tests/test_oracle_pins.py`` to facts that
do not come from the oracle itself (closed forms, invariants, finite
differences, library routines); no function is left "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_reduce.c")
_LIB_PATH = os.path.join(_HERE, "libref_reduce.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add, so x86 and Arm builds round alike.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile ``ref_reduce.c`` into ``libref_reduce.so`` (gcc); return its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # REF_REDUCE_LIB: a deliberately broken copy of the oracle, built by the
        # mutation test to show that the pins reject it.
        lib = ctypes.CDLL(os.environ.get("REF_REDUCE_LIB") or build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.ref_softmax_fw.argtypes = [dp, dp, dp, ip, ip, i64, i64, ctypes.c_int]
        lib.ref_softmax_fw.restype = None
        lib.ref_softmax_bw.argtypes = [dp, dp, dp, i64, i64]
        lib.ref_softmax_bw.restype = None
        lib.ref_softmax_fw_offset.argtypes = [dp, dp, dp, ip, ip, i64, i64, ctypes.c_int, i64]
        lib.ref_softmax_fw_offset.restype = None
        lib.ref_softmax_bw_masked.argtypes = [dp, dp, dp, dp, ip, ip, i64, i64, ctypes.c_int, i64]
        lib.ref_softmax_bw_masked.restype = None
        lib.ref_softmax_fw_scaled.argtypes = [dp, dp, dp, ip, ip, i64, i64, ctypes.c_int, i64,
                                              ctypes.c_double]
        lib.ref_softmax_fw_scaled.restype = None
        lib.ref_softmax_bw_masked_scaled.argtypes = [dp, dp, dp, dp, ip, ip, i64, i64,
                                                     ctypes.c_int, i64, ctypes.c_double]
        lib.ref_softmax_bw_masked_scaled.restype = None
        lib.ref_layernorm_fw.argtypes = [dp, dp, dp, dp, dp, dp, i64, i64,
                                         ctypes.c_double]
        lib.ref_layernorm_fw.restype = None
        lib.ref_variance_one_pass.argtypes = [dp, i64, ctypes.c_int]
        lib.ref_variance_one_pass.restype = ctypes.c_double
        lib.ref_variance_two_pass.argtypes = [dp, i64]
        lib.ref_variance_two_pass.restype = ctypes.c_double
        lib.ref_layernorm_bw_dinp.argtypes = [dp, dp, dp, dp, dp, dp, i64, i64]
        lib.ref_layernorm_bw_dinp.restype = None
        lib.ref_layernorm_bw_dgamma_dbeta.argtypes = [dp, dp, dp, dp, dp, dp,
                                                      i64, i64]
        lib.ref_layernorm_bw_dgamma_dbeta.restype = None
        lib.ref_rmsnorm_fw.argtypes = [dp, dp, dp, dp, i64, i64, ctypes.c_double]
        lib.ref_rmsnorm_fw.restype = None
        lib.ref_rmsnorm_bw_dinp.argtypes = [dp, dp, dp, dp, dp, i64, i64]
        lib.ref_rmsnorm_bw_dinp.restype = None
        lib.ref_rmsnorm_bw_dgamma.argtypes = [dp, dp, dp, dp, i64, i64]
        i32p = ctypes.POINTER(ctypes.c_int32)
        lib.ref_cross_entropy_fw.argtypes = [dp, dp, dp, i32p, i64, i64]
        lib.ref_cross_entropy_fw.restype = None
        lib.ref_cross_entropy_bw.argtypes = [dp, dp, i32p, dp, dp, i64, i64]
        lib.ref_cross_entropy_bw.restype = None
        lib.ref_rmsnorm_bw_dgamma.restype = None
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    """Exact conversion of a numpy / torch array to a C-contiguous float64 array."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen on the torch side (bf16 has no numpy dtype)
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def softmax_fw(x, mask=None, batch=None, query=None, causal=False):
    """Softmax of (scores + additive mask) over the last axis, per listed row.

    x      : [nrows, Tk] scores (each row one (b, h, i) of a [B,H,Tq,Tk] tensor)
    mask   : [B, Tk] additive mask or None
    batch  : [nrows] batch index b of each row (needed with a mask)
    query  : [nrows] query index i of each row (needed when causal)
    Returns y [nrows, Tk] float64.
    """
    x = _f64(x)
    nrows, tk = x.shape
    m = _f64(mask)
    if m is not None:
        assert m.ndim == 2 and m.shape[1] == tk
        batch = np.ascontiguousarray(np.asarray(batch, dtype=np.int64))
        assert batch.shape == (nrows,)
        assert batch.size == 0 or (batch.min() >= 0 and batch.max() < m.shape[0])
    if causal:
        query = np.ascontiguousarray(np.asarray(query, dtype=np.int64))
        assert query.shape == (nrows,)
    y = np.empty_like(x)
    _load().ref_softmax_fw(_ptr(y), _ptr(x), _ptr(m),
                           _ptr(batch if m is not None else None, ctypes.c_int64),
                           _ptr(query if causal else None, ctypes.c_int64),
                           nrows, tk, int(bool(causal)))
    return y


def softmax_fw_tensor(x4, mask=None, causal=False):
    """Softmax forward of a whole [B,H,Tq,Tk] tensor; returns [B,H,Tq,Tk] float64."""
    x4 = _f64(x4)
    B, H, Tq, Tk = x4.shape
    rows = np.arange(B * H * Tq, dtype=np.int64)
    y = softmax_fw(x4.reshape(-1, Tk), mask, batch=rows // (H * Tq),
                   query=rows % Tq, causal=causal)
    return y.reshape(B, H, Tq, Tk)


def softmax_bw(dy, y):
    """dx = y * (dy - sum(y * dy)) per row; dy, y [nrows, Tk] -> dx float64."""
    dy, y = _f64(dy), _f64(y)
    assert dy.shape == y.shape
    tk = dy.shape[-1]
    nrows = dy.size // tk if tk else 0
    dx = np.empty_like(dy)
    _load().ref_softmax_bw(_ptr(dx), _ptr(dy), _ptr(y), nrows, tk)
    return dx


def _rows_meta(nrows, mask, batch, query, causal):
    if mask is not None:
        batch = np.ascontiguousarray(np.asarray(batch, dtype=np.int64))
        assert batch.shape == (nrows,)
        assert batch.size == 0 or (batch.min() >= 0 and batch.max() < mask.shape[0])
    if causal:
        query = np.ascontiguousarray(np.asarray(query, dtype=np.int64))
        assert query.shape == (nrows,)
    return (_ptr(batch if mask is not None else None, ctypes.c_int64),
            _ptr(query if causal else None, ctypes.c_int64), batch, query)


def softmax_fw_offset(x, mask=None, batch=None, query=None, causal=False, offset=0):
    """Softmax forward, causal keys visible up to query + offset (Tk - Tq)."""
    x = _f64(x)
    nrows, tk = x.shape
    m = _f64(mask)
    pb, pq, batch, query = _rows_meta(nrows, m, batch, query, causal)
    y = np.empty_like(x)
    _load().ref_softmax_fw_offset(_ptr(y), _ptr(x), _ptr(m), pb, pq, nrows, tk,
                                  int(bool(causal)), int(offset))
    return y


def softmax_fw_tensor_offset(x4, mask=None, causal=False):
    """Softmax forward of [B,H,Tq,Tk], Tq <= Tk, bottom-right causal alignment."""
    x4 = _f64(x4)
    B, H, Tq, Tk = x4.shape
    rows = np.arange(B * H * Tq, dtype=np.int64)
    y = softmax_fw_offset(x4.reshape(-1, Tk), mask, batch=rows // (H * Tq), query=rows % Tq,
                          causal=causal, offset=Tk - Tq)
    return y.reshape(B, H, Tq, Tk)


def softmax_bw_masked(dy, y, mask=None, batch=None, query=None, causal=False, offset=0):
    """Softmax backward over the visible keys only (0 on masked / future keys)."""
    dy, y = _f64(dy), _f64(y)
    assert dy.shape == y.shape
    nrows, tk = dy.shape
    m = _f64(mask)
    pb, pq, batch, query = _rows_meta(nrows, m, batch, query, causal)
    dx = np.empty_like(dy)
    _load().ref_softmax_bw_masked(_ptr(dx), _ptr(dy), _ptr(y), _ptr(m), pb, pq, nrows, tk,
                                  int(bool(causal)), int(offset))
    return dx


def softmax_bw_masked_tensor(dy4, y4, mask=None, causal=False):
    """Masked softmax backward of [B,H,Tq,Tk] tensors (bottom-right causal)."""
    dy4, y4 = _f64(dy4), _f64(y4)
    B, H, Tq, Tk = dy4.shape
    rows = np.arange(B * H * Tq, dtype=np.int64)
    dx = softmax_bw_masked(dy4.reshape(-1, Tk), y4.reshape(-1, Tk), mask, batch=rows // (H * Tq),
                           query=rows % Tq, causal=causal, offset=Tk - Tq)
    return dx.reshape(B, H, Tq, Tk)


def softmax_fw_scaled(x, mask=None, batch=None, query=None, causal=False, offset=0, scale=1.0):
    """Softmax of scale * x + mask, causal keys visible up to query + offset."""
    x = _f64(x)
    nrows, tk = x.shape
    m = _f64(mask)
    pb, pq, batch, query = _rows_meta(nrows, m, batch, query, causal)
    y = np.empty_like(x)
    _load().ref_softmax_fw_scaled(_ptr(y), _ptr(x), _ptr(m), pb, pq, nrows, tk,
                                  int(bool(causal)), int(offset), float(scale))
    return y


def softmax_fw_tensor_scaled(x4, mask=None, causal=False, scale=1.0):
    """Scaled softmax forward of [B,H,Tq,Tk], Tq <= Tk, bottom-right causal."""
    x4 = _f64(x4)
    B, H, Tq, Tk = x4.shape
    rows = np.arange(B * H * Tq, dtype=np.int64)
    y = softmax_fw_scaled(x4.reshape(-1, Tk), mask, batch=rows // (H * Tq), query=rows % Tq,
                          causal=causal, offset=Tk - Tq, scale=scale)
    return y.reshape(B, H, Tq, Tk)


def softmax_bw_masked_scaled(dy, y, mask=None, batch=None, query=None, causal=False, offset=0,
                             scale=1.0):
    """Backward of the scaled softmax over the visible keys (0 elsewhere)."""
    dy, y = _f64(dy), _f64(y)
    assert dy.shape == y.shape
    nrows, tk = dy.shape
    m = _f64(mask)
    pb, pq, batch, query = _rows_meta(nrows, m, batch, query, causal)
    dx = np.empty_like(dy)
    _load().ref_softmax_bw_masked_scaled(_ptr(dx), _ptr(dy), _ptr(y), _ptr(m), pb, pq, nrows, tk,
                                         int(bool(causal)), int(offset), float(scale))
    return dx


def softmax_bw_masked_scaled_tensor(dy4, y4, mask=None, causal=False, scale=1.0):
    dy4, y4 = _f64(dy4), _f64(y4)
    B, H, Tq, Tk = dy4.shape
    rows = np.arange(B * H * Tq, dtype=np.int64)
    dx = softmax_bw_masked_scaled(dy4.reshape(-1, Tk), y4.reshape(-1, Tk), mask,
                                  batch=rows // (H * Tq), query=rows % Tq, causal=causal,
                                  offset=Tk - Tq, scale=scale)
    return dx.reshape(B, H, Tq, Tk)


def layernorm_fw(x, gamma, beta, eps):
    """Two-pass LayerNorm; returns (y, mean, rstd) in float64."""
    x, gamma, beta = _f64(x), _f64(gamma), _f64(beta)
    rows, n = x.shape
    assert gamma.shape == (n,) and beta.shape == (n,)
    y = np.empty_like(x)
    mean = np.empty(rows)
    rstd = np.empty(rows)
    _load().ref_layernorm_fw(_ptr(y), _ptr(mean), _ptr(rstd), _ptr(x),
                             _ptr(gamma), _ptr(beta), rows, n, float(eps))
    return y, mean, rstd


def variance_one_pass(row, single=False):
    """mu(x^2) - mu(x)^2 of one row, accumulated in double or float."""
    row = _f64(row).ravel()
    return _load().ref_variance_one_pass(_ptr(row), row.size, int(bool(single)))


def variance_two_pass(row):
    """Two-pass population variance of one row."""
    row = _f64(row).ravel()
    return _load().ref_variance_two_pass(_ptr(row), row.size)


def layernorm_bw_dinp(dy, x, gamma, mean, rstd):
    """Input gradient of LayerNorm given the saved row statistics."""
    dy, x, gamma, mean, rstd = map(_f64, (dy, x, gamma, mean, rstd))
    rows, n = x.shape
    assert dy.shape == x.shape and gamma.shape == (n,)
    assert mean.shape == (rows,) and rstd.shape == (rows,)
    dx = np.empty_like(x)
    _load().ref_layernorm_bw_dinp(_ptr(dx), _ptr(dy), _ptr(x), _ptr(gamma),
                                  _ptr(mean), _ptr(rstd), rows, n)
    return dx


def layernorm_bw_dgamma_dbeta(dy, x, mean, rstd):
    """Column sums dgamma = sum_r dy*xhat, dbeta = sum_r dy; returns float64 pair."""
    dy, x, mean, rstd = map(_f64, (dy, x, mean, rstd))
    rows, n = x.shape
    assert dy.shape == x.shape
    assert mean.shape == (rows,) and rstd.shape == (rows,)
    dgamma = np.empty(n)
    dbeta = np.empty(n)
    _load().ref_layernorm_bw_dgamma_dbeta(_ptr(dgamma), _ptr(dbeta), _ptr(dy),
                                          _ptr(x), _ptr(mean), _ptr(rstd), rows, n)
    return dgamma, dbeta


def rmsnorm_fw(x, gamma, eps):
    """RMSNorm: y = x * rsqrt(mean(x^2) + eps) * gamma; returns (y, rstd) float64."""
    x, gamma = _f64(x), _f64(gamma)
    rows, n = x.shape
    assert gamma.shape == (n,)
    y = np.empty_like(x)
    rstd = np.empty(rows)
    _load().ref_rmsnorm_fw(_ptr(y), _ptr(rstd), _ptr(x), _ptr(gamma), rows, n, float(eps))
    return y, rstd


def rmsnorm_bw_dinp(dy, x, gamma, rstd):
    """Input gradient of RMSNorm given the saved rstd."""
    dy, x, gamma, rstd = map(_f64, (dy, x, gamma, rstd))
    rows, n = x.shape
    assert dy.shape == x.shape and gamma.shape == (n,) and rstd.shape == (rows,)
    dx = np.empty_like(x)
    _load().ref_rmsnorm_bw_dinp(_ptr(dx), _ptr(dy), _ptr(x), _ptr(gamma), _ptr(rstd), rows, n)
    return dx


def rmsnorm_bw_dgamma(dy, x, rstd):
    """gamma gradient of RMSNorm: column sums of dy * x * rstd."""
    dy, x, rstd = map(_f64, (dy, x, rstd))
    rows, n = x.shape
    assert dy.shape == x.shape and rstd.shape == (rows,)
    dg = np.empty(n)
    _load().ref_rmsnorm_bw_dgamma(_ptr(dg), _ptr(dy), _ptr(x), _ptr(rstd), rows, n)
    return dg


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def cross_entropy_fw(z, target):
    """Softmax cross entropy of each row of z [rows, V] against its int32
    target class; returns (loss, lse) float64 [rows].  target < 0: ignored
    row (0, 0); target >= V: NaN."""
    z, target = _f64(z), _i32(target)
    rows, v = z.shape
    assert target.shape == (rows,)
    loss = np.empty(rows)
    lse = np.empty(rows)
    _load().ref_cross_entropy_fw(_ptr(loss), _ptr(lse), _ptr(z), _ptr(target, ctypes.c_int32),
                                 rows, v)
    return loss, lse


def cross_entropy_bw(z, target, lse, dloss):
    """dz = dloss * (softmax(z) - onehot(target)) from the saved log-sum-exp."""
    z, lse, dloss, target = _f64(z), _f64(lse), _f64(dloss), _i32(target)
    rows, v = z.shape
    assert target.shape == (rows,) and lse.shape == (rows,) and dloss.shape == (rows,)
    dz = np.empty_like(z)
    _load().ref_cross_entropy_bw(_ptr(dz), _ptr(z), _ptr(target, ctypes.c_int32), _ptr(lse),
                                 _ptr(dloss), rows, v)
    return dz
