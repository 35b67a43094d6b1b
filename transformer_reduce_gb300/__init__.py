"""transformer_reduce_gb300 -- fused softmax and LayerNorm reduce kernels of a
Transformer layer, forward and backward, for NVIDIA GB300 (sm_103a).

The compute is hand-written CUDA in ``libls_reduce.so`` behind a C ABI
(``include/ls_reduce.h``).  ``transformer_reduce_gb300._lib`` mirrors that ABI
one-for-one (raw pointers); the functions below are the PyTorch-facing
convenience layer: they check shapes, allocate outputs with torch, and pass
pointers and the current CUDA stream to the library.  There is no fallback:
if the library is missing or a call fails, they raise.
"""
from __future__ import annotations

from ._lib import (LS_BF16, LS_ERR_CUDA, ls_cross_entropy_bw, ls_cross_entropy_fw,
                   ls_softmax_bw_masked_scaled, ls_softmax_fw_scaled, LS_ERR_INVALID_ARG, LS_ERR_MISALIGNED,  # noqa: F401
                   LS_ERR_UNSUPPORTED, LS_ERR_WORKSPACE, LS_F16, LS_F32, LS_OK, LsError,
                   ls_layernorm_bw_dgamma_dbeta, ls_layernorm_bw_dgamma_dbeta_workspace_size,
                   ls_layernorm_bw, ls_layernorm_bw_dinp, ls_layernorm_bw_workspace_size,
                   ls_layernorm_fw, ls_rmsnorm_bw_dgamma,
                   ls_rmsnorm_bw_dinp, ls_rmsnorm_fw, ls_softmax_bw, ls_softmax_bw_masked,
                   ls_softmax_fw, load, status_string)

__all__ = [
    "softmax_fw", "softmax_bw", "softmax_bw_masked", "layernorm_fw", "layernorm_bw_dinp",
    "layernorm_bw_dgamma_dbeta", "dgamma_dbeta_workspace", "layernorm_bw", "rmsnorm_fw", "rmsnorm_bw_dinp",
    "rmsnorm_bw_dgamma", "cross_entropy_fw", "cross_entropy_bw", "LsError", "load",
    "ls_cross_entropy_fw", "ls_cross_entropy_bw", "ls_softmax_fw_scaled",
    "ls_softmax_bw_masked_scaled",
    "ls_softmax_fw", "ls_softmax_bw", "ls_softmax_bw_masked", "ls_layernorm_fw", "ls_layernorm_bw_dinp",
    "ls_layernorm_bw_dgamma_dbeta", "ls_layernorm_bw_dgamma_dbeta_workspace_size",
    "ls_layernorm_bw", "ls_layernorm_bw_workspace_size", "ls_rmsnorm_fw", "ls_rmsnorm_bw_dinp", "ls_rmsnorm_bw_dgamma",
]


def _torch():
    import torch
    return torch


def ls_dtype(t) -> int:
    torch = _torch()
    m = {torch.float32: LS_F32, torch.float16: LS_F16, torch.bfloat16: LS_BF16}
    if t.dtype not in m:
        raise TypeError(f"unsupported storage dtype {t.dtype} (float32, float16, bfloat16)")
    return m[t.dtype]


def _stream(t) -> int:
    torch = _torch()
    return torch.cuda.current_stream(t.device).cuda_stream


def _dev(*ts):
    """The one CUDA device all given tensors live on (None entries skipped);
    every tensor must be contiguous."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device (there is no CPU path)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on different devices ({dev} and {t.device})")
    return dev


def _want(name, t, shape, dtype):
    """Reject a tensor whose shape or dtype differs from what the kernels will
    read or write through its pointer (they trust the sizes they are given)."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} of shape {list(shape)}, "
                         f"got {t.dtype} of shape {list(t.shape)}")


def _workspace(name, t):
    torch = _torch()
    if t.dtype != torch.float32 or t.dim() != 1:
        raise ValueError(f"{name} must be a 1-D float32 tensor")


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _ok(status: int, where: str):
    if status != LS_OK:
        raise LsError(status, where)


def _call(where: str, dev, fn, *args):
    """Run one library call with ``dev`` as the current device (the library
    launches on the current device, on the stream it is given)."""
    with _torch().cuda.device(dev):
        _ok(fn(*args), where)


def _rows_hidden(x, name="x"):
    if x.dim() != 2:
        raise ValueError(f"{name} must be [rows, hidden]")
    return x.shape


def softmax_fw(scores, mask=None, causal: bool = False, out=None, scale=None):
    """Softmax over the last axis of scale * scores [B,H,Tq,Tk] plus an
    additive mask [B,Tk] (broadcast over heads and queries), future keys
    j > i + Tk - Tq masked when ``causal`` (Tq <= Tk).  ``scale`` None is 1.
    ``out`` may be ``scores`` (in place)."""
    torch = _torch()
    if scores.dim() != 4:
        raise ValueError("scores must be [B, H, Tq, Tk]")
    B, H, Tq, Tk = scores.shape
    _want("mask", mask, (B, Tk), scores.dtype)
    _want("out", out, scores.shape, scores.dtype)
    out = torch.empty_like(scores) if out is None else out
    dev = _dev(scores, mask, out)
    if scale is None:
        _call("ls_softmax_fw", dev, ls_softmax_fw, _ptr(out), _ptr(scores), _ptr(mask), B, H, Tq,
              Tk, causal, ls_dtype(scores), _stream(scores))
    else:
        _call("ls_softmax_fw_scaled", dev, ls_softmax_fw_scaled, _ptr(out), _ptr(scores),
              _ptr(mask), B, H, Tq, Tk, causal, float(scale), ls_dtype(scores), _stream(scores))
    return out


def softmax_bw(dout, out_fw, dinp=None):
    """Gradient of the softmax input from the output gradient ``dout`` and the
    forward output ``out_fw`` (both [B,H,Tq,Tk]).  ``dinp`` may be ``dout``."""
    torch = _torch()
    if dout.dim() != 4:
        raise ValueError("dout must be [B, H, Tq, Tk]")
    _want("out_fw", out_fw, dout.shape, dout.dtype)
    _want("dinp", dinp, dout.shape, dout.dtype)
    B, H, Tq, Tk = dout.shape
    dinp = torch.empty_like(dout) if dinp is None else dinp
    dev = _dev(dout, out_fw, dinp)
    _call("ls_softmax_bw", dev, ls_softmax_bw, _ptr(dinp), _ptr(dout), _ptr(out_fw), B, H, Tq, Tk,
          ls_dtype(dout), _stream(dout))
    return dinp


def softmax_bw_masked(dout, out_fw, mask=None, causal: bool = False, dinp=None, scale=None):
    """Softmax backward that reads only visible keys (mask != -inf, not in the
    causal future) and writes 0 on the others; with ``scale`` the gradient of
    the scores of ``softmax_fw(..., scale=scale)``."""
    torch = _torch()
    if dout.dim() != 4:
        raise ValueError("dout must be [B, H, Tq, Tk]")
    B, H, Tq, Tk = dout.shape
    _want("out_fw", out_fw, dout.shape, dout.dtype)
    _want("mask", mask, (B, Tk), dout.dtype)
    _want("dinp", dinp, dout.shape, dout.dtype)
    dinp = torch.empty_like(dout) if dinp is None else dinp
    dev = _dev(dout, out_fw, mask, dinp)
    if scale is None:
        _call("ls_softmax_bw_masked", dev, ls_softmax_bw_masked, _ptr(dinp), _ptr(dout),
              _ptr(out_fw), _ptr(mask), B, H, Tq, Tk, causal, ls_dtype(dout), _stream(dout))
    else:
        _call("ls_softmax_bw_masked_scaled", dev, ls_softmax_bw_masked_scaled, _ptr(dinp),
              _ptr(dout), _ptr(out_fw), _ptr(mask), B, H, Tq, Tk, causal, float(scale),
              ls_dtype(dout), _stream(dout))
    return dinp


def _stats(rows, x, **named):
    torch = _torch()
    for name, t in named.items():
        _want(name, t, (rows,), torch.float32)


def layernorm_fw(x, gamma, beta, eps: float = 1e-8, y=None, mean=None, rstd=None):
    """LayerNorm of x [rows, hidden]; returns (y, mean, rstd), the statistics fp32."""
    torch = _torch()
    rows, hidden = _rows_hidden(x)
    _want("gamma", gamma, (hidden,), x.dtype)
    _want("beta", beta, (hidden,), x.dtype)
    _want("y", y, x.shape, x.dtype)
    _stats(rows, x, mean=mean, rstd=rstd)
    y = torch.empty_like(x) if y is None else y
    mean = torch.empty(rows, device=x.device, dtype=torch.float32) if mean is None else mean
    rstd = torch.empty(rows, device=x.device, dtype=torch.float32) if rstd is None else rstd
    dev = _dev(x, gamma, beta, y, mean, rstd)
    _call("ls_layernorm_fw", dev, ls_layernorm_fw, _ptr(y), _ptr(mean), _ptr(rstd), _ptr(x),
          _ptr(gamma), _ptr(beta), rows, hidden, float(eps), ls_dtype(x), _stream(x))
    return y, mean, rstd


def layernorm_bw_dinp(dy, x, gamma, mean, rstd, dx=None):
    """Input gradient of LayerNorm from dy, x and the saved fp32 mean / rstd."""
    torch = _torch()
    rows, hidden = _rows_hidden(x)
    _want("dy", dy, x.shape, x.dtype)
    _want("gamma", gamma, (hidden,), x.dtype)
    _stats(rows, x, mean=mean, rstd=rstd)
    _want("dx", dx, x.shape, x.dtype)
    dx = torch.empty_like(x) if dx is None else dx
    dev = _dev(dy, x, gamma, mean, rstd, dx)
    _call("ls_layernorm_bw_dinp", dev, ls_layernorm_bw_dinp, _ptr(dx), _ptr(dy), _ptr(x),
          _ptr(gamma), _ptr(mean), _ptr(rstd), rows, hidden, ls_dtype(x), _stream(x))
    return dx


def dgamma_dbeta_workspace(rows: int, hidden: int, device):
    """A workspace tensor of the size ls_layernorm_bw_dgamma_dbeta needs."""
    torch = _torch()
    n = ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden)
    return torch.empty(max(n, 16) // 4, device=device, dtype=torch.float32)


def layernorm_bw_dgamma_dbeta(dy, x, mean, rstd, workspace=None, dgamma=None, dbeta=None):
    """gamma / beta gradients (fp32 [hidden]) summed over all rows, in a fixed
    order (bitwise reproducible)."""
    torch = _torch()
    rows, hidden = _rows_hidden(x)
    _want("dy", dy, x.shape, x.dtype)
    _stats(rows, x, mean=mean, rstd=rstd)
    _want("dgamma", dgamma, (hidden,), torch.float32)
    _want("dbeta", dbeta, (hidden,), torch.float32)
    if workspace is None:
        workspace = dgamma_dbeta_workspace(rows, hidden, x.device)
    _workspace("workspace", workspace)
    dgamma = torch.empty(hidden, device=x.device, dtype=torch.float32) if dgamma is None else dgamma
    dbeta = torch.empty(hidden, device=x.device, dtype=torch.float32) if dbeta is None else dbeta
    dev = _dev(dy, x, mean, rstd, workspace, dgamma, dbeta)
    _call("ls_layernorm_bw_dgamma_dbeta", dev, ls_layernorm_bw_dgamma_dbeta, _ptr(dgamma),
          _ptr(dbeta), _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), rows, hidden, _ptr(workspace),
          workspace.numel() * workspace.element_size(), ls_dtype(x), _stream(x))
    return dgamma, dbeta


def layernorm_bw(dy, x, gamma, mean, rstd, workspace=None, dx=None, dgamma=None, dbeta=None):
    """Whole LayerNorm backward in one pass over dy and x: returns
    (dx, dgamma, dbeta), the parameter gradients fp32 in a fixed order."""
    torch = _torch()
    rows, hidden = _rows_hidden(x)
    _want("dy", dy, x.shape, x.dtype)
    _want("gamma", gamma, (hidden,), x.dtype)
    _stats(rows, x, mean=mean, rstd=rstd)
    _want("dx", dx, x.shape, x.dtype)
    _want("dgamma", dgamma, (hidden,), torch.float32)
    _want("dbeta", dbeta, (hidden,), torch.float32)
    if workspace is None:
        n = ls_layernorm_bw_workspace_size(rows, hidden)
        workspace = torch.empty(max(n, 16) // 4, device=x.device, dtype=torch.float32)
    _workspace("workspace", workspace)
    dx = torch.empty_like(x) if dx is None else dx
    dgamma = torch.empty(hidden, device=x.device, dtype=torch.float32) if dgamma is None else dgamma
    dbeta = torch.empty(hidden, device=x.device, dtype=torch.float32) if dbeta is None else dbeta
    dev = _dev(dy, x, gamma, mean, rstd, workspace, dx, dgamma, dbeta)
    _call("ls_layernorm_bw", dev, ls_layernorm_bw, _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(dy),
          _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd), rows, hidden, _ptr(workspace),
          workspace.numel() * workspace.element_size(), ls_dtype(x), _stream(x))
    return dx, dgamma, dbeta


def rmsnorm_fw(x, gamma, eps: float = 1e-6, y=None, rstd=None):
    """RMSNorm of x [rows, hidden]: y = x * rsqrt(mean(x^2) + eps) * gamma;
    returns (y, rstd), rstd fp32."""
    torch = _torch()
    rows, hidden = _rows_hidden(x)
    _want("gamma", gamma, (hidden,), x.dtype)
    _want("y", y, x.shape, x.dtype)
    _stats(rows, x, rstd=rstd)
    y = torch.empty_like(x) if y is None else y
    rstd = torch.empty(rows, device=x.device, dtype=torch.float32) if rstd is None else rstd
    dev = _dev(x, gamma, y, rstd)
    _call("ls_rmsnorm_fw", dev, ls_rmsnorm_fw, _ptr(y), _ptr(rstd), _ptr(x), _ptr(gamma), rows,
          hidden, float(eps), ls_dtype(x), _stream(x))
    return y, rstd


def rmsnorm_bw_dinp(dy, x, gamma, rstd, dx=None):
    """Input gradient of RMSNorm from dy, x and the saved fp32 rstd."""
    torch = _torch()
    rows, hidden = _rows_hidden(x)
    _want("dy", dy, x.shape, x.dtype)
    _want("gamma", gamma, (hidden,), x.dtype)
    _stats(rows, x, rstd=rstd)
    _want("dx", dx, x.shape, x.dtype)
    dx = torch.empty_like(x) if dx is None else dx
    dev = _dev(dy, x, gamma, rstd, dx)
    _call("ls_rmsnorm_bw_dinp", dev, ls_rmsnorm_bw_dinp, _ptr(dx), _ptr(dy), _ptr(x), _ptr(gamma),
          _ptr(rstd), rows, hidden, ls_dtype(x), _stream(x))
    return dx


def rmsnorm_bw_dgamma(dy, x, rstd, workspace=None, dgamma=None):
    """gamma gradient of RMSNorm (fp32 [hidden]), fixed summation order."""
    torch = _torch()
    rows, hidden = _rows_hidden(x)
    _want("dy", dy, x.shape, x.dtype)
    _stats(rows, x, rstd=rstd)
    _want("dgamma", dgamma, (hidden,), torch.float32)
    if workspace is None:
        workspace = dgamma_dbeta_workspace(rows, hidden, x.device)
    _workspace("workspace", workspace)
    dgamma = torch.empty(hidden, device=x.device, dtype=torch.float32) if dgamma is None else dgamma
    dev = _dev(dy, x, rstd, workspace, dgamma)
    _call("ls_rmsnorm_bw_dgamma", dev, ls_rmsnorm_bw_dgamma, _ptr(dgamma), _ptr(dy), _ptr(x),
          _ptr(rstd), rows, hidden, _ptr(workspace), workspace.numel() * workspace.element_size(),
          ls_dtype(x), _stream(x))
    return dgamma


def cross_entropy_fw(logits, target, loss=None, lse=None):
    """Per-row softmax cross entropy of logits [rows, vocab] against int32
    target [rows] (negative = ignored row); returns (loss, lse), fp32."""
    torch = _torch()
    if logits.dim() != 2:
        raise ValueError("logits must be [rows, vocab]")
    rows, vocab = logits.shape
    _want("target", target, (rows,), torch.int32)
    _stats(rows, logits, loss=loss, lse=lse)
    loss = torch.empty(rows, device=logits.device, dtype=torch.float32) if loss is None else loss
    lse = torch.empty(rows, device=logits.device, dtype=torch.float32) if lse is None else lse
    dev = _dev(logits, target, loss, lse)
    _call("ls_cross_entropy_fw", dev, ls_cross_entropy_fw, _ptr(loss), _ptr(lse), _ptr(logits),
          _ptr(target), rows, vocab, ls_dtype(logits), _stream(logits))
    return loss, lse


def cross_entropy_bw(logits, target, lse, dloss, dlogits=None):
    """Gradient dloss * (softmax(logits) - onehot(target)) per row, from the
    forward's lse; ``dlogits`` may be ``logits`` (in place)."""
    torch = _torch()
    if logits.dim() != 2:
        raise ValueError("logits must be [rows, vocab]")
    rows, vocab = logits.shape
    _want("target", target, (rows,), torch.int32)
    _stats(rows, logits, lse=lse, dloss=dloss)
    _want("dlogits", dlogits, logits.shape, logits.dtype)
    dlogits = torch.empty_like(logits) if dlogits is None else dlogits
    dev = _dev(logits, target, lse, dloss, dlogits)
    _call("ls_cross_entropy_bw", dev, ls_cross_entropy_bw, _ptr(dlogits), _ptr(logits),
          _ptr(target), _ptr(lse), _ptr(dloss), rows, vocab, ls_dtype(logits), _stream(logits))
    return dlogits
