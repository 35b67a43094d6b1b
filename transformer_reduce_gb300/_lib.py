"""ctypes binding of libls_reduce.so (argument marshalling only).

The functions named ``ls_*`` mirror the C ABI of ``include/ls_reduce.h``
one-for-one: device pointers are passed as Python ints, sizes as ints, the
stream as an int handle (0 = legacy default stream).  They return the
``ls_status`` code unchanged.  All computation happens in the CUDA kernels of
the library; nothing here touches tensor data.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libls_reduce.so")

LS_F32, LS_F16, LS_BF16 = 0, 1, 2
LS_OK = 0
LS_ERR_INVALID_ARG = 1
LS_ERR_UNSUPPORTED = 2
LS_ERR_MISALIGNED = 3
LS_ERR_WORKSPACE = 4
LS_ERR_CUDA = 5

# Every function the header declares, with its ctypes signature.
_VP, _I64, _INT, _F32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "ls_softmax_fw": ([_VP, _VP, _VP, _I64, _I64, _I64, _I64, _INT, _INT, _VP], _INT),
    "ls_softmax_bw": ([_VP, _VP, _VP, _I64, _I64, _I64, _I64, _INT, _VP], _INT),
    "ls_softmax_bw_masked": ([_VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _INT, _INT, _VP], _INT),
    "ls_softmax_fw_scaled": ([_VP, _VP, _VP, _I64, _I64, _I64, _I64, _INT, _F32, _INT, _VP], _INT),
    "ls_softmax_bw_masked_scaled": ([_VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _INT, _F32, _INT,
                                     _VP], _INT),
    "ls_layernorm_fw": ([_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _F32, _INT, _VP], _INT),
    "ls_layernorm_bw_dinp": ([_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _INT, _VP], _INT),
    "ls_layernorm_bw_dgamma_dbeta_workspace_size": ([_I64, _I64], _SZ),
    "ls_layernorm_bw_dgamma_dbeta": ([_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _VP, _SZ, _INT, _VP],
                                     _INT),
    "ls_layernorm_bw_dgamma_dbeta_noalloc": ([_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _INT, _VP],
                                             _INT),
    "ls_layernorm_bw_workspace_size": ([_I64, _I64], _SZ),
    "ls_layernorm_bw": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _VP, _SZ, _INT, _VP],
                        _INT),
    "ls_rmsnorm_fw": ([_VP, _VP, _VP, _VP, _I64, _I64, _F32, _INT, _VP], _INT),
    "ls_rmsnorm_bw_dinp": ([_VP, _VP, _VP, _VP, _VP, _I64, _I64, _INT, _VP], _INT),
    "ls_rmsnorm_bw_dgamma": ([_VP, _VP, _VP, _VP, _I64, _I64, _VP, _SZ, _INT, _VP], _INT),
    "ls_cross_entropy_fw": ([_VP, _VP, _VP, _VP, _I64, _I64, _INT, _VP], _INT),
    "ls_cross_entropy_bw": ([_VP, _VP, _VP, _VP, _VP, _I64, _I64, _INT, _VP], _INT),
    "ls_status_string": ([_INT], ctypes.c_char_p),
}

_lib = None


class LsError(RuntimeError):
    """A non-zero ls_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load() -> ctypes.CDLL:
    """Load libls_reduce.so.  Fails loudly if it has not been built: there is
    no fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m transformer_reduce_gb300.build` "
                "(the CUDA library is required; there is no CPU or PyTorch fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().ls_status_string(int(status)).decode()


def ls_softmax_fw(out, inp, mask, B, H, Tq, Tk, causal, dt, stream=0) -> int:
    return load().ls_softmax_fw(out, inp, mask, B, H, Tq, Tk, int(bool(causal)), dt, stream)


def ls_softmax_bw(dinp, dout, out_fw, B, H, Tq, Tk, dt, stream=0) -> int:
    return load().ls_softmax_bw(dinp, dout, out_fw, B, H, Tq, Tk, dt, stream)


def ls_softmax_bw_masked(dinp, dout, out_fw, mask, B, H, Tq, Tk, causal, dt, stream=0) -> int:
    return load().ls_softmax_bw_masked(dinp, dout, out_fw, mask, B, H, Tq, Tk, int(bool(causal)),
                                       dt, stream)


def ls_layernorm_fw(y, mean, rstd, x, gamma, beta, rows, hidden, eps, dt, stream=0) -> int:
    return load().ls_layernorm_fw(y, mean, rstd, x, gamma, beta, rows, hidden, eps, dt, stream)


def ls_layernorm_bw_dinp(dx, dy, x, gamma, mean, rstd, rows, hidden, dt, stream=0) -> int:
    return load().ls_layernorm_bw_dinp(dx, dy, x, gamma, mean, rstd, rows, hidden, dt, stream)


def ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden) -> int:
    return load().ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden)


def ls_layernorm_bw_dgamma_dbeta(dgamma, dbeta, dy, x, mean, rstd, rows, hidden, workspace,
                                 workspace_bytes, dt, stream=0) -> int:
    return load().ls_layernorm_bw_dgamma_dbeta(dgamma, dbeta, dy, x, mean, rstd, rows, hidden,
                                               workspace, workspace_bytes, dt, stream)


def ls_layernorm_bw_dgamma_dbeta_noalloc(dgamma, dbeta, dy, x, mean, rstd, rows, hidden, dt,
                                         stream=0) -> int:
    """The gamma/beta gradient for callers that cannot allocate a workspace:
    the library's own fixed device array holds the partial sums (see the
    header for its size limit and the rule that overlapping calls race)."""
    return load().ls_layernorm_bw_dgamma_dbeta_noalloc(dgamma, dbeta, dy, x, mean, rstd, rows,
                                                       hidden, dt, stream)


def ls_layernorm_bw_workspace_size(rows, hidden) -> int:
    return load().ls_layernorm_bw_workspace_size(rows, hidden)


def ls_layernorm_bw(dx, dgamma, dbeta, dy, x, gamma, mean, rstd, rows, hidden, workspace,
                    workspace_bytes, dt, stream=0) -> int:
    return load().ls_layernorm_bw(dx, dgamma, dbeta, dy, x, gamma, mean, rstd, rows, hidden,
                                  workspace, workspace_bytes, dt, stream)


def ls_rmsnorm_fw(y, rstd, x, gamma, rows, hidden, eps, dt, stream=0) -> int:
    return load().ls_rmsnorm_fw(y, rstd, x, gamma, rows, hidden, eps, dt, stream)


def ls_rmsnorm_bw_dinp(dx, dy, x, gamma, rstd, rows, hidden, dt, stream=0) -> int:
    return load().ls_rmsnorm_bw_dinp(dx, dy, x, gamma, rstd, rows, hidden, dt, stream)


def ls_rmsnorm_bw_dgamma(dgamma, dy, x, rstd, rows, hidden, workspace, workspace_bytes, dt,
                         stream=0) -> int:
    return load().ls_rmsnorm_bw_dgamma(dgamma, dy, x, rstd, rows, hidden, workspace,
                                       workspace_bytes, dt, stream)


def ls_cross_entropy_fw(loss, lse, logits, target, rows, vocab, dt, stream=0) -> int:
    return load().ls_cross_entropy_fw(loss, lse, logits, target, rows, vocab, dt, stream)


def ls_cross_entropy_bw(dlogits, logits, target, lse, dloss, rows, vocab, dt, stream=0) -> int:
    return load().ls_cross_entropy_bw(dlogits, logits, target, lse, dloss, rows, vocab, dt, stream)


def ls_softmax_fw_scaled(out, inp, mask, B, H, Tq, Tk, causal, scale, dt, stream=0) -> int:
    return load().ls_softmax_fw_scaled(out, inp, mask, B, H, Tq, Tk, causal, scale, dt, stream)


def ls_softmax_bw_masked_scaled(dinp, dout, out_fw, mask, B, H, Tq, Tk, causal, scale, dt,
                                stream=0) -> int:
    return load().ls_softmax_bw_masked_scaled(dinp, dout, out_fw, mask, B, H, Tq, Tk, causal,
                                              scale, dt, stream)
