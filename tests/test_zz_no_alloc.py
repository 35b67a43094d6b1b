"""The allocation-free gamma/beta gradient entry point.

ls_layernorm_bw_dgamma_dbeta_noalloc serves callers that cannot give the
library a workspace: code that only receives tensor pointers and a stream
from a host program, or code that may not call cudaMalloc at that point
(cudaMalloc can synchronise the device or break the host's memory budget).
It keeps its partial sums in a fixed device array inside the library.

This test calls it through the C ABI twice in a row, on two different
problems, and checks each result against the workspace entry point
ls_layernorm_bw_dgamma_dbeta: within the tolerance rule of the parity tests,
and bit for bit, since both run the same kernels in the same fixed summation
order (the second call must not see the first call's leftovers in the shared
array).  It also checks that a problem too large for the array is refused.
The file name makes pytest collect it last.
"""
import pytest
import torch

from _parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def abi():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_reduce_gb300 import build
    build.build()
    from transformer_reduce_gb300 import _lib
    _lib.load()
    return _lib


def _problem(rows, hidden, dtype, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = (torch.randn(rows, hidden, generator=g, device=DEV) * 2 + 1).to(dtype)
    dy = torch.randn(rows, hidden, generator=g, device=DEV).to(dtype)
    mean = 1 + 0.01 * torch.randn(rows, generator=g, device=DEV)
    rstd = 0.45 + 0.1 * torch.rand(rows, generator=g, device=DEV)
    return x, dy, mean, rstd


def _with_workspace(abi, x, dy, mean, rstd, dt):
    rows, hidden = x.shape
    n = abi.ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden)
    ws = torch.empty(max(n, 16) // 4, device=DEV, dtype=torch.float32)
    dg = torch.empty(hidden, device=DEV)
    db = torch.empty(hidden, device=DEV)
    st = abi.ls_layernorm_bw_dgamma_dbeta(dg.data_ptr(), db.data_ptr(), dy.data_ptr(),
                                          x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), rows,
                                          hidden, ws.data_ptr(), ws.numel() * 4, dt,
                                          torch.cuda.current_stream().cuda_stream)
    assert st == abi.LS_OK
    return dg, db


def _no_alloc(abi, x, dy, mean, rstd, dt):
    rows, hidden = x.shape
    dg = torch.full((hidden,), float("nan"), device=DEV)
    db = torch.full((hidden,), float("nan"), device=DEV)
    st = abi.ls_layernorm_bw_dgamma_dbeta_noalloc(dg.data_ptr(), db.data_ptr(), dy.data_ptr(),
                                                  x.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                                                  rows, hidden, dt,
                                                  torch.cuda.current_stream().cuda_stream)
    assert st == abi.LS_OK, abi.status_string(st)
    return dg, db


def test_no_alloc_matches_workspace_entry_point_on_two_calls_in_a_row(abi):
    # first call: the Transformer-big encoder LayerNorm shape (bf16);
    # second call: a smaller fp16 problem that reads fewer partials
    problems = [((16384, 1024), torch.bfloat16, abi.LS_BF16, "bf16", 1),
                ((8192, 256), torch.float16, abi.LS_F16, "f16", 2)]
    for (rows, hidden), tdt, dt, name, seed in problems:
        x, dy, mean, rstd = _problem(rows, hidden, tdt, seed)
        want_g, want_b = _with_workspace(abi, x, dy, mean, rstd, dt)
        got_g, got_b = _no_alloc(abi, x, dy, mean, rstd, dt)
        torch.cuda.synchronize()
        compare(got_g, want_g.double().cpu().numpy(), name, f"no-alloc dgamma {rows}x{hidden}")
        compare(got_b, want_b.double().cpu().numpy(), name, f"no-alloc dbeta {rows}x{hidden}")
        assert torch.equal(got_g, want_g), f"dgamma {rows}x{hidden} differs bitwise"
        assert torch.equal(got_b, want_b), f"dbeta {rows}x{hidden} differs bitwise"


def test_no_alloc_refuses_problems_beyond_its_array(abi):
    # one chunk of partial sums for a row of 2^20 features already needs 8 MiB
    rows, hidden = 16, 1 << 20
    need = abi.ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden)
    assert need > 4 << 20
    fake = 0x10000  # refused on the host before any pointer is used
    st = abi.ls_layernorm_bw_dgamma_dbeta_noalloc(fake, fake, fake, fake, fake, fake, rows,
                                                  hidden, abi.LS_BF16, 0)
    assert st == abi.LS_ERR_UNSUPPORTED
