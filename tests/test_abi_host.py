"""Host-side checks of the C ABI, the byte model and the input generator.

These run without a GPU: the library is loaded and its exports are compared
with the header; only calls that the ABI rejects (or treats as no-ops) before
touching the CUDA runtime are made.  No kernel is launched here.
"""
import ctypes
import json
import math
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ls_reduce.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "pages_figures.json")


@pytest.fixture(scope="module")
def abi():
    from transformer_reduce_gb300 import build as b
    b.build()
    from transformer_reduce_gb300 import _lib
    _lib.load()
    return _lib


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ls_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_function(abi):
    declared = _declared_functions()
    assert {"ls_softmax_fw", "ls_softmax_bw", "ls_layernorm_fw", "ls_layernorm_bw_dinp",
            "ls_layernorm_bw_dgamma_dbeta", "ls_layernorm_bw_dgamma_dbeta_workspace_size",
            "ls_status_string"} <= declared
    lib = ctypes.CDLL(abi.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    # and the Python binding mirrors each one under the same name
    assert declared <= set(abi.SIGNATURES)


def test_status_strings(abi):
    for code in range(6):
        s = abi.status_string(code)
        assert s.startswith("LS_")
    assert "unknown" in abi.status_string(99)


def test_rejections_before_launch(abi):
    F32, BF16 = abi.LS_F32, abi.LS_BF16
    fake = 0x10000  # never dereferenced: every call below returns on the host
    # unknown dtype
    assert abi.ls_softmax_fw(fake, fake, None, 1, 1, 4, 4, 0, 7) == abi.LS_ERR_UNSUPPORTED
    # negative sizes, missing pointers, causal with Tq != Tk
    assert abi.ls_softmax_fw(fake, fake, None, -1, 1, 4, 4, 0, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_softmax_fw(None, fake, None, 1, 1, 4, 4, 0, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_softmax_fw(fake, fake, None, 1, 1, 5, 4, 1, F32) == abi.LS_ERR_INVALID_ARG  # causal, Tq > Tk
    assert abi.ls_softmax_bw_masked(fake, fake, fake, None, 1, 1, 5, 4, 1, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_softmax_bw_masked(fake, None, fake, None, 1, 1, 4, 4, 0, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_softmax_bw_masked(fake, fake, fake, fake + 2, 1, 1, 4, 4, 0, F32) == abi.LS_ERR_MISALIGNED
    assert abi.ls_softmax_bw_masked(None, None, None, None, 0, 1, 4, 4, 1, BF16) == abi.LS_OK
    assert abi.ls_softmax_bw(fake, None, fake, 1, 1, 4, 4, F32) == abi.LS_ERR_INVALID_ARG
    # misaligned element pointers
    assert abi.ls_softmax_fw(fake + 2, fake, None, 1, 1, 4, 4, 0, F32) == abi.LS_ERR_MISALIGNED
    assert abi.ls_softmax_bw(fake, fake + 1, fake, 1, 1, 4, 4, BF16) == abi.LS_ERR_MISALIGNED
    # rows beyond the row-length limit
    assert abi.ls_softmax_fw(fake, fake, None, 1, 1, 1, (1 << 30) + 1, 0, F32) == abi.LS_ERR_UNSUPPORTED
    # empty problems are no-ops, even with NULL pointers
    assert abi.ls_softmax_fw(None, None, None, 0, 8, 4, 4, 0, F32) == abi.LS_OK
    assert abi.ls_softmax_fw(None, None, None, 2, 8, 4, 0, 0, F32) == abi.LS_OK
    assert abi.ls_softmax_bw(None, None, None, 2, 0, 4, 4, F32) == abi.LS_OK
    # LayerNorm
    assert abi.ls_layernorm_fw(fake, fake, fake, fake, fake, fake, 4, 0, 1e-8, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_layernorm_fw(fake, fake, fake, fake, fake, fake, -1, 8, 1e-8, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_layernorm_fw(fake, fake, fake, fake, fake, fake, 4, 8, -1.0, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_layernorm_fw(fake, fake, fake, fake, fake, fake, 4, 8, math.nan, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_layernorm_fw(fake, None, fake, fake, fake, fake, 4, 8, 1e-8, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_layernorm_fw(fake, fake + 2, fake, fake, fake, fake, 4, 8, 1e-8, BF16) == abi.LS_ERR_MISALIGNED
    assert abi.ls_layernorm_fw(None, None, None, None, None, None, 0, 8, 1e-8, F32) == abi.LS_OK
    assert abi.ls_layernorm_bw_dinp(fake, fake, None, fake, fake, fake, 4, 8, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_layernorm_bw_dinp(None, None, None, None, None, None, 0, 8, F32) == abi.LS_OK
    # RMSNorm
    assert abi.ls_rmsnorm_fw(fake, fake, fake, fake, 4, 0, 1e-6, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_rmsnorm_fw(fake, None, fake, fake, 4, 8, 1e-6, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_rmsnorm_fw(fake, fake, fake, fake, 4, 8, -1.0, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_rmsnorm_fw(None, None, None, None, 0, 8, 1e-6, F32) == abi.LS_OK
    assert abi.ls_rmsnorm_bw_dinp(fake, fake, fake, fake, fake + 2, 4, 8, F32) == abi.LS_ERR_MISALIGNED
    assert abi.ls_rmsnorm_bw_dgamma(fake, fake, fake, fake, 16384, 1024, None, 0, BF16) == abi.LS_ERR_WORKSPACE
    # scaled softmax: the scale must be finite and > 0
    for bad in (0.0, -0.5, math.inf, math.nan):
        assert abi.ls_softmax_fw_scaled(fake, fake, None, 1, 1, 4, 4, 0, bad, F32) == abi.LS_ERR_INVALID_ARG
        assert abi.ls_softmax_bw_masked_scaled(fake, fake, fake, None, 1, 1, 4, 4, 0, bad,
                                               F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_softmax_fw_scaled(fake, fake, None, 1, 1, 4, 4, 0, 0.5, 9) == abi.LS_ERR_UNSUPPORTED
    assert abi.ls_softmax_fw_scaled(fake, fake, None, 1, 1, 5, 4, 1, 0.5, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_softmax_fw_scaled(None, None, None, 0, 1, 4, 4, 0, 0.5, BF16) == abi.LS_OK
    assert abi.ls_softmax_bw_masked_scaled(None, None, None, None, 0, 1, 4, 4, 1, 0.5, BF16) == abi.LS_OK
    # cross entropy
    assert abi.ls_cross_entropy_fw(fake, fake, fake, fake, 4, 0, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_cross_entropy_fw(fake, fake, fake, fake, -1, 9, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_cross_entropy_fw(fake, None, fake, fake, 4, 9, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_cross_entropy_fw(fake, fake, fake, fake + 2, 4, 9, F32) == abi.LS_ERR_MISALIGNED
    assert abi.ls_cross_entropy_fw(fake, fake, fake + 1, fake, 4, 9, BF16) == abi.LS_ERR_MISALIGNED
    assert abi.ls_cross_entropy_fw(fake, fake, fake, fake, 4, (1 << 30) + 1, F32) == abi.LS_ERR_UNSUPPORTED
    assert abi.ls_cross_entropy_fw(fake, fake, fake, fake, 4, 9, 3) == abi.LS_ERR_UNSUPPORTED
    assert abi.ls_cross_entropy_fw(None, None, None, None, 0, 9, F32) == abi.LS_OK
    assert abi.ls_cross_entropy_bw(fake, fake, fake, fake, None, 4, 9, F32) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_cross_entropy_bw(fake, fake, fake, fake + 1, fake, 4, 9, F32) == abi.LS_ERR_MISALIGNED
    assert abi.ls_cross_entropy_bw(None, None, None, None, None, 0, 9, BF16) == abi.LS_OK
    # fused LayerNorm backward
    nf = abi.ls_layernorm_bw_workspace_size(16384, 1024)
    assert abi.ls_layernorm_bw(fake, fake, fake, fake, fake, fake, fake, fake, 16384, 1024,
                               None, 0, BF16) == abi.LS_ERR_WORKSPACE
    assert abi.ls_layernorm_bw(fake, fake, fake, fake, fake, fake, fake, fake, 16384, 1024,
                               fake, nf - 4, BF16) == abi.LS_ERR_WORKSPACE
    assert abi.ls_layernorm_bw(fake, None, fake, fake, fake, fake, fake, fake, 16384, 1024,
                               fake, nf, BF16) == abi.LS_ERR_INVALID_ARG
    assert abi.ls_layernorm_bw(fake, fake, fake, fake, fake, fake, fake, fake + 2, 16384, 1024,
                               fake, nf, BF16) == abi.LS_ERR_MISALIGNED
    assert abi.ls_layernorm_bw(fake, fake, fake, fake, fake, fake, fake, fake, 16384, 0,
                               fake, nf, BF16) == abi.LS_ERR_INVALID_ARG
    # gamma / beta gradient: workspace checks
    need = abi.ls_layernorm_bw_dgamma_dbeta_workspace_size(16384, 1024)
    assert need > 0
    assert abi.ls_layernorm_bw_dgamma_dbeta(fake, fake, fake, fake, fake, fake, 16384, 1024,
                                            None, 0, BF16) == abi.LS_ERR_WORKSPACE
    assert abi.ls_layernorm_bw_dgamma_dbeta(fake, fake, fake, fake, fake, fake, 16384, 1024,
                                            fake, need - 4, BF16) == abi.LS_ERR_WORKSPACE
    assert abi.ls_layernorm_bw_dgamma_dbeta(fake, fake, fake, fake, fake, fake, 16384, 1024,
                                            fake + 8, need, BF16) == abi.LS_ERR_WORKSPACE
    assert abi.ls_layernorm_bw_dgamma_dbeta(None, fake, fake, fake, fake, fake, 16384, 1024,
                                            fake, need, BF16) == abi.LS_ERR_INVALID_ARG


def test_workspace_size_depends_only_on_shape(abi):
    ws = abi.ls_layernorm_bw_dgamma_dbeta_workspace_size
    assert ws(0, 1024) == 0 and ws(16, 0) == 0 and ws(-3, 8) == 0
    for rows, hidden in [(1, 1), (64, 128), (8192, 256), (16384, 1024), (16384, 8192),
                         (3, 770), (100000, 64)]:
        n = ws(rows, hidden)
        assert n % (2 * 4 * hidden) == 0
        nchunks = n // (2 * 4 * hidden)
        assert 1 <= nchunks <= 65535
        # at least 16 rows per chunk unless the problem is smaller
        assert nchunks <= max(1, math.ceil(rows / 16))
        # the chunk partials stay small next to the inputs for large problems
        if rows * hidden >= 1 << 22:
            assert n <= 0.1 * rows * hidden * 2 * 2


def test_fused_backward_workspace_size():
    from transformer_reduce_gb300 import _lib
    _lib.load()
    ws = _lib.ls_layernorm_bw_workspace_size
    assert ws(0, 1024) == 0 and ws(16, 0) == 0
    for rows, hidden in [(1, 1), (303, 64), (304, 64), (305, 64), (16384, 1024), (7, 20000)]:
        n = ws(rows, hidden)
        # one chunk per row up to 456 rows, then at most 456 chunks; one
        # partial sum per chunk
        chunks = rows if rows <= 456 else len(range(0, rows, -(-rows // 456)))
        assert n >= chunks * 2 * 4 * hidden
        assert n <= max(456 * 2 * 4 * hidden,
                        _lib.ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden))
        assert n >= _lib.ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden)


def test_no_alloc_scratch_covers_the_stated_widths(abi):
    # the header's bound: every hidden <= 2^19 fits the 4 MiB array
    ws = abi.ls_layernorm_bw_dgamma_dbeta_workspace_size
    for hidden in [1, 255, 256, 257, 1000, 1024, 8192, 65536, 100003, 155647, 155648, 368640,
                   524287, 1 << 19]:
        for rows in [1, 15, 16, 17, 1000, 9727, 9728, 16384, 100000, 1 << 22]:
            assert ws(rows, hidden) <= 4 << 20, (rows, hidden)
    assert ws(1 << 16, (1 << 19) + 1) > 4 << 20


def test_byte_model_reproduces_the_pages_figure():
    from transformer_reduce_gb300 import traffic
    g = json.load(open(GOLDEN, encoding="utf-8"))
    fig = g["attention_probability_traffic"]
    B, H, T, L = (fig["shape"][k] for k in ("B", "H", "T", "layers"))
    total = L * (traffic.softmax_fw_write_bytes(B, H, T, "f32")
                 + traffic.softmax_bw_out_fw_read_bytes(B, H, T, "f32"))
    assert round(total / 1e6) == fig["value_mb"]
    assert g["tokens_per_step"]["value"] == fig["shape"]["B"] * fig["shape"]["T"]


def test_byte_model_visible_keys():
    from transformer_reduce_gb300.traffic import visible_keys
    # causal, no padding: row i sees i + 1 keys
    assert visible_keys(4, [4], True, 1) == 1 + 2 + 3 + 4
    # causal with padding length 2: rows see 1, 2, 2, 2 keys
    assert visible_keys(4, [2], True, 3) == 3 * (1 + 2 + 2 + 2)
    assert visible_keys(5, [3, 5], False, 2) == 2 * 5 * 3 + 2 * 5 * 5


def test_configs_restate_the_workloads():
    from transformer_reduce_gb300 import workloads as w
    g = json.load(open(GOLDEN, encoding="utf-8"))
    assert tuple(g["softmax_bw_length_buckets"]["value"]) == w.SWEEP_T
    assert w.LN_EPS == g["layernorm_eps"]["value"]
    assert w.GPT2_SMALL["layernorm"].rows == g["tokens_per_step"]["value"]
    assert w.GPT2_SMALL["softmax"].shape == (32, 8, 256, 256)
    assert w.ENCODER_BIG["softmax"].shape == (32, 16, 512, 512)


def test_generator_is_seeded_and_shaped():
    from transformer_reduce_gb300 import workloads as w
    case = w.TINY["softmax"]
    a = w.softmax_inputs(case)
    b = w.softmax_inputs(case)
    assert torch.equal(a["scores"], b["scores"]) and torch.equal(a["dout"], b["dout"])
    assert a["lengths"] == b["lengths"]
    assert all(16 <= n <= 32 for n in a["lengths"])
    m = a["mask"]
    for bb, n in enumerate(a["lengths"]):
        assert torch.all(m[bb, :n] == 0) and torch.all(torch.isinf(m[bb, n:]))
    ln = w.layernorm_inputs(w.LAYERNORM_SWEEP[0])
    assert ln["x"].dtype == torch.bfloat16 and ln["x"].shape == (16384, 768)
    assert 0.9 < ln["x"].float().mean().item() < 1.1
    assert 1.9 < ln["x"].float().std().item() < 2.1
    assert float(ln["gamma"].min()) >= 0.5 and float(ln["gamma"].max()) <= 1.5
    y = w.softmax_probability_like(case, a["lengths"])
    assert torch.all(y[..., 31:, :].float() >= 0)
    # future keys of a causal case are exactly zero
    assert torch.all(torch.triu(y.float()[0, 0], diagonal=1) == 0)
