"""Host-side checks of the PyTorch binding: it refuses tensors whose shape,
dtype or device would make a kernel read or write past a buffer, before any
pointer reaches the library (no GPU needed: the checks run first)."""
import pytest
import torch

import transformer_reduce_gb300 as L


def _raises(match, fn, *a, **k):
    with pytest.raises(ValueError, match=match):
        fn(*a, **k)


def test_softmax_outputs_and_mask_are_checked():
    s = torch.zeros(2, 3, 4, 8, dtype=torch.bfloat16)
    _raises("out must be", L.softmax_fw, s, out=torch.zeros(2, 3, 4, 7, dtype=torch.bfloat16))
    _raises("out must be", L.softmax_fw, s, out=torch.zeros(2, 3, 4, 8, dtype=torch.float16))
    _raises("mask must be", L.softmax_fw, s, torch.zeros(2, 7, dtype=torch.bfloat16))
    _raises("mask must be", L.softmax_fw, s, torch.zeros(2, 8, dtype=torch.float32))
    _raises("out_fw must be", L.softmax_bw, s, s[..., :4])
    _raises("dinp must be", L.softmax_bw, s, s, dinp=torch.zeros(2, 3, 4, 8))
    _raises("mask must be", L.softmax_bw_masked, s, s, torch.zeros(3, 8, dtype=torch.bfloat16))
    # well-formed CPU tensors get as far as the device check
    _raises("CUDA device", L.softmax_fw, s)


def test_layernorm_parameters_statistics_and_outputs_are_checked():
    x = torch.zeros(5, 16, dtype=torch.float16)
    g = torch.ones(16, dtype=torch.float16)
    f32 = torch.float32
    _raises("gamma must be", L.layernorm_fw, x, g[:8], g)
    _raises("beta must be", L.layernorm_fw, x, g, g.float())
    _raises("y must be", L.layernorm_fw, x, g, g, y=torch.zeros(5, 15, dtype=torch.float16))
    _raises("mean must be", L.layernorm_fw, x, g, g, mean=torch.zeros(4, dtype=f32))
    _raises("rstd must be", L.layernorm_fw, x, g, g, rstd=torch.zeros(5, dtype=torch.float16))
    m = torch.zeros(5, dtype=f32)
    _raises("dy must be", L.layernorm_bw_dinp, x[:4], x, g, m, m)
    _raises("gamma must be", L.layernorm_bw_dinp, x, x, g.float(), m, m)
    _raises("mean must be", L.layernorm_bw_dinp, x, x, g, m[:3], m)
    _raises("dgamma must be", L.layernorm_bw_dgamma_dbeta, x, x, m, m,
            dgamma=torch.zeros(16, dtype=torch.float16))
    _raises("workspace must be", L.layernorm_bw, x, x, g, m, m,
            workspace=torch.zeros(64, dtype=torch.float16))
    _raises("dbeta must be", L.layernorm_bw, x, x, g, m, m, dbeta=torch.zeros(17, dtype=f32))
    _raises("gamma must be", L.rmsnorm_fw, x, g[:15])
    _raises("rstd must be", L.rmsnorm_bw_dinp, x, x, g, m[:1])
    _raises("dgamma must be", L.rmsnorm_bw_dgamma, x, x, m, dgamma=torch.zeros(15, dtype=f32))
    _raises(r"\[rows, hidden\]", L.layernorm_fw, x.view(5, 4, 4), g, g)
    _raises("CUDA device", L.layernorm_fw, x, g, g)


def test_cross_entropy_arguments_are_checked():
    z = torch.zeros(4, 9)
    t = torch.zeros(4, dtype=torch.int32)
    _raises("target must be", L.cross_entropy_fw, z, t.long())
    _raises("target must be", L.cross_entropy_fw, z, t[:3])
    _raises("loss must be", L.cross_entropy_fw, z, t, loss=torch.zeros(5))
    lse = torch.zeros(4)
    _raises("dloss must be", L.cross_entropy_bw, z, t, lse, torch.zeros(4, dtype=torch.float64))
    _raises("lse must be", L.cross_entropy_bw, z, t, lse[:2], lse)
    _raises("dlogits must be", L.cross_entropy_bw, z, t, lse, lse, dlogits=torch.zeros(4, 8))
    _raises("CUDA device", L.cross_entropy_fw, z, t)
