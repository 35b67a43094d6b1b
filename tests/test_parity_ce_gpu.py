"""GPU parity of the cross-entropy kernels (through the C ABI) against the
fp64 CPU oracle, on the seeded inputs of ``workloads.cross_entropy_inputs``.

Forward: loss and log-sum-exp per row.  Backward: dlogits from the oracle's
log-sum-exp (never the GPU's), with a per-row upstream gradient of 1 so the
gradient entries are probabilities, not probabilities divided by the token
count.  Beyond the tolerance rule of ``_parity.compare`` every gradient entry
is also held to a relative bound of a few storage steps, since most entries
are far below the absolute tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from _parity import compare, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
# relative step of each storage type, and an absolute floor: two fp16
# subnormal steps for fp16, far below anything else for fp32 / bf16
STEP = {"f32": 2.0 ** -23, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}
FLOOR = {"f32": 1e-37, "f16": 1.2e-7, "bf16": 1e-37}


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


def _case(rows, vocab, dtype, seed=5, pad=None):
    from transformer_reduce_gb300.workloads import CrossEntropyCase
    return CrossEntropyCase(f"ce_edge_{dtype}_{rows}x{vocab}", 1, rows, vocab, pad, 3.0, dtype,
                            seed)


def relative_check(got: torch.Tensor, ref: np.ndarray, target, dtype: str, what: str,
                   k: float = 4.0):
    """|got - ref| <= k storage steps of |ref| + the FP32 arithmetic's error
    (4e-6 relative) + the absolute floor of the storage type.  At the target
    entry the gradient is p - 1 (upstream gradient 1): its error is p's, so
    the scale there is |ref| + p rather than |ref| (p - 1 may cancel to 0)."""
    g = got.detach().cpu().to(torch.float64).numpy()
    ref = np.asarray(ref, dtype=np.float64).reshape(g.shape)
    scale = np.abs(ref).copy()
    t = np.asarray(target)
    for r in np.nonzero((t >= 0) & (t < ref.shape[1]))[0]:
        scale[r, t[r]] += abs(ref[r, t[r]] + 1.0)
    bound = k * STEP[dtype] * scale + 4e-6 * scale + FLOOR[dtype]
    bad = np.abs(g - ref) > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} entries off by more than {k} steps, "
                             f"e.g. {i}: {g[i]} vs {ref[i]}")


def check_ce(case, full=True, seed=0, logits=None):
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    inp = W.cross_entropy_inputs(case, device=DEV)
    z = inp["logits"] if logits is None else logits
    t = inp["target"]
    R, V = z.shape
    loss, lse = L.cross_entropy_fw(z, t)
    torch.cuda.synchronize()
    rows = np.arange(R) if full else sample_rows(R, seed=seed, k=48)
    ri = torch.from_numpy(rows).to(DEV)
    zr = z.index_select(0, ri).cpu()
    tr = t.index_select(0, ri).cpu()
    rl, rs = oracle.cross_entropy_fw(zr, tr)
    compare(loss.cpu()[rows], rl, case.dtype, f"{case.name} ce loss")
    compare(lse.cpu()[rows], rs, case.dtype, f"{case.name} ce lse")
    # backward input: the oracle's lse as fp32 on the checked rows (other rows
    # get 30, which keeps their unchecked gradients small and finite)
    lse_in = torch.full((R,), 30.0, dtype=torch.float32)
    lse_in[torch.from_numpy(rows)] = torch.from_numpy(rs).float()
    lse_in = lse_in.to(DEV)
    dz = L.cross_entropy_bw(z, t, lse_in, torch.ones(R, device=DEV))
    torch.cuda.synchronize()
    ref = oracle.cross_entropy_bw(zr, tr, lse_in.cpu()[rows], np.ones(len(rows)))
    got = dz.index_select(0, ri)
    compare(got, ref, case.dtype, f"{case.name} ce dlogits")
    relative_check(got, ref, tr.numpy(), case.dtype, f"{case.name} ce dlogits")
    return z, t, lse_in, dz


def test_ce_tiny_with_ignored_rows():
    from transformer_reduce_gb300 import workloads as W
    z, t, _, dz = check_ce(W.CE_TINY, full=True)
    ign = (t < 0).cpu()
    assert ign.any()
    assert torch.all(dz.cpu()[ign] == 0)


def test_ce_gpt2_vocab_50257_f16_sampled():
    from transformer_reduce_gb300 import workloads as W
    check_ce(W.CE_GPT2, full=False, seed=1)


def test_ce_padded_vocab_bf16_sampled():
    from transformer_reduce_gb300 import workloads as W
    check_ce(W.CE_GPT2_PADDED, full=False, seed=2)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("vocab", [1, 2, 7, 8, 9, 65, 4095, 4096, 4097, 4103, 32003])
def test_ce_vocab_edges(dtype, vocab):
    # rows at every start offset modulo 16 bytes (odd vocab), the one-warp and
    # the one-block paths (4096 16-bit logits = 512 vectors), one ignored row
    check_ce(_case(11, vocab, dtype, pad=(9, 10)), full=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ce_unaligned_base_and_scalar_backward(dtype):
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    case = _case(13, 4099, dtype)
    inp = W.cross_entropy_inputs(case, device=DEV)
    R, V = inp["logits"].shape
    # logits one element past a 16-byte boundary
    buf = torch.empty(R * V + 8, device=DEV, dtype=inp["logits"].dtype)
    z = buf[1:1 + R * V].view(R, V)
    z.copy_(inp["logits"])
    check_ce(case, full=True, logits=z)
    loss, lse = L.cross_entropy_fw(z, inp["target"])
    # dlogits at another offset modulo 16 bytes takes the element-by-element
    # path; its values are bitwise the vector path's
    d_scalar = torch.empty(R * V + 8, device=DEV, dtype=z.dtype)[2:2 + R * V].view(R, V)
    d_vec = torch.empty(R * V + 8, device=DEV, dtype=z.dtype)[1:1 + R * V].view(R, V)
    L.cross_entropy_bw(z, inp["target"], lse, inp["dloss"], dlogits=d_scalar)
    L.cross_entropy_bw(z, inp["target"], lse, inp["dloss"], dlogits=d_vec)
    torch.cuda.synchronize()
    assert torch.equal(d_scalar, d_vec)


def test_ce_in_place_backward_and_out_of_range_target():
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    case = _case(6, 1000, "bf16")
    inp = W.cross_entropy_inputs(case, device=DEV)
    z, t = inp["logits"], inp["target"].clone()
    t[2] = 1000  # out of range
    t[4] = -7    # ignored
    loss, lse = L.cross_entropy_fw(z, t)
    torch.cuda.synchronize()
    lc, sc = loss.cpu(), lse.cpu()
    assert math.isnan(lc[2]) and math.isnan(sc[2])
    assert lc[4] == 0 and sc[4] == 0
    rl, rs = oracle.cross_entropy_fw(z.cpu(), t.cpu())
    keep = [0, 1, 3, 5]
    compare(lc[keep], rl[keep], "bf16", "ce loss next to bad rows")
    dz = L.cross_entropy_bw(z, t, lse, torch.ones(6, device=DEV))
    zz = z.clone()
    L.cross_entropy_bw(zz, t, lse, torch.ones(6, device=DEV), dlogits=zz)
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(dz[2].float())) and torch.all(dz[4] == 0)
    assert torch.equal(zz[keep], dz[keep])
    assert torch.all(torch.isnan(zz[2].float())) and torch.all(zz[4] == 0)


def test_ce_large_logits_fp32():
    from transformer_reduce_gb300 import workloads as W
    L = _L()
    case = _case(9, 3001, "f32")
    inp = W.cross_entropy_inputs(case, device=DEV)
    z = inp["logits"] + 1.0e4  # exp(z) overflows fp32 without the max shift
    loss, lse = L.cross_entropy_fw(z, inp["target"])
    torch.cuda.synchronize()
    rl, rs = oracle.cross_entropy_fw(z.cpu(), inp["target"].cpu())
    # lse ~ 1e4: an fp32 ulp there is ~1e-3, which bounds both outputs
    np.testing.assert_allclose(loss.cpu().numpy(), rl, atol=3e-3)
    np.testing.assert_allclose(lse.cpu().numpy(), rs, rtol=1e-6)


def test_ce_empty_problem():
    L = _L()
    z = torch.empty(0, 50257, device=DEV, dtype=torch.float16)
    t = torch.empty(0, device=DEV, dtype=torch.int32)
    loss, lse = L.cross_entropy_fw(z, t)
    dz = L.cross_entropy_bw(z, t, lse, torch.empty(0, device=DEV))
    torch.cuda.synchronize()
    assert loss.numel() == 0 and dz.numel() == 0
