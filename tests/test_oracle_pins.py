"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, an invariant, a
central finite difference, or an independent library routine (scipy /
torch float64 autograd -- the oracle itself is plain C and calls neither).
Together they are chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign, an off-by-one in the causal test, the mask indexed by the
wrong axis, eps outside the square root, N-1 instead of N) fails at least one
of them; ``test_oracle_mutants.py`` plants such slips and checks exactly that.

Sources: "CMU 11-868 L10: Accelerating Transformers on GPUs, and Where
LightSeq Finds the Time", "Technique 2" (slides 21-24); "CMU 11-868 HW4：把
Softmax 與 LayerNorm 寫成 CUDA 融合 kernel", section 題目結構與配分 (Problems
1.1-2.2, eps = 1e-8) and section 那些「快幾倍」是跟誰比 (softmax(inp + mask)).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

EPS = float(np.float32(1e-8))


def _padding_mask(lengths, tk):
    m = np.zeros((len(lengths), tk))
    for b, n in enumerate(lengths):
        m[b, n:] = -np.inf
    return m


# ----------------------------------------------------------------------------
# softmax forward
# ----------------------------------------------------------------------------

def test_softmax_fw_plain_rows_match_scipy(ref):
    rng = np.random.default_rng(11)
    x = rng.normal(0, 3, size=(37, 53))
    y = ref.softmax_fw(x)
    np.testing.assert_allclose(y, scipy.special.softmax(x, axis=-1), rtol=1e-13, atol=1e-16)


def test_softmax_fw_additive_mask_uses_batch_axis(ref):
    # Non-binary additive mask differing per batch entry; H != B so a mask
    # indexed by head instead of batch disagrees.
    rng = np.random.default_rng(12)
    B, H, T = 3, 2, 9
    x = rng.normal(0, 2, size=(B, H, T, T))
    mask = rng.normal(0, 1.5, size=(B, T))
    y = ref.softmax_fw_tensor(x, mask)
    want = scipy.special.softmax(x + mask[:, None, None, :], axis=-1)
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-16)


def test_softmax_fw_causal_and_padding_zero_pattern(ref):
    rng = np.random.default_rng(13)
    B, H, T = 3, 2, 11
    lengths = [11, 4, 7]
    x = rng.normal(0, 3, size=(B, H, T, T))
    mask = _padding_mask(lengths, T)
    y = ref.softmax_fw_tensor(x, mask, causal=True)
    for b in range(B):
        for h in range(H):
            for i in range(T):
                valid = np.array([(j <= i) and (j < lengths[b]) for j in range(T)])
                row = y[b, h, i]
                # future and padded keys are exactly zero, all others positive
                assert np.all(row[~valid] == 0.0)
                assert np.all(row[valid] > 0.0)
                assert abs(row.sum() - 1.0) < 1e-12
                np.testing.assert_allclose(
                    row[valid], scipy.special.softmax(x[b, h, i, valid]), rtol=1e-13)


def test_softmax_fw_closed_forms(ref):
    # two keys: the logistic function of the score difference
    x = np.array([[0.7, -1.9], [5.0, 5.0], [-30.0, 4.0]])
    y = ref.softmax_fw(x)
    for r in range(3):
        d = x[r, 0] - x[r, 1]
        assert y[r, 0] == pytest.approx(1.0 / (1.0 + math.exp(-d)), rel=1e-15)
        assert y[r, 1] == pytest.approx(1.0 / (1.0 + math.exp(d)), rel=1e-14)
    # equal valid scores: exactly 1/(number of valid keys)
    x = np.full((1, 8), 2.25)
    mask = _padding_mask([5], 8)
    y = ref.softmax_fw(x, mask, batch=[0])
    assert np.all(y[0, :5] == 0.2) and np.all(y[0, 5:] == 0.0)
    # a single key gets probability one
    assert ref.softmax_fw(np.array([[-123.5]]))[0, 0] == 1.0


def test_softmax_fw_shift_invariance_and_no_overflow(ref):
    rng = np.random.default_rng(14)
    x = rng.normal(0, 3, size=(5, 31))
    y0 = ref.softmax_fw(x)
    y1 = ref.softmax_fw(x + 1000.0)   # exp(1000) overflows without the max shift
    assert np.all(np.isfinite(y1))
    np.testing.assert_allclose(y1, y0, rtol=1e-10, atol=1e-15)


def test_softmax_fw_fully_masked_row_is_zero(ref):
    x = np.array([[1.0, 2.0, 3.0], [1.0, 2.0, 3.0]])
    mask = np.array([[-np.inf, -np.inf, -np.inf], [0.0, -np.inf, 0.0]])
    y = ref.softmax_fw(x, mask, batch=[0, 1])
    assert np.all(y[0] == 0.0)
    np.testing.assert_allclose(y[1], [1 / (1 + math.e ** 2), 0.0, math.e ** 2 / (1 + math.e ** 2)],
                               rtol=1e-15)


def test_softmax_fw_empty(ref):
    assert ref.softmax_fw(np.zeros((0, 7))).shape == (0, 7)
    assert ref.softmax_fw(np.zeros((3, 0))).shape == (3, 0)


# ----------------------------------------------------------------------------
# softmax backward
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("shape,causal,lengths", [
    ((1, 2, 3, 3), True, None),
    ((1, 1, 5, 5), True, [3]),
    ((2, 1, 4, 4), False, [2, 4]),
])
def test_softmax_bw_central_differences(ref, shape, causal, lengths):
    rng = np.random.default_rng(21)
    B, H, Tq, Tk = shape
    x = rng.normal(0, 1, size=shape)
    dy = rng.normal(0, 1, size=shape)
    mask = _padding_mask(lengths, Tk) if lengths else None

    def loss(xx):
        return float(np.sum(dy * ref.softmax_fw_tensor(xx, mask, causal=causal)))

    y = ref.softmax_fw_tensor(x, mask, causal=causal)
    dx = ref.softmax_bw(dy.reshape(-1, Tk), y.reshape(-1, Tk)).reshape(shape)
    h = 1e-6
    fd = np.zeros(shape)
    for idx in np.ndindex(shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (loss(xp) - loss(xm)) / (2 * h)
    scale = np.max(np.abs(fd))
    assert np.max(np.abs(dx - fd)) <= 1e-6 * scale


def test_softmax_bw_matches_torch_autograd(ref):
    rng = np.random.default_rng(22)
    B, H, T = 2, 3, 6
    x = torch.tensor(rng.normal(0, 2, size=(B, H, T, T)), requires_grad=True)
    dy = torch.tensor(rng.normal(0, 1, size=(B, H, T, T)))
    mask = torch.tensor(_padding_mask([6, 3], T))
    causal = torch.triu(torch.full((T, T), -math.inf, dtype=torch.float64), diagonal=1)
    y = torch.softmax(x + mask[:, None, None, :] + causal, dim=-1)
    y.backward(dy)
    yo = ref.softmax_fw_tensor(x.detach().numpy(), mask.numpy(), causal=True)
    np.testing.assert_allclose(yo, y.detach().numpy(), rtol=1e-13, atol=1e-16)
    dx = ref.softmax_bw(dy.numpy().reshape(-1, T), yo.reshape(-1, T)).reshape(B, H, T, T)
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_softmax_bw_invariants(ref):
    rng = np.random.default_rng(23)
    y = scipy.special.softmax(rng.normal(0, 2, size=(9, 17)), axis=-1)
    dy = rng.normal(0, 1, size=(9, 17))
    dx = ref.softmax_bw(dy, y)
    np.testing.assert_allclose(dx.sum(axis=-1), 0.0, atol=1e-14)
    # a constant upstream gradient has no effect on a normalised output
    dx_c = ref.softmax_bw(np.full((9, 17), 3.5), y)
    np.testing.assert_allclose(dx_c, 0.0, atol=1e-14)
    # zero probabilities give zero gradient whatever dy is
    y0 = y.copy()
    y0[:, :4] = 0.0
    assert np.all(ref.softmax_bw(dy, y0)[:, :4] == 0.0)


# ----------------------------------------------------------------------------
# LayerNorm forward
# ----------------------------------------------------------------------------

def test_layernorm_fw_matches_torch(ref):
    rng = np.random.default_rng(31)
    x = rng.normal(1, 2, size=(13, 96))
    g = rng.uniform(0.5, 1.5, size=96)
    b = rng.normal(0, 0.1, size=96)
    for eps in (EPS, 0.25):   # a large eps makes "eps inside the root" visible
        y, mean, rstd = ref.layernorm_fw(x, g, b, eps)
        want = torch.nn.functional.layer_norm(
            torch.tensor(x), (96,), torch.tensor(g), torch.tensor(b), eps)
        np.testing.assert_allclose(y, want.numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-14)
        np.testing.assert_allclose(rstd, 1 / np.sqrt(x.var(axis=1) + eps), rtol=1e-13)


def test_layernorm_fw_unit_affine_invariants(ref):
    rng = np.random.default_rng(32)
    x = rng.normal(0, 1, size=(64, 128))
    y, mean, rstd = ref.layernorm_fw(x, np.ones(128), np.zeros(128), EPS)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    var = x.var(axis=1)
    np.testing.assert_allclose(y.var(axis=1), var / (var + EPS), rtol=1e-12)
    # affine invariance: y(a x + c) = y(x) up to the eps term (a > 0)
    y2, _, _ = ref.layernorm_fw(3.0 * x - 7.0, np.ones(128), np.zeros(128), EPS)
    np.testing.assert_allclose(y2, y, rtol=1e-7, atol=1e-7)


def test_layernorm_fw_constant_row(ref):
    # dyadic constants: the mean is exact, so x - mean is exactly 0
    x = np.full((2, 40), 0.375)
    x[1] = -3.0
    g = np.linspace(0.5, 1.5, 40)
    b = np.linspace(-0.2, 0.2, 40)
    y, mean, rstd = ref.layernorm_fw(x, g, b, EPS)
    assert np.all(y == b)
    np.testing.assert_allclose(rstd, 1 / math.sqrt(EPS), rtol=1e-12)
    assert list(mean) == [0.375, -3.0]


def test_layernorm_fw_hand_example(ref):
    # x = [1,2,3,4]: mu = 2.5, population var = 1.25 (not 5/3)
    y, mean, rstd = ref.layernorm_fw(np.array([[1.0, 2, 3, 4]]), np.ones(4), np.zeros(4), 0.0)
    assert mean[0] == 2.5
    assert rstd[0] == pytest.approx(1 / math.sqrt(1.25), rel=1e-15)
    np.testing.assert_allclose(y[0], np.array([-1.5, -0.5, 0.5, 1.5]) / math.sqrt(1.25),
                               rtol=1e-15)


def test_one_pass_vs_two_pass_variance(ref):
    """The slide-21 rewrite agrees with the definition; fp32 accumulation loses digits."""
    assert ref.variance_one_pass([1.0, 2, 3, 4]) == 1.25
    assert ref.variance_two_pass([1.0, 2, 3, 4]) == 1.25
    rng = np.random.default_rng(33)
    worst_d, worst_f = 0.0, 0.0
    for n in (8, 128, 768, 8192):
        for mu, sd in ((0.0, 1.0), (1.0, 2.0)):
            row = rng.normal(mu, sd, size=n).astype(np.float32).astype(np.float64)
            v2 = ref.variance_two_pass(row)
            assert v2 == pytest.approx(np.var(row), rel=1e-13)
            worst_d = max(worst_d, abs(ref.variance_one_pass(row) - v2) / v2)
            worst_f = max(worst_f, abs(ref.variance_one_pass(row, single=True) - v2) / v2)
    assert worst_d < 1e-12            # same value in double
    assert 1e-9 < worst_f < 1e-3      # float accumulation: visibly fp32, still close
    # a large common offset makes the float form cancel catastrophically
    row = 1.0e4 + rng.normal(0, 1, size=1024)
    v2 = ref.variance_two_pass(row)
    assert abs(ref.variance_one_pass(row, single=True) - v2) / v2 > 0.1


# ----------------------------------------------------------------------------
# LayerNorm backward
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("rows,n", [(3, 5), (4, 8)])
def test_layernorm_dinp_central_differences(ref, rows, n):
    rng = np.random.default_rng(41)
    x = rng.normal(1, 2, size=(rows, n))
    g = rng.uniform(0.5, 1.5, size=n)
    b = rng.normal(0, 0.1, size=n)
    dy = rng.normal(0, 1, size=(rows, n))
    eps = 1e-3

    def loss(xx):
        return float(np.sum(dy * ref.layernorm_fw(xx, g, b, eps)[0]))

    _, mean, rstd = ref.layernorm_fw(x, g, b, eps)
    dx = ref.layernorm_bw_dinp(dy, x, g, mean, rstd)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (loss(xp) - loss(xm)) / (2 * h)
    assert np.max(np.abs(dx - fd)) <= 1e-6 * np.max(np.abs(fd))


def test_layernorm_bw_matches_torch_autograd(ref):
    rng = np.random.default_rng(42)
    rows, n = 7, 24
    x = torch.tensor(rng.normal(1, 2, size=(rows, n)), requires_grad=True)
    g = torch.tensor(rng.uniform(0.5, 1.5, size=n), requires_grad=True)
    b = torch.tensor(rng.normal(0, 0.1, size=n), requires_grad=True)
    dy = torch.tensor(rng.normal(0, 1, size=(rows, n)))
    torch.nn.functional.layer_norm(x, (n,), g, b, EPS).backward(dy)
    _, mean, rstd = ref.layernorm_fw(x.detach().numpy(), g.detach().numpy(),
                                     b.detach().numpy(), EPS)
    dx = ref.layernorm_bw_dinp(dy.numpy(), x.detach().numpy(), g.detach().numpy(), mean, rstd)
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-11, atol=1e-12)
    dg, db = ref.layernorm_bw_dgamma_dbeta(dy.numpy(), x.detach().numpy(), mean, rstd)
    np.testing.assert_allclose(dg, g.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(db, b.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_layernorm_dinp_row_sum_is_zero(ref):
    rng = np.random.default_rng(43)
    x = rng.normal(1, 2, size=(16, 33))
    g = rng.uniform(0.5, 1.5, size=33)
    _, mean, rstd = ref.layernorm_fw(x, g, np.zeros(33), EPS)
    dx = ref.layernorm_bw_dinp(rng.normal(size=(16, 33)), x, g, mean, rstd)
    np.testing.assert_allclose(dx.sum(axis=1), 0.0, atol=1e-12)


def test_layernorm_dgamma_dbeta_central_differences(ref):
    rng = np.random.default_rng(44)
    rows, n = 6, 5
    x = rng.normal(0, 1, size=(rows, n))
    g = rng.uniform(0.5, 1.5, size=n)
    b = rng.normal(0, 0.1, size=n)
    dy = rng.normal(0, 1, size=(rows, n))
    _, mean, rstd = ref.layernorm_fw(x, g, b, EPS)
    dg, db = ref.layernorm_bw_dgamma_dbeta(dy, x, mean, rstd)
    h = 1e-6
    for j in range(n):
        gp, gm = g.copy(), g.copy()
        gp[j] += h
        gm[j] -= h
        fd = (np.sum(dy * ref.layernorm_fw(x, gp, b, EPS)[0])
              - np.sum(dy * ref.layernorm_fw(x, gm, b, EPS)[0])) / (2 * h)
        assert dg[j] == pytest.approx(fd, rel=1e-6, abs=1e-8)
    # dbeta is the plain column sum of dy
    np.testing.assert_allclose(db, dy.sum(axis=0), rtol=1e-14)


def test_layernorm_empty_rows(ref):
    y, mean, rstd = ref.layernorm_fw(np.zeros((0, 4)), np.ones(4), np.zeros(4), EPS)
    assert y.shape == (0, 4) and mean.shape == (0,)
    dg, db = ref.layernorm_bw_dgamma_dbeta(np.zeros((0, 4)), np.zeros((0, 4)),
                                           np.zeros(0), np.zeros(0))
    assert np.all(dg == 0.0) and np.all(db == 0.0)


# ----------------------------------------------------------------------------
# causal with Tq < Tk (bottom-right alignment) and the masked backward
# ----------------------------------------------------------------------------

def test_softmax_fw_offset_is_the_tail_of_the_square_causal_problem(ref):
    # Tq queries over Tk keys, bottom-right aligned, are the last Tq rows of
    # the square causal problem over Tk keys (pinned above).
    rng = np.random.default_rng(51)
    Tq, Tk = 3, 7
    x = rng.normal(0, 2, size=(Tq, Tk))
    sq = rng.normal(0, 2, size=(Tk, Tk))
    sq[Tk - Tq:] = x
    mask = _padding_mask([6], Tk)
    want = ref.softmax_fw(sq, mask, batch=np.zeros(Tk, np.int64), query=np.arange(Tk),
                          causal=True)[Tk - Tq:]
    got = ref.softmax_fw_offset(x, mask, batch=np.zeros(Tq, np.int64), query=np.arange(Tq),
                                causal=True, offset=Tk - Tq)
    np.testing.assert_array_equal(got, want)
    # offset 0 on a square problem is the plain causal forward
    y0 = ref.softmax_fw_offset(sq, mask, batch=np.zeros(Tk, np.int64), query=np.arange(Tk),
                               causal=True, offset=0)
    np.testing.assert_array_equal(
        y0, ref.softmax_fw(sq, mask, batch=np.zeros(Tk, np.int64), query=np.arange(Tk), causal=True))


def test_softmax_bw_masked_central_differences(ref):
    rng = np.random.default_rng(52)
    B, H, Tq, Tk = 2, 1, 3, 5
    x = rng.normal(0, 1, size=(B, H, Tq, Tk))
    dy = rng.normal(0, 1, size=(B, H, Tq, Tk))
    mask = _padding_mask([4, 5], Tk)

    def loss(xx):
        return float(np.sum(dy * ref.softmax_fw_tensor_offset(xx, mask, causal=True)))

    y = ref.softmax_fw_tensor_offset(x, mask, causal=True)
    dx = ref.softmax_bw_masked_tensor(dy, y, mask, causal=True)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (loss(xp) - loss(xm)) / (2 * h)
    assert np.max(np.abs(dx - fd)) <= 1e-6 * np.max(np.abs(fd))


def test_softmax_bw_masked_matches_torch_autograd(ref):
    rng = np.random.default_rng(53)
    B, H, Tq, Tk = 2, 2, 4, 6
    x = torch.tensor(rng.normal(0, 2, size=(B, H, Tq, Tk)), requires_grad=True)
    dy = torch.tensor(rng.normal(0, 1, size=(B, H, Tq, Tk)))
    mask = torch.tensor(_padding_mask([6, 4], Tk))
    i = torch.arange(Tq).view(Tq, 1)
    j = torch.arange(Tk).view(1, Tk)
    future = torch.where(j > i + (Tk - Tq), -math.inf, 0.0).to(torch.float64)
    y = torch.softmax(x + mask[:, None, None, :] + future, dim=-1)
    y.backward(dy)
    yo = ref.softmax_fw_tensor_offset(x.detach().numpy(), mask.numpy(), causal=True)
    np.testing.assert_allclose(yo, y.detach().numpy(), rtol=1e-13, atol=1e-16)
    dx = ref.softmax_bw_masked_tensor(dy.numpy(), yo, mask.numpy(), causal=True)
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_softmax_bw_masked_ignores_invisible_inputs(ref):
    # Garbage in y / dy at invisible keys changes nothing and gives exact zeros.
    rng = np.random.default_rng(54)
    B, H, Tq, Tk = 2, 2, 5, 5
    mask = _padding_mask([3, 5], Tk)
    y = ref.softmax_fw_tensor_offset(rng.normal(size=(B, H, Tq, Tk)), mask, causal=True)
    dy = rng.normal(size=(B, H, Tq, Tk))
    invisible = (y == 0.0)
    y_dirty, dy_dirty = y.copy(), dy.copy()
    y_dirty[invisible] = rng.uniform(1, 2, size=int(invisible.sum()))
    dy_dirty[invisible] = 1e6
    dx = ref.softmax_bw_masked_tensor(dy_dirty, y_dirty, mask, causal=True)
    assert np.all(dx[invisible] == 0.0)
    np.testing.assert_allclose(dx, ref.softmax_bw(dy.reshape(-1, Tk), y.reshape(-1, Tk)).reshape(y.shape),
                               rtol=1e-13, atol=1e-16)


# ----------------------------------------------------------------------------
# RMSNorm (FastTransformer page, section 5.4)
# ----------------------------------------------------------------------------

def test_rmsnorm_fw_matches_torch(ref):
    rng = np.random.default_rng(71)
    x = rng.normal(1, 2, size=(11, 40))
    g = rng.uniform(0.5, 1.5, size=40)
    for eps in (1e-6, 0.5):   # a large eps shows where it enters
        y, rstd = ref.rmsnorm_fw(x, g, eps)
        want = torch.nn.functional.rms_norm(torch.tensor(x), (40,), torch.tensor(g), eps)
        np.testing.assert_allclose(y, want.numpy(), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(rstd, 1 / np.sqrt((x * x).mean(axis=1) + eps), rtol=1e-14)


def test_rmsnorm_fw_closed_forms(ref):
    # a constant row c: y = c / sqrt(c^2 + eps) * gamma; with gamma = 1 the
    # output's mean square is ms / (ms + eps)
    x = np.full((1, 16), -2.5)
    g = np.linspace(0.5, 1.5, 16)
    y, rstd = ref.rmsnorm_fw(x, g, 1e-6)
    np.testing.assert_allclose(y[0], -2.5 / math.sqrt(6.25 + 1e-6) * g, rtol=1e-15)
    rng = np.random.default_rng(72)
    x = rng.normal(0, 3, size=(9, 64))
    y, rstd = ref.rmsnorm_fw(x, np.ones(64), 1e-3)
    ms = (x * x).mean(axis=1)
    np.testing.assert_allclose((y * y).mean(axis=1), ms / (ms + 1e-3), rtol=1e-13)
    # no mean centring: a shifted row is NOT normalised to the same output
    y2, _ = ref.rmsnorm_fw(x + 5.0, np.ones(64), 1e-3)
    assert np.max(np.abs(y2 - y)) > 0.1


@pytest.mark.parametrize("rows,n", [(3, 5), (4, 9)])
def test_rmsnorm_bw_central_differences(ref, rows, n):
    rng = np.random.default_rng(73)
    x = rng.normal(0.5, 1.5, size=(rows, n))
    g = rng.uniform(0.5, 1.5, size=n)
    dy = rng.normal(size=(rows, n))
    eps = 1e-3

    def loss(xx, gg):
        return float(np.sum(dy * ref.rmsnorm_fw(xx, gg, eps)[0]))

    _, rstd = ref.rmsnorm_fw(x, g, eps)
    dx = ref.rmsnorm_bw_dinp(dy, x, g, rstd)
    dg = ref.rmsnorm_bw_dgamma(dy, x, rstd)
    h = 1e-6
    fdx = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fdx[idx] = (loss(xp, g) - loss(xm, g)) / (2 * h)
    assert np.max(np.abs(dx - fdx)) <= 1e-6 * np.max(np.abs(fdx))
    for j in range(n):
        gp, gm = g.copy(), g.copy()
        gp[j] += h
        gm[j] -= h
        assert dg[j] == pytest.approx((loss(x, gp) - loss(x, gm)) / (2 * h), rel=1e-6, abs=1e-8)


def test_rmsnorm_bw_matches_torch_autograd(ref):
    rng = np.random.default_rng(74)
    rows, n = 6, 33
    x = torch.tensor(rng.normal(1, 2, size=(rows, n)), requires_grad=True)
    g = torch.tensor(rng.uniform(0.5, 1.5, size=n), requires_grad=True)
    dy = torch.tensor(rng.normal(size=(rows, n)))
    torch.nn.functional.rms_norm(x, (n,), g, 1e-6).backward(dy)
    _, rstd = ref.rmsnorm_fw(x.detach().numpy(), g.detach().numpy(), 1e-6)
    np.testing.assert_allclose(ref.rmsnorm_bw_dinp(dy.numpy(), x.detach().numpy(), g.detach().numpy(), rstd),
                               x.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ref.rmsnorm_bw_dgamma(dy.numpy(), x.detach().numpy(), rstd),
                               g.grad.numpy(), rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------
# cross entropy over a vocabulary (L10 page, "Technique 1", slide 12: the
# third reduce kernel; the textbook softmax cross entropy)
# ----------------------------------------------------------------------------

def test_cross_entropy_fw_closed_forms(ref):
    # equal logits: every class has probability 1/V, loss = log V
    z = np.full((3, 7), 0.375)
    loss, lse = ref.cross_entropy_fw(z, np.array([0, 3, 6]))
    np.testing.assert_allclose(loss, math.log(7), rtol=1e-15)
    np.testing.assert_allclose(lse, 0.375 + math.log(7), rtol=1e-15)
    # two classes: loss = log(1 + exp(other - target)), the softplus
    a, b = 1.25, -0.5
    loss, _ = ref.cross_entropy_fw(np.array([[a, b], [a, b]]), np.array([0, 1]))
    assert loss[0] == pytest.approx(math.log1p(math.exp(b - a)), rel=1e-14)
    assert loss[1] == pytest.approx(math.log1p(math.exp(a - b)), rel=1e-14)


def test_cross_entropy_fw_matches_scipy_and_torch(ref):
    rng = np.random.default_rng(81)
    rows, v = 19, 301
    z = rng.normal(0, 3, size=(rows, v))
    t = rng.integers(0, v, size=rows)
    loss, lse = ref.cross_entropy_fw(z, t)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=1), rtol=1e-14)
    want = torch.nn.functional.cross_entropy(torch.tensor(z), torch.tensor(t), reduction="none")
    np.testing.assert_allclose(loss, want.numpy(), rtol=1e-12, atol=1e-13)
    # exp(-loss) is the softmax probability of the target class
    p = ref.softmax_fw(z)
    np.testing.assert_allclose(np.exp(-loss), p[np.arange(rows), t], rtol=1e-12)


def test_cross_entropy_fw_large_logits_and_shift(ref):
    rng = np.random.default_rng(82)
    z = rng.normal(0, 1, size=(4, 50))
    t = np.array([0, 7, 49, 21])
    loss, lse = ref.cross_entropy_fw(z, t)
    loss2, lse2 = ref.cross_entropy_fw(z + 1.0e4, t)  # exp would overflow without the max shift
    assert np.all(np.isfinite(loss2))
    np.testing.assert_allclose(loss2, loss, atol=1e-9)
    np.testing.assert_allclose(lse2 - 1.0e4, lse, atol=1e-9)


def test_cross_entropy_ignored_and_out_of_range_targets(ref):
    rng = np.random.default_rng(83)
    z = rng.normal(0, 2, size=(4, 9))
    t = np.array([-1, 3, 9, -100])
    loss, lse = ref.cross_entropy_fw(z, t)
    assert loss[0] == 0.0 and lse[0] == 0.0 and loss[3] == 0.0 and lse[3] == 0.0
    assert math.isnan(loss[2]) and math.isnan(lse[2])
    assert loss[1] == pytest.approx(scipy.special.logsumexp(z[1]) - z[1, 3], rel=1e-14)
    dz = ref.cross_entropy_bw(z, t, lse, np.ones(4))
    assert np.all(dz[0] == 0.0) and np.all(dz[3] == 0.0) and np.all(np.isnan(dz[2]))
    # NaN for a target >= V even when the saved log-sum-exp is finite
    assert np.all(np.isnan(ref.cross_entropy_bw(z, t, np.zeros(4), np.ones(4))[2]))
    # an ignored row is not read: NaN logits there change nothing
    z2 = z.copy()
    z2[0] = np.nan
    l2, s2 = ref.cross_entropy_fw(z2, t)
    assert l2[0] == 0.0 and s2[0] == 0.0
    assert np.all(ref.cross_entropy_bw(z2, t, s2, np.ones(4))[0] == 0.0)


@pytest.mark.parametrize("rows,v", [(3, 5), (2, 11)])
def test_cross_entropy_bw_central_differences(ref, rows, v):
    rng = np.random.default_rng(84)
    z = rng.normal(0, 2, size=(rows, v))
    t = rng.integers(0, v, size=rows)
    dloss = rng.uniform(0.5, 2.0, size=rows)

    def total(zz):
        return float(np.sum(dloss * ref.cross_entropy_fw(zz, t)[0]))

    _, lse = ref.cross_entropy_fw(z, t)
    dz = ref.cross_entropy_bw(z, t, lse, dloss)
    h = 1e-6
    fd = np.zeros_like(z)
    for idx in np.ndindex(z.shape):
        zp, zm = z.copy(), z.copy()
        zp[idx] += h
        zm[idx] -= h
        fd[idx] = (total(zp) - total(zm)) / (2 * h)
    assert np.max(np.abs(dz - fd)) <= 1e-7 * max(1.0, np.max(np.abs(fd)))
    # rows of the gradient sum to zero; only the target entry is negative
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-14)
    for r in range(rows):
        assert dz[r, t[r]] < 0 and np.all(np.delete(dz[r], t[r]) > 0)


def test_cross_entropy_bw_matches_torch_autograd(ref):
    rng = np.random.default_rng(85)
    rows, v = 7, 129
    z = torch.tensor(rng.normal(0, 3, size=(rows, v)), requires_grad=True)
    t = torch.tensor(rng.integers(0, v, size=rows))
    dl = torch.tensor(rng.normal(size=rows))
    torch.nn.functional.cross_entropy(z, t, reduction="none").backward(dl)
    _, lse = ref.cross_entropy_fw(z.detach().numpy(), t.numpy())
    np.testing.assert_allclose(ref.cross_entropy_bw(z.detach().numpy(), t.numpy(), lse, dl.numpy()),
                               z.grad.numpy(), rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------
# scaled softmax (the fused "scale + mask + softmax"): z = scale * x + mask
# ----------------------------------------------------------------------------

def _torch_scaled_softmax(x4, mask, causal, scale):
    B, H, Tq, Tk = x4.shape
    z = scale * x4 + torch.as_tensor(mask).view(B, 1, 1, Tk)
    if causal:
        i = torch.arange(Tq).view(Tq, 1)
        j = torch.arange(Tk).view(1, Tk)
        z = z.masked_fill(j > i + (Tk - Tq), float("-inf"))
    return torch.softmax(z, dim=-1)


@pytest.mark.parametrize("causal,Tq,Tk", [(False, 7, 7), (True, 5, 9), (True, 6, 6)])
def test_scaled_softmax_matches_torch_autograd(ref, causal, Tq, Tk):
    rng = np.random.default_rng(91)
    B, H, scale = 2, 3, 0.125
    x = torch.tensor(rng.normal(0, 3, size=(B, H, Tq, Tk)), requires_grad=True)
    mask = rng.normal(0, 1, size=(B, Tk))  # a non-binary additive bias
    mask[0, Tk - 2:] = -np.inf
    dy = torch.tensor(rng.normal(size=(B, H, Tq, Tk)))
    yt = _torch_scaled_softmax(x, mask, causal, scale)
    yt.backward(dy)
    y = ref.softmax_fw_tensor_scaled(x.detach().numpy(), mask, causal=causal, scale=scale)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-15)
    dx = ref.softmax_bw_masked_scaled_tensor(dy.numpy(), y, mask, causal=causal, scale=scale)
    np.testing.assert_allclose(dx, x.grad.numpy(), rtol=1e-10, atol=1e-13)


def test_scaled_softmax_reduces_to_the_unscaled_one(ref):
    rng = np.random.default_rng(92)
    x = rng.normal(0, 2, size=(4, 2, 6, 10))
    mask = _padding_mask([7, 10, 3, 9], 10)
    # scale 2: z = 2x + mask exactly, the unscaled softmax of 2x
    y2 = ref.softmax_fw_tensor_scaled(x, mask, causal=True, scale=2.0)
    assert np.array_equal(y2, ref.softmax_fw_tensor_offset(2.0 * x, mask, causal=True))
    y1 = ref.softmax_fw_tensor_scaled(x, mask, causal=True, scale=1.0)
    dy = rng.normal(size=x.shape)
    assert np.array_equal(ref.softmax_bw_masked_scaled_tensor(dy, y1, mask, causal=True, scale=1.0),
                          ref.softmax_bw_masked_tensor(dy, y1, mask, causal=True))
    # scale 0.5 on the backward is half the unscaled backward, exactly
    assert np.array_equal(ref.softmax_bw_masked_scaled_tensor(dy, y1, mask, causal=True, scale=0.5),
                          0.5 * ref.softmax_bw_masked_tensor(dy, y1, mask, causal=True))


def test_scaled_softmax_bw_central_differences(ref):
    rng = np.random.default_rng(93)
    B, H, Tq, Tk, scale = 1, 2, 3, 5, 0.35
    x = rng.normal(0, 1.5, size=(B, H, Tq, Tk))
    mask = np.array([[0.0, 0.5, -np.inf, -0.25, 0.0]])
    dy = rng.normal(size=x.shape)

    def loss(xx):
        return float(np.sum(dy * ref.softmax_fw_tensor_scaled(xx, mask, causal=True, scale=scale)))

    y = ref.softmax_fw_tensor_scaled(x, mask, causal=True, scale=scale)
    dx = ref.softmax_bw_masked_scaled_tensor(dy, y, mask, causal=True, scale=scale)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (loss(xp) - loss(xm)) / (2 * h)
    assert np.max(np.abs(dx - fd)) <= 1e-7
    # masked key 2 and (bottom-right causal, offset 2) keys j > i + 2 are exactly 0
    assert np.all(y[..., 2] == 0) and np.all(dx[..., 2] == 0)
    assert np.all(y[:, :, 0, 3:] == 0) and np.all(y[:, :, 1, 4:] == 0)
