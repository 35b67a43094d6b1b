"""Seeded synthetic workloads for the softmax / LayerNorm reduce path.

This module only draws random inputs; it holds none of the method's
arithmetic.  The tests feed the same tensors to the CUDA library and to the
CPU oracle, and the benchmark times the library on them.

The shapes follow the pages' own workloads: the GPT-2 decoder of
"FastTransformer: Breaking the Compiler Ceiling via Architectural Co-Design"
(section 1: B=32, T=256, C=256, H=8; section 2: 8,192 tokens per step), the
softmax length buckets {32, ..., 2048} of "CMU 11-868 HW4：把 Softmax 與
LayerNorm 寫成 CUDA 融合 kernel" (Problem 1.2), and a Transformer-big encoder
layer (the LightSeq setting of the L10 page).  No dataset is involved.

Recipe: every tensor is drawn by torch's generator on the requested device
from a seed derived from (config seed, tensor name), in float32, then
rounded to the storage dtype (round to nearest even).  Padding lengths are
drawn on the CPU.  The additive mask is 0 on valid keys and -inf on padded
keys.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
LN_EPS = 1e-8  # the HW4 page, Problem 2.1


@dataclasses.dataclass(frozen=True)
class SoftmaxCase:
    name: str
    B: int
    H: int
    T: int                     # Tq == Tk
    causal: bool
    pad: Optional[tuple]       # (lo, hi) inclusive per-batch valid length, or None
    score_std: float
    dtype: str
    seed: int

    @property
    def shape(self):
        return (self.B, self.H, self.T, self.T)

    @property
    def rows(self):
        return self.B * self.H * self.T


@dataclasses.dataclass(frozen=True)
class LayerNormCase:
    name: str
    rows: int
    hidden: int
    x_mean: float
    x_std: float
    dtype: str
    seed: int
    eps: float = LN_EPS


SWEEP_T = (32, 64, 128, 256, 384, 512, 768, 1024, 2048)
SWEEP_HIDDEN = (768, 1024, 2048, 4096, 8192)

# The five configurations.  Seeds: 0 for the tiny layer, 1-4 for the others.
TINY = {
    "softmax": SoftmaxCase("tiny", 2, 4, 32, True, (16, 32), 3.0, "f32", 0),
    "layernorm": LayerNormCase("tiny", 64, 128, 0.0, 1.0, "f32", 0),
}
GPT2_SMALL = {
    "softmax": SoftmaxCase("gpt2_small", 32, 8, 256, True, None, 2.0, "f16", 1),
    "layernorm": LayerNormCase("gpt2_small", 8192, 256, 0.0, 1.0, "f16", 1),
}
SOFTMAX_SWEEP = [SoftmaxCase(f"softmax_T{T}", 8, 16, T, False, (T // 2, T), 3.0, "bf16", 2)
                 for T in SWEEP_T]
LAYERNORM_SWEEP = [LayerNormCase(f"layernorm_N{N}", 16384, N, 1.0, 2.0, "bf16", 3)
                   for N in SWEEP_HIDDEN]
# Transformer-big encoder layer: one attention softmax and two LayerNorms,
# value distributions as in the two sweeps.
ENCODER_BIG = {
    "softmax": SoftmaxCase("encoder_big", 32, 16, 512, False, (256, 512), 3.0, "bf16", 4),
    "layernorm": [LayerNormCase("encoder_big_ln1", 16384, 1024, 1.0, 2.0, "bf16", 4),
                  LayerNormCase("encoder_big_ln2", 16384, 1024, 1.0, 2.0, "bf16", 5)],
}


def sub_seed(seed: int, name: str) -> int:
    return (seed * 1_000_003 + zlib.crc32(name.encode())) % (2 ** 63)


def _gen(device, seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, name))
    return g


def _normal(shape, mean, std, dtype, device, seed, name):
    g = _gen(device, seed, name)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def _uniform(shape, lo, hi, dtype, device, seed, name):
    g = _gen(device, seed, name)
    t = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo).to(dtype)


def padding_lengths(case: SoftmaxCase):
    """Per-batch valid key counts (all T when the case has no padding)."""
    if case.pad is None:
        return [case.T] * case.B
    g = torch.Generator().manual_seed(sub_seed(case.seed, "softmax.lengths"))
    lo, hi = case.pad
    return torch.randint(lo, hi + 1, (case.B,), generator=g).tolist()


def padding_mask(lengths, T: int, dtype, device):
    m = torch.zeros(len(lengths), T, dtype=torch.float32)
    for b, n in enumerate(lengths):
        m[b, n:] = -math.inf
    return m.to(dtype).to(device)


def softmax_inputs(case: SoftmaxCase, device="cpu"):
    """scores ~ N(0, std^2), mask [B, T] (or None), dout ~ N(0, 1)."""
    dt = DTYPES[case.dtype]
    lengths = padding_lengths(case)
    return {
        "scores": _normal(case.shape, 0.0, case.score_std, dt, device, case.seed, "softmax.x"),
        "mask": padding_mask(lengths, case.T, dt, device) if case.pad is not None else None,
        "dout": _normal(case.shape, 0.0, 1.0, dt, device, case.seed, "softmax.dy"),
        "lengths": lengths,
    }


def softmax_probability_like(case: SoftmaxCase, lengths, device="cpu"):
    """A stand-in forward output for backward tests at full size: uniform
    values in [0, 2/v) on the keys a row can see (v of them), exactly 0 on
    masked and future keys.  The backward formula holds for any such tensor."""
    dt = DTYPES[case.dtype]
    B, H, T, _ = case.shape
    u = _uniform(case.shape, 0.0, 1.0, torch.float32, device, case.seed, "softmax.yfake")
    j = torch.arange(T, device=device)
    visible = j.view(1, 1, 1, T) < torch.tensor(lengths, device=device).view(B, 1, 1, 1)
    if case.causal:
        visible = visible & (j.view(1, 1, 1, T) <= j.view(1, 1, T, 1))
    v = visible.sum(-1, keepdim=True).clamp(min=1).to(torch.float32)
    return torch.where(visible, u * (2.0 / v), torch.zeros((), device=device)).to(dt)


def layernorm_inputs(case: LayerNormCase, device="cpu"):
    """x ~ N(mean, std^2), gamma ~ U(0.5, 1.5), beta ~ N(0, 0.1^2), dy ~ N(0, 1)."""
    dt = DTYPES[case.dtype]
    shape = (case.rows, case.hidden)
    return {
        "x": _normal(shape, case.x_mean, case.x_std, dt, device, case.seed, "ln.x"),
        "gamma": _uniform((case.hidden,), 0.5, 1.5, dt, device, case.seed, "ln.gamma"),
        "beta": _normal((case.hidden,), 0.0, 0.1, dt, device, case.seed, "ln.beta"),
        "dy": _normal(shape, 0.0, 1.0, dt, device, case.seed, "ln.dy"),
    }


# ----------------------------------------------------------------------------
# cross entropy over a vocabulary
# ----------------------------------------------------------------------------
# One row per token: the GPT-2 decoder step above has B*T = 8,192 tokens.  The
# pages give no vocabulary size; the stand-ins are GPT-2's byte-pair vocabulary
# (50,257 entries: rows start off the 16-byte grid), the same padded to a
# multiple of 64 (50,304), and a character vocabulary of 65 symbols for the
# small case (the FastTransformer page trains on TinyShakespeare).
@dataclasses.dataclass(frozen=True)
class CrossEntropyCase:
    name: str
    B: int
    T: int
    vocab: int
    pad: Optional[tuple]       # (lo, hi) valid tokens per sequence; the rest are ignored
    logit_std: float
    dtype: str
    seed: int

    @property
    def rows(self):
        return self.B * self.T


CE_TINY = CrossEntropyCase("ce_tiny", 2, 32, 65, (16, 32), 3.0, "f32", 0)
CE_GPT2 = CrossEntropyCase("ce_gpt2", 32, 256, 50257, None, 3.0, "f16", 1)
CE_GPT2_PADDED = CrossEntropyCase("ce_gpt2_v50304", 32, 256, 50304, None, 3.0, "bf16", 1)
CE_CASES = [CE_TINY, CE_GPT2, CE_GPT2_PADDED]


def cross_entropy_inputs(case: CrossEntropyCase, device="cpu"):
    """logits ~ N(0, std^2) [rows, vocab]; int32 targets uniform in [0, vocab),
    -1 on the padded positions of each sequence; dloss = 1 / (valid rows)
    on valid rows (a mean loss) and 0 elsewhere."""
    dt = DTYPES[case.dtype]
    logits = _normal((case.rows, case.vocab), 0.0, case.logit_std, dt, device, case.seed,
                     "ce.logits")
    g = torch.Generator().manual_seed(sub_seed(case.seed, "ce.target"))
    target = torch.randint(0, case.vocab, (case.rows,), generator=g, dtype=torch.int64)
    if case.pad is not None:
        g2 = torch.Generator().manual_seed(sub_seed(case.seed, "ce.lengths"))
        lens = torch.randint(case.pad[0], case.pad[1] + 1, (case.B,), generator=g2)
        pos = torch.arange(case.T).view(1, case.T)
        target = torch.where(pos < lens.view(case.B, 1), target.view(case.B, case.T),
                             torch.full((), -1, dtype=torch.int64)).reshape(-1)
    valid = target >= 0
    dloss = valid.to(torch.float32) / max(1, int(valid.sum()))
    return {
        "logits": logits,
        "target": target.to(torch.int32).to(device),
        "dloss": dloss.to(device),
    }
