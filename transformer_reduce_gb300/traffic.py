"""Algorithmic HBM bytes of each kernel: what the method must move, not what a
given kernel happens to move.  Roofline fractions divide these by the measured
time.  s = storage bytes per element; statistics and parameter gradients are
fp32.

Per row (Tk keys, N features):
  softmax fw : reads the v visible keys (v = unmasked, non-future), writes Tk
  softmax bw : reads out_fw and dout (2 Tk), writes dinp (Tk)
  softmax bw, masked : reads out_fw and dout on the v visible keys (2 v), writes Tk
  LN fw      : reads x (N), writes y (N) and mean, rstd (8 bytes)
  LN dinp    : reads dy, x (2N) and mean, rstd, writes dx (N)
  LN dg/db   : reads dy, x (2N) and mean, rstd
  LN bw, fused : reads dy, x (2N) and mean, rstd, writes dx (N)
  RMS fw     : reads x (N), writes y (N) and rstd (4 bytes)
  RMS dinp   : reads dy, x (2N) and rstd, writes dx (N)
  CE fw      : reads the V logits of each non-ignored row; per row the target
               (4 bytes) and loss, lse (8 bytes)
  CE bw      : reads the V logits of each non-ignored row; per row target, lse,
               dloss (12 bytes) and dlogits (V) written for every row
plus the per-call operands read once (mask [B, Tk]; gamma, beta [N]) and
written once (dgamma, dbeta [N] fp32).  The FastTransformer page's figure of
805 MB per step for writing and re-reading the (B,H,T,T) fp32 probability
tensor of a 6-layer B=32, H=8, T=256 decoder (section 3) is the fw write term
plus the bw out_fw read term of this model, times six layers.
"""
from __future__ import annotations

ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def visible_keys(T: int, lengths, causal: bool, H: int) -> int:
    """Sum over all rows (b, h, i) of the number of keys the row can see."""
    total = 0
    for n in lengths:
        if causal:
            # row i sees keys j <= i with j < n: min(i + 1, n) keys
            per_head = sum(min(i + 1, n) for i in range(T))
        else:
            per_head = n * T
        total += per_head * H
    return total


def softmax_fw_bytes(B, H, T, lengths, causal, dtype, has_mask=True) -> int:
    s = ELEM_BYTES[dtype]
    reads = visible_keys(T, lengths, causal, H) * s
    writes = B * H * T * T * s
    mask = B * T * s if has_mask else 0
    return reads + writes + mask


def softmax_fw_write_bytes(B, H, T, dtype) -> int:
    return B * H * T * T * ELEM_BYTES[dtype]


def softmax_bw_out_fw_read_bytes(B, H, T, dtype) -> int:
    return B * H * T * T * ELEM_BYTES[dtype]


def softmax_bw_bytes(B, H, T, dtype) -> int:
    return 3 * B * H * T * T * ELEM_BYTES[dtype]


def softmax_bw_masked_bytes(B, H, T, lengths, causal, dtype, has_mask=True) -> int:
    s = ELEM_BYTES[dtype]
    reads = 2 * visible_keys(T, lengths, causal, H) * s
    writes = B * H * T * T * s
    mask = B * T * s if has_mask else 0
    return reads + writes + mask


def layernorm_fw_bytes(rows, N, dtype) -> int:
    s = ELEM_BYTES[dtype]
    return rows * (2 * N * s + 8) + 2 * N * s


def layernorm_dinp_bytes(rows, N, dtype) -> int:
    s = ELEM_BYTES[dtype]
    return rows * (3 * N * s + 8) + N * s


def layernorm_dgdb_bytes(rows, N, dtype) -> int:
    s = ELEM_BYTES[dtype]
    return rows * (2 * N * s + 8) + 2 * N * 4


def layernorm_bw_fused_bytes(rows, N, dtype) -> int:
    """dx, dgamma and dbeta from one read of dy and x: the dinp bytes plus the
    two fp32 gradient vectors."""
    s = ELEM_BYTES[dtype]
    return rows * (3 * N * s + 8) + N * s + 2 * N * 4


def rmsnorm_fw_bytes(rows, N, dtype) -> int:
    s = ELEM_BYTES[dtype]
    return rows * (2 * N * s + 4) + N * s


def rmsnorm_dinp_bytes(rows, N, dtype) -> int:
    s = ELEM_BYTES[dtype]
    return rows * (3 * N * s + 4) + N * s


def cross_entropy_fw_bytes(rows, valid_rows, V, dtype) -> int:
    s = ELEM_BYTES[dtype]
    return valid_rows * V * s + rows * 12


def cross_entropy_bw_bytes(rows, valid_rows, V, dtype) -> int:
    s = ELEM_BYTES[dtype]
    return valid_rows * V * s + rows * (V * s + 12)
