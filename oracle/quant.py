"""INT8 quantisation of the pruned middle region (KIVI-style), in fp32 / fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix:
* LeanK article (framerc.cn) §4.2: LeanK stacks with KIVI quantisation;
  §5.2 problem 3: the order is prune -> reorganise -> quantise, so the
  quantiser sees K_prun (kept channels only) and the middle V rows.
* "Intelligent pruning white paper" (yyx235 blog) §5.2.1: KIVI quantises K
  per channel and V per token; INT8 is one of the named precisions.

Readings (the pages give no group size, rounding or scale formula):
* Middle rows of a (FULL, k > 0) head, in K_prun order (token t at row
  t - S), form blocks of 128 rows.  A block is quantised once all its 128 rows
  exist; the rows of the last, incomplete block stay bf16 -- KIVI's
  full-precision residual.
* K block [128, k]: one scale per channel, s_c = max_t |K[t, c]| / 127.
  V block [128, 128]: one scale per token, s_t = max_c |V[t, c]| / 127.
* Symmetric INT8: code = round_half_even(x / s) clipped to [-127, 127];
  s = 0 gives code 0.  Scales and quotients are fp32 with round-to-nearest
  (an fp32 decision that fixes integers, taken in the same precision the
  kernel stores the scale in).  The dequantised value is code * s.
"""
from __future__ import annotations

import numpy as np

from .attention import decode_head
from .footprint import resident_bytes as _resident_bytes_bf16

BLOCK_ROWS = 128
QMAX = 127


def _quantize(x: np.ndarray, absmax: np.ndarray):
    """Codes and fp32 scales for fp32 values x given the fp32 absmax that
    broadcasts against x."""
    x = np.asarray(x, dtype=np.float32)
    absmax = np.asarray(absmax, dtype=np.float32)
    scale = absmax / np.float32(QMAX)                      # fp32, round to nearest
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = np.rint(x / safe)                                  # fp32 quotient, half to even
    q = np.where(scale > 0, q, 0.0)
    codes = np.clip(q, -QMAX, QMAX).astype(np.int8)
    return codes, scale.astype(np.float32)


def quantize_per_channel(x: np.ndarray):
    """K block [R, C] -> (codes int8 [R, C], scales fp32 [C])."""
    x = np.asarray(x, dtype=np.float32)
    absmax = np.abs(x).max(axis=0)
    codes, scale = _quantize(x, absmax[None, :])
    return codes, scale.reshape(-1)


def quantize_per_token(x: np.ndarray):
    """V block [R, C] -> (codes int8 [R, C], scales fp32 [R])."""
    x = np.asarray(x, dtype=np.float32)
    absmax = np.abs(x).max(axis=1)
    codes, scale = _quantize(x, absmax[:, None])
    return codes, scale.reshape(-1)


def dequantize_per_channel(codes, scales) -> np.ndarray:
    return np.asarray(codes, np.float64) * np.asarray(scales, np.float64)[None, :]


def dequantize_per_token(codes, scales) -> np.ndarray:
    return np.asarray(codes, np.float64) * np.asarray(scales, np.float64)[:, None]


def sealed_blocks(n_kept: int, N: int, S: int, W: int) -> int:
    """Complete 128-row blocks of the middle region after N tokens."""
    if n_kept == 0:
        return 0
    return max(0, N - S - W) // BLOCK_ROWS


def middle_blocks(K, V, kept, N: int, S: int, W: int):
    """Per sealed block j: (k_codes [128, k], k_scales [k], v_codes [128, 128],
    v_scales [128]) of middle tokens S + 128 j .. S + 128 j + 127.
    K, V: dense history [>= N, d] of one kv head (bf16 values, any float type)."""
    kept = np.asarray(kept, dtype=np.int64)
    out = []
    for j in range(sealed_blocks(len(kept), N, S, W)):
        t0 = S + BLOCK_ROWS * j
        kb = np.asarray(K[t0:t0 + BLOCK_ROWS], dtype=np.float32)[:, kept]
        vb = np.asarray(V[t0:t0 + BLOCK_ROWS], dtype=np.float32)
        kc, ks = quantize_per_channel(kb)
        vc, vs = quantize_per_token(vb)
        out.append((kc, ks, vc, vs))
    return out


def quantized_history(K, V, kept, policy: int, N: int, S: int, W: int):
    """fp64 copies of the first N rows of the dense history where the middle
    tokens of sealed blocks hold their dequantised values (K on the kept
    channels, V on all), i.e. what a quantised cache represents.  Other rows
    are the exact inputs."""
    Kq = np.array(np.asarray(K[:N], dtype=np.float64))
    Vq = np.array(np.asarray(V[:N], dtype=np.float64))
    if policy != 0:
        return Kq, Vq
    kept = np.asarray(kept, dtype=np.int64)
    for j, (kc, ks, vc, vs) in enumerate(middle_blocks(K, V, kept, N, S, W)):
        t0 = S + BLOCK_ROWS * j
        rows = np.arange(t0, t0 + BLOCK_ROWS)
        Kq[np.ix_(rows, kept)] = dequantize_per_channel(kc, ks)
        Vq[rows] = dequantize_per_token(vc, vs)
    return Kq, Vq


def decode_head_quantized(q, K, V, policy: int, kept, N: int, S: int, W: int, W_loc: int,
                          special_flags=None) -> np.ndarray:
    """``attention.decode_head`` over the quantised cache's values."""
    Kq, Vq = quantized_history(K, V, kept, policy, N, S, W)
    return decode_head(q, Kq, Vq, policy, kept, N, S, W, W_loc, special_flags)


def resident_bytes_quantized(policy: int, n_kept: int, N: int, S: int, W: int, W_loc: int,
                             n_special: int = 0, head_dim: int = 128) -> int:
    """Bytes one decode step reads for one (b, kv head) of a cache whose
    complete middle blocks are quantised: the bf16 bytes of every row that is
    not in a sealed block (sinks, window, LOCAL / SPECIAL rows, the open
    middle block) plus, per sealed block, its int8 codes (128 x k for K,
    128 x d for V, one byte each) and fp32 scales (k for K, 128 for V)."""
    bf16 = _resident_bytes_bf16(policy, n_kept, N, S, W, W_loc, n_special, head_dim)
    nb = sealed_blocks(n_kept, N, S, W) if policy == 0 and 0 < n_kept else 0
    if nb == 0:
        return bf16
    mid_row_bf16 = (n_kept + head_dim) * 2
    block = BLOCK_ROWS * (n_kept + head_dim) + 4 * (n_kept + BLOCK_ROWS)
    return bf16 - nb * BLOCK_ROWS * mid_row_bf16 + nb * block
