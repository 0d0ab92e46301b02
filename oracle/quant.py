"""Quantisation of the pruned middle region (KIVI-style), INT8 or FP8 (e4m3),
in fp32 / fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix:
* LeanK article (framerc.cn) §4.2: LeanK stacks with KIVI quantisation;
  §5.2 problem 3: the order is prune -> reorganise -> quantise, so the
  quantiser sees K_prun (kept channels only) and the middle V rows.
* "Intelligent pruning white paper" (yyx235 blog) §5.2.1: KIVI quantises K
  per channel and V per token; INT8 is one of the named precisions, and
  FP8 is one of the low-precision formats it lists.

Readings (the pages give no group size, rounding, scale formula or FP8
variant):
* Middle rows of a (FULL, k > 0) head, in K_prun order (token t at row
  t - S), form blocks of 128 rows.  A block is quantised once all its 128 rows
  exist; the rows of the last, incomplete block stay bf16 -- KIVI's
  full-precision residual.
* K block [128, k]: one scale per channel; V block [128, 128]: one scale per
  token.  The scale is absmax / Q with Q the format's largest code value,
  in fp32 round-to-nearest; s = 0 gives code 0.  The quotient x / s is fp32
  round-to-nearest (an fp32 decision that fixes integers, taken in the same
  precision the kernel stores the scale in).
* INT8: symmetric, Q = 127, code = round_half_even(x / s) clipped to
  [-127, 127].
* FP8: the OCP 8-bit e4m3 format (1 sign, 4 exponent bits with bias 7, 3
  mantissa bits; exponent 0 holds the subnormals m * 2^-9; no infinities;
  S.1111.111 is NaN, so the largest finite value is 448), Q = 448, code =
  x / s rounded to the nearest e4m3 value, ties to the even code, |x / s|
  beyond 448 saturated to 448; the sign of x stays in the code, zero
  included.
* The dequantised value is value(code) * s.
"""
from __future__ import annotations

import numpy as np

from .attention import decode_head
from .footprint import resident_bytes as _resident_bytes_bf16

BLOCK_ROWS = 128
QMAX = 127
FP8_MAX = 448.0
FORMATS = ("int8", "fp8")


def e4m3_value(code) -> np.ndarray:
    """The value of e4m3 codes (uint8; NaN for S.1111.111), from the format's
    fields: (-1)^S * 2^(E - 7) * (1 + M / 8) for E > 0, (-1)^S * M * 2^-9 for
    E = 0."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, 2.0 ** (e - 7.0) * (1.0 + m / 8.0))
    return np.where((c & 0x7F) == 0x7F, np.nan, sign * mag)


_E4M3_POS = e4m3_value(np.arange(0x7F))        # codes 0x00 .. 0x7E: ascending magnitudes


def encode_e4m3(x) -> np.ndarray:
    """fp32 values -> e4m3 codes (uint8): the nearest finite e4m3 magnitude,
    ties to the even code, saturated at 448; the sign bit of x is kept."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, len(_E4M3_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = np.abs(a - _E4M3_POS[lo])
    d_hi = np.abs(_E4M3_POS[hi] - a)
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= _E4M3_POS[-1], len(_E4M3_POS) - 1, pick)
    return (pick | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def _quantize(x: np.ndarray, absmax: np.ndarray, fmt: str = "int8"):
    """Codes and fp32 scales for fp32 values x given the fp32 absmax that
    broadcasts against x.  int8: int8 codes; fp8: e4m3 codes (uint8)."""
    x = np.asarray(x, dtype=np.float32)
    absmax = np.asarray(absmax, dtype=np.float32)
    qmax = np.float32(QMAX if fmt == "int8" else FP8_MAX)
    scale = absmax / qmax                                  # fp32, round to nearest
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    y = (x / safe).astype(np.float32)                      # fp32 quotient
    if fmt == "int8":
        q = np.where(scale > 0, np.rint(y), 0.0)           # half to even
        codes = np.clip(q, -QMAX, QMAX).astype(np.int8)
    elif fmt == "fp8":
        codes = np.where(scale > 0, encode_e4m3(y), np.uint8(0)).astype(np.uint8)
    else:
        raise ValueError(fmt)
    return codes, scale.astype(np.float32)


def code_value(codes, fmt: str = "int8") -> np.ndarray:
    """fp64 values of codes."""
    return np.asarray(codes, np.float64) if fmt == "int8" else e4m3_value(codes)


def quantize_per_channel(x: np.ndarray, fmt: str = "int8"):
    """K block [R, C] -> (codes [R, C], scales fp32 [C])."""
    x = np.asarray(x, dtype=np.float32)
    absmax = np.abs(x).max(axis=0)
    codes, scale = _quantize(x, absmax[None, :], fmt)
    return codes, scale.reshape(-1)


def quantize_per_token(x: np.ndarray, fmt: str = "int8"):
    """V block [R, C] -> (codes [R, C], scales fp32 [R])."""
    x = np.asarray(x, dtype=np.float32)
    absmax = np.abs(x).max(axis=1)
    codes, scale = _quantize(x, absmax[:, None], fmt)
    return codes, scale.reshape(-1)


def dequantize_per_channel(codes, scales, fmt: str = "int8") -> np.ndarray:
    return code_value(codes, fmt) * np.asarray(scales, np.float64)[None, :]


def dequantize_per_token(codes, scales, fmt: str = "int8") -> np.ndarray:
    return code_value(codes, fmt) * np.asarray(scales, np.float64)[:, None]


def sealed_blocks(n_kept: int, N: int, S: int, W: int) -> int:
    """Complete 128-row blocks of the middle region after N tokens."""
    if n_kept == 0:
        return 0
    return max(0, N - S - W) // BLOCK_ROWS


def middle_blocks(K, V, kept, N: int, S: int, W: int, fmt: str = "int8"):
    """Per sealed block j: (k_codes [128, k], k_scales [k], v_codes [128, 128],
    v_scales [128]) of middle tokens S + 128 j .. S + 128 j + 127.
    K, V: dense history [>= N, d] of one kv head (bf16 values, any float type)."""
    kept = np.asarray(kept, dtype=np.int64)
    out = []
    for j in range(sealed_blocks(len(kept), N, S, W)):
        t0 = S + BLOCK_ROWS * j
        kb = np.asarray(K[t0:t0 + BLOCK_ROWS], dtype=np.float32)[:, kept]
        vb = np.asarray(V[t0:t0 + BLOCK_ROWS], dtype=np.float32)
        kc, ks = quantize_per_channel(kb, fmt)
        vc, vs = quantize_per_token(vb, fmt)
        out.append((kc, ks, vc, vs))
    return out


def quantized_history(K, V, kept, policy: int, N: int, S: int, W: int, fmt: str = "int8"):
    """fp64 copies of the first N rows of the dense history where the middle
    tokens of sealed blocks hold their dequantised values (K on the kept
    channels, V on all), i.e. what a quantised cache represents.  Other rows
    are the exact inputs."""
    Kq = np.array(np.asarray(K[:N], dtype=np.float64))
    Vq = np.array(np.asarray(V[:N], dtype=np.float64))
    if policy != 0:
        return Kq, Vq
    kept = np.asarray(kept, dtype=np.int64)
    for j, (kc, ks, vc, vs) in enumerate(middle_blocks(K, V, kept, N, S, W, fmt)):
        t0 = S + BLOCK_ROWS * j
        rows = np.arange(t0, t0 + BLOCK_ROWS)
        Kq[np.ix_(rows, kept)] = dequantize_per_channel(kc, ks, fmt)
        Vq[rows] = dequantize_per_token(vc, vs, fmt)
    return Kq, Vq


def decode_head_quantized(q, K, V, policy: int, kept, N: int, S: int, W: int, W_loc: int,
                          special_flags=None, fmt: str = "int8") -> np.ndarray:
    """``attention.decode_head`` over the quantised cache's values."""
    Kq, Vq = quantized_history(K, V, kept, policy, N, S, W, fmt)
    return decode_head(q, Kq, Vq, policy, kept, N, S, W, W_loc, special_flags)


def resident_bytes_quantized(policy: int, n_kept: int, N: int, S: int, W: int, W_loc: int,
                             n_special: int = 0, head_dim: int = 128) -> int:
    """Bytes one decode step reads for one (b, kv head) of a cache whose
    complete middle blocks are quantised (INT8 or FP8: one byte per code): the
    bf16 bytes of every row that is not in a sealed block (sinks, window,
    LOCAL / SPECIAL rows, the open middle block) plus, per sealed block, its
    codes (128 x k for K, 128 x d for V) and fp32 scales (k for K, 128 for
    V)."""
    bf16 = _resident_bytes_bf16(policy, n_kept, N, S, W, W_loc, n_special, head_dim)
    nb = sealed_blocks(n_kept, N, S, W) if policy == 0 and 0 < n_kept else 0
    if nb == 0:
        return bf16
    mid_row_bf16 = (n_kept + head_dim) * 2
    block = BLOCK_ROWS * (n_kept + head_dim) + 4 * (n_kept + BLOCK_ROWS)
    return bf16 - nb * BLOCK_ROWS * mid_row_bf16 + nb * block
