"""Decode attention over a LeanK / FastGen compressed KV cache, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What one decode step computes, per batch element b and query head j:

* GQA: query head j reads KV head h = j // G, G = Hq / Hkv (query heads map
  contiguously onto KV heads; the pages only say a group shares one K/V --
  "intelligent pruning white paper" (yyx235 blog) §5.2.3).
* Append first, then attend: the current token is already in the cache, so
  the context has N tokens including it -- FastGen article (mhpn.cn) §2.1.
* FULL heads, LeanK article (framerc.cn) §2.2 and §3.1: the attention-sink
  tokens [0, S) and the local window [N-W, N) are scored with all 128
  channels; the middle tokens [S, N-W) are scored with only the head's kept
  channels beta (K_prun holds only those).  §3.2: a head with no kept channel
  drops its middle K and V, so its middle tokens leave the softmax entirely.
  A head that keeps all 128 channels is plain dense attention.
* LOCAL heads, FastGen §3.2 stage 2: only the last W_loc tokens.
* SPECIAL heads, FastGen §3.2 stage 2: only tokens whose id is in the special
  set; an empty set gives o = 0.
* Scores are q.k / sqrt(d) with d = 128 on every region (pruning zeroes
  channels, it does not change d), then one softmax over all included tokens
  and o = sum_t softmax(s)_t V[t].
"""
from __future__ import annotations

import math

import numpy as np

FULL, LOCAL, SPECIAL = 0, 1, 2


def score_scale(head_dim: int) -> float:
    """1/sqrt(d): the scaled-dot-product factor, the same on every region."""
    return 1.0 / math.sqrt(head_dim)


def full_width_tokens(policy: int, n_kept: int, N: int, S: int, W: int, W_loc: int,
                      special_flags=None) -> np.ndarray:
    """Token positions scored with all channels, ascending."""
    if policy == FULL:
        if n_kept == 128:
            return np.arange(N)
        sink = np.arange(min(S, N))
        window = np.arange(max(S, N - W), N)
        return np.concatenate([sink, window])
    if policy == LOCAL:
        return np.arange(max(0, N - W_loc), N)
    if policy == SPECIAL:
        flags = np.asarray(special_flags[:N], dtype=bool)
        return np.nonzero(flags)[0]
    raise ValueError(policy)


def kept_channel_tokens(policy: int, n_kept: int, N: int, S: int, W: int) -> np.ndarray:
    """Middle token positions scored with the kept channels only (FULL heads
    with 0 < k < 128); empty otherwise."""
    if policy != FULL or n_kept in (0, 128):
        return np.arange(0)
    return np.arange(S, max(S, N - W))


def decode_head(q: np.ndarray, K: np.ndarray, V: np.ndarray, policy: int,
                kept: np.ndarray, N: int, S: int, W: int, W_loc: int,
                special_flags=None) -> np.ndarray:
    """Outputs of the G query heads that share one KV head.

    q: [G, d] query rows; K, V: [>=N, d] dense history of the KV head (rows are
    token positions); kept: ascending kept channel indices (the mask beta).
    Returns o: [G, d] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K[:N], dtype=np.float64)
    V = np.asarray(V[:N], dtype=np.float64)
    G, d = q.shape
    kept = np.asarray(kept, dtype=np.int64)
    t_full = full_width_tokens(policy, len(kept), N, S, W, W_loc, special_flags)
    t_mid = kept_channel_tokens(policy, len(kept), N, S, W)
    scale = score_scale(d)
    s_full = (K[t_full] @ q.T) * scale                                # [n_full, G]
    s_mid = (K[t_mid][:, kept] @ q[:, kept].T) * scale                # [n_mid, G]
    s = np.concatenate([s_full, s_mid], axis=0)
    vrows = V[np.concatenate([t_full, t_mid])]
    if s.shape[0] == 0:
        return np.zeros((G, d))
    m = s.max(axis=0, keepdims=True)
    p = np.exp(s - m)
    return (p.T @ vrows) / p.sum(axis=0)[:, None]


def decode_layer(q, K, V, masks, policies, N: int, S: int, W: int, W_loc: int,
                 special_flags=None, heads=None) -> np.ndarray:
    """Decode attention for one layer.

    q [B, Hq, d]; K, V [B, >=N, Hkv, d]; masks [Hkv, d] 0/1; policies [Hkv];
    special_flags [B, >=N] (bool, token id in the special set) or None.
    ``heads``: optional iterable of (b, h) pairs to compute (others stay 0).
    Returns o [B, Hq, d] float64.
    """
    q = np.asarray(q)
    B, Hq, d = q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    for b, h in pairs:
        kept = np.nonzero(np.asarray(masks[h]))[0]
        flags = None if special_flags is None else special_flags[b]
        out[b, h * G:(h + 1) * G] = decode_head(
            q[b, h * G:(h + 1) * G], K[b, :, h], V[b, :, h], int(policies[h]), kept,
            N, S, W, W_loc, flags)
    return out
