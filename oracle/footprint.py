"""KV-cache byte counts.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* Dense cache: LeanK article (framerc.cn) §1 gives 2 x L x h x d x N elements
  for L layers, h heads of dimension d and N tokens (the 2 is K and V).  The
  FastGen article (mhpn.cn) §2.2 works it per token: (d_k + d_v) x 2 bytes
  per head, times heads, times layers, times the sequence.
* Pruned cache (what one decode step reads per (b, kv head)): sinks and
  window at full width for K and V; middle tokens with k kept K channels plus
  the full V row; nothing in the middle for k = 0 (LeanK §3.1, §3.2); the last
  W_loc tokens for LOCAL heads and the special tokens for SPECIAL heads
  (FastGen §3.2).
"""
from __future__ import annotations

FULL, LOCAL, SPECIAL = 0, 1, 2


def dense_kv_elements(layers: int, heads: int, head_dim: int, tokens: int) -> int:
    return 2 * layers * heads * head_dim * tokens


def dense_kv_bytes(layers: int, heads: int, head_dim: int, tokens: int,
                   elem_bytes: int = 2, batch: int = 1) -> int:
    return dense_kv_elements(layers, heads, head_dim, tokens) * elem_bytes * batch


def resident_tokens(policy: int, n_kept: int, N: int, S: int, W: int, W_loc: int,
                    n_special: int = 0):
    """(full-width token count, kept-channel token count) resident for one head."""
    if policy == FULL:
        if n_kept == 128:
            return N, 0
        n_sl = min(N, S + W)
        n_mid = max(0, N - S - W)
        return (n_sl, n_mid) if n_kept > 0 else (n_sl, 0)
    if policy == LOCAL:
        return min(N, W_loc), 0
    if policy == SPECIAL:
        return n_special, 0
    raise ValueError(policy)


def resident_bytes(policy: int, n_kept: int, N: int, S: int, W: int, W_loc: int,
                   n_special: int = 0, head_dim: int = 128, elem_bytes: int = 2) -> int:
    """Bytes of K and V one decode step reads for one (b, kv head)."""
    n_full, n_mid = resident_tokens(policy, n_kept, N, S, W, W_loc, n_special)
    full_row = 2 * head_dim * elem_bytes                 # K row + V row
    mid_row = (n_kept + head_dim) * elem_bytes           # kept K channels + V row
    return n_full * full_row + n_mid * mid_row
