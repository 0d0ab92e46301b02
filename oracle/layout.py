"""Which token each compressed-cache row holds after N tokens, per (b, kv head).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The rules restate the pages' cache editing:

* LeanK article (framerc.cn) §3.1 "cache partition": a full-width K cache for
  the attention sinks plus the local window, and K_prun for the middle tokens
  holding only the kept channels.  §2.2 stage 1: sinks and window are never
  channel-pruned.  §3.2: a head with no kept channel keeps no middle K or V.
* StreamingLLM reading of the window ("intelligent pruning white paper",
  yyx235 blog, §3.3.1): the first S tokens are kept for good, the last W
  tokens slide; when a token leaves the window it moves to the middle.
* FastGen article (mhpn.cn) §3.2 stage 2: a LOCAL head keeps the last W_loc
  tokens; a SPECIAL head appends a token only when its id is special, in
  arrival order.

Row numbering (a reading: the pages fix contents, not addresses):
  region A (full width): sink token t < S at row t; window token t >= S at
  ring row S + (t - S) mod W.  LOCAL heads: ring row t mod W_loc.  SPECIAL
  heads: row r for the r-th special token.
  region B (FULL heads with k > 0): middle token t at row t - S; its K row is
  K[t] restricted to the kept channels in ascending channel order; V row V[t].
"""
from __future__ import annotations

import numpy as np

FULL, LOCAL, SPECIAL = 0, 1, 2


def region_a(policy: int, N: int, S: int, W: int, W_loc: int, special_flags=None,
             special_capacity: int | None = None):
    """(rows, tokens) of the full-width region after N tokens."""
    if policy == FULL:
        sink = np.arange(min(S, N))
        window = np.arange(max(S, N - W), N)
        rows = np.concatenate([sink, S + (window - S) % W]) if W > 0 else sink
        toks = np.concatenate([sink, window]) if W > 0 else sink
        return rows.astype(np.int64), toks.astype(np.int64)
    if policy == LOCAL:
        toks = np.arange(max(0, N - W_loc), N)
        return (toks % W_loc).astype(np.int64), toks.astype(np.int64)
    if policy == SPECIAL:
        toks = np.nonzero(np.asarray(special_flags[:N], dtype=bool))[0]
        if special_capacity is not None:
            toks = toks[:special_capacity]
        return np.arange(len(toks), dtype=np.int64), toks.astype(np.int64)
    raise ValueError(policy)


def region_b(policy: int, n_kept: int, N: int, S: int, W: int):
    """(rows, tokens) of the kept-channel middle region after N tokens."""
    if policy != FULL or n_kept == 0:
        return np.arange(0, dtype=np.int64), np.arange(0, dtype=np.int64)
    toks = np.arange(S, max(S, N - W))
    return (toks - S).astype(np.int64), toks.astype(np.int64)
