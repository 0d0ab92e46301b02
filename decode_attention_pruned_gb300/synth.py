"""Seeded synthetic inputs for decode attention over a LeanK-pruned KV cache.

This module only draws inputs: workload shapes, channel importances (the
input of LeanK's mask construction) or drawn kept counts, per-head policies,
token ids, and the bf16 Q/K/V tensors.  It computes no mask threshold, no
attention, no cache layout and no byte count; the CUDA path and the fp64
oracle both consume what it returns and nothing else is shared between them.

Sources of the workload shapes (page titles as cited throughout the repo):
  * "LeanK pruning technique analysis" (framerc.cn), §1: Llama-3.1-8B serving
    at 4096 input tokens, batch 64; §2.2 stage 2: the static mask beta is built
    from a learned importance alpha by a global percentile threshold and a
    per-head channel count aligned to 32; §3.2: heads whose channels are all
    pruned drop their V; §6: 50-80 % prune rates.
  * "FastGen: profile-based adaptive KV compression" (mhpn.cn), §3.1-3.2:
    per-head local-window / special-token / full policies.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEAD_DIM = 128

POLICY_FULL = 0
POLICY_LOCAL = 1
POLICY_SPECIAL = 2

# independent random streams per (config, layer)
STREAM_MASK, STREAM_SPREAD, STREAM_Q, STREAM_K, STREAM_V, STREAM_IDS, STREAM_POLICY, STREAM_OUTLIER = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.  ``context`` is N, the resident token count at
    the decode step, counting the token appended just before it."""
    name: str
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    context: int
    sink: int
    local: int
    seed: int
    prune_pct: Optional[float] = None      # s: percent of K channels pruned
    budget: str = "round_down"             # "round_down" | "exact" | "choice64"
    tau: float = 0.0                       # per-head spread of log-alpha
    align: int = 32
    local_only_window: int = 0             # W_loc of LOCAL heads
    policy_counts: Optional[tuple] = None  # (#LOCAL, #SPECIAL, #FULL) over all (layer, kv head)
    vocab: int = 0
    num_special_ids: int = 0
    outlier_pairs: int = 0
    outlier_scale: float = 1.0
    rope_base: Optional[float] = None
    head_dim: int = HEAD_DIM

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads.  Index 0 is the tiny case; index 2, the 32-layer
# batch-64 serving step, is the largest one and the default of the throughput
# measurement.
WORKLOADS = [
    Workload("tiny", num_layers=1, batch=1, num_q_heads=4, num_kv_heads=2, context=512,
             sink=4, local=64, seed=1001, budget="choice64"),
    Workload("llama31_8b_layer", num_layers=1, batch=1, num_q_heads=32, num_kv_heads=8,
             context=32768, sink=16, local=1024, seed=1002, prune_pct=70.0,
             budget="round_down", tau=0.12, outlier_pairs=4, outlier_scale=8.0),
    Workload("serving_b64", num_layers=32, batch=64, num_q_heads=32, num_kv_heads=8,
             context=4096, sink=16, local=512, seed=1003, prune_pct=70.0,
             budget="round_down", tau=0.12),
    Workload("qwen25_7b_long", num_layers=1, batch=4, num_q_heads=28, num_kv_heads=4,
             context=131072, sink=16, local=2048, seed=1004, prune_pct=80.0,
             budget="exact", tau=0.0, rope_base=1.0e6),
    Workload("fastgen_mix", num_layers=32, batch=16, num_q_heads=32, num_kv_heads=8,
             context=16384, sink=16, local=512, seed=1005, prune_pct=60.0,
             budget="exact", tau=0.0, local_only_window=256,
             policy_counts=(102, 51, 103), vocab=32000, num_special_ids=1600),
]

WORKLOAD_BY_NAME = {w.name: w for w in WORKLOADS}


def rng(seed: int, layer: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, stream])))


# --------------------------------------------------------------------------
# masks and policies
# --------------------------------------------------------------------------

def draw_alpha(w: Workload) -> np.ndarray:
    """Channel importance alpha[l,h,c] = exp(z + tau*u): z per channel and u
    per head are independent N(0,1).  tau=0 gives i.i.d. LogNormal(0,1)."""
    z = rng(w.seed, 0, STREAM_MASK).standard_normal((w.num_layers, w.num_kv_heads, w.head_dim))
    u = rng(w.seed, 0, STREAM_SPREAD).standard_normal((w.num_layers, w.num_kv_heads, 1))
    return np.exp(z + w.tau * u)


def make_policies(w: Workload) -> np.ndarray:
    """Per (layer, kv head) policy ids; exact counts by a seeded permutation."""
    L, H = w.num_layers, w.num_kv_heads
    if w.policy_counts is None:
        return np.full((L, H), POLICY_FULL, dtype=np.int32)
    n_loc, n_spec, n_full = w.policy_counts
    assert n_loc + n_spec + n_full == L * H
    flat = np.array([POLICY_LOCAL] * n_loc + [POLICY_SPECIAL] * n_spec + [POLICY_FULL] * n_full,
                    dtype=np.int32)
    perm = rng(w.seed, 0, STREAM_POLICY).permutation(L * H)
    return flat[perm].reshape(L, H)


def stage2_inputs(w: Workload, policies: Optional[np.ndarray] = None):
    """What LeanK's stage 2 builds a pruned workload's mask from: the
    importances alpha [L, Hkv, 128] (float32) and the heads that take a mask
    (FULL policy), bool [L, Hkv].  With ``w.prune_pct``, ``w.align`` and
    ``w.budget`` these fully determine the mask; this module does not build
    it (the library's mask builder does, and so does the oracle)."""
    if policies is None:
        policies = make_policies(w)
    return draw_alpha(w).astype(np.float32), np.asarray(policies) == POLICY_FULL


def drawn_counts(w: Workload) -> np.ndarray:
    """Kept-channel counts [L, Hkv] of a workload whose counts are drawn
    rather than derived from a prune ratio: the tiny case draws 0 or 64 per
    head (seeded); a workload without a prune ratio keeps all 128."""
    if w.budget == "choice64":
        r = rng(w.seed, 0, STREAM_POLICY + 100)
        return r.choice([0, 64], size=(w.num_layers, w.num_kv_heads))
    if w.prune_pct is None:
        return np.full((w.num_layers, w.num_kv_heads), w.head_dim)
    raise ValueError(f"{w.name}: counts follow from the prune ratio (stage 2), not from a draw")


def masks_with_counts(w: Workload, counts) -> np.ndarray:
    """Masks whose per-head kept counts are given explicitly (top-k of alpha)."""
    alpha = draw_alpha(w)
    counts = np.asarray(counts).reshape(w.num_layers, w.num_kv_heads)
    mask = np.zeros(alpha.shape, dtype=np.uint8)
    for l in range(w.num_layers):
        for h in range(w.num_kv_heads):
            order = np.argsort(-alpha[l, h], kind="stable")
            mask[l, h, order[: int(counts[l, h])]] = 1
    return mask


def make_special_table(w: Workload) -> np.ndarray:
    """uint8 [vocab] flags of the special-token id set (empty if no vocab)."""
    if w.vocab == 0:
        return np.zeros(0, dtype=np.uint8)
    table = np.zeros(w.vocab, dtype=np.uint8)
    ids = rng(w.seed, 0, STREAM_IDS + 100).choice(w.vocab, size=w.num_special_ids, replace=False)
    table[ids] = 1
    return table


def make_token_ids(w: Workload, n_tokens: int) -> np.ndarray:
    """int32 [B, n_tokens] token ids of positions 0 .. n_tokens-1 (one draw
    for the whole history; callers slice it for prefill and appends)."""
    if w.vocab == 0:
        return np.zeros((w.batch, n_tokens), dtype=np.int32)
    return rng(w.seed, 0, STREAM_IDS).integers(0, w.vocab, size=(w.batch, n_tokens),
                                               dtype=np.int64).astype(np.int32)


# --------------------------------------------------------------------------
# Q / K / V
# --------------------------------------------------------------------------

def _rope_rotate(x, positions, base: float):
    """Rotate-half RoPE on the last dim (pairs (i, i+64)), angle p*base^(-2i/d).
    x: float64 torch tensor [..., n, H, d]; positions: [n]."""
    import torch
    d = x.shape[-1]
    half = d // 2
    i = torch.arange(half, dtype=torch.float64, device=x.device)
    inv_freq = base ** (-2.0 * i / d)
    ang = positions.to(torch.float64)[:, None] * inv_freq[None, :]          # [n, half]
    cos = torch.cos(ang)[:, None, :]
    sin = torch.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def _normal(w: Workload, layer: int, stream: int, shape, device):
    """float32 standard normals: numpy PCG64 on the host, torch Philox on a device."""
    import torch
    if device is None or str(device) == "cpu":
        a = rng(w.seed, layer, stream).standard_normal(shape, dtype=np.float32)
        return torch.from_numpy(a)
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence([w.seed, layer, stream]).generate_state(1)[0]))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def make_kv(w: Workload, layer: int, n_tokens: int, device=None):
    """bf16 K, V [B, n_tokens, Hkv, 128]: the dense history of one layer,
    positions 0 .. n_tokens-1 (one draw; callers slice it for prefill and
    appends).  Workload structure: ``outlier_pairs`` channel pairs (i, i+64)
    of K scaled by ``outlier_scale``; RoPE on K at each token's position."""
    import torch
    B, H, D = w.batch, w.num_kv_heads, w.head_dim
    total = n_tokens
    k = _normal(w, layer, STREAM_K, (B, total, H, D), device)
    v = _normal(w, layer, STREAM_V, (B, total, H, D), device)
    if w.outlier_pairs:
        r = rng(w.seed, layer, STREAM_OUTLIER)
        scale = torch.ones(H, D, dtype=torch.float32)
        for h in range(H):
            pairs = r.choice(D // 2, size=w.outlier_pairs, replace=False)
            for i in pairs:
                scale[h, i] = w.outlier_scale
                scale[h, i + D // 2] = w.outlier_scale
        k = k * scale.to(k.device)
    if w.rope_base is not None:
        pos = torch.arange(0, total, device=k.device)
        k = _rope_rotate(k.to(torch.float64), pos, w.rope_base)
    return k.to(torch.bfloat16).contiguous(), v.to(torch.bfloat16).contiguous()


def make_q(w: Workload, layer: int, position: int, device=None, step: int = 0):
    """bf16 q [B, Hq, 128] for the decode step at ``position`` (RoPE'd for
    rope workloads).  ``step`` selects an independent draw."""
    import torch
    q = _normal(w, layer, STREAM_Q + 16 * step, (w.batch, w.num_q_heads, w.head_dim), device)
    if w.rope_base is not None:
        pos = torch.tensor([position], device=q.device)
        q = _rope_rotate(q.to(torch.float64)[:, None], pos, w.rope_base)[:, 0]
    return q.to(torch.bfloat16).contiguous()


def mask_stats(w: Workload, masks: np.ndarray, policies: np.ndarray) -> dict:
    """Realised prune ratio and zero-head fraction over the FULL heads."""
    full = policies == POLICY_FULL
    counts = masks.sum(-1)[full]
    if counts.size == 0:
        return {"full_heads": 0}
    return {
        "full_heads": int(counts.size),
        "prune_ratio": float(1.0 - counts.sum() / (counts.size * w.head_dim)),
        "zero_head_fraction": float((counts == 0).mean()),
        "kept_hist": {int(k): int((counts == k).sum()) for k in range(0, w.head_dim + 1, 32)},
    }
