"""The static channel mask beta of LeanK's stage 2, from importances alpha.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

LeanK article (framerc.cn) §2.2 stage 2 ("hardware-friendly mask"): a global
threshold keeps the most important channels over all (layer, head) pairs,
each head's kept count is brought to a multiple of the alignment, and each
head keeps its most important channels.  Readings (the printed routine is
garbled; these are the plainest readings the rest of the section supports):

* ``prune_pct`` = s is the share of channels pruned: the threshold is the
  s-th percentile of the eligible alphas, and a channel stays when
  alpha >= threshold.
* The percentile interpolates linearly between order statistics (the numpy
  default): with the n values sorted ascending, position p = s/100 * (n-1),
  i = floor(p), threshold = x_i + frac(p) * (x_{i+1} - x_i).  That formula is
  evaluated in fp32 with no fused multiply-add, the precision the device
  builder compares in, because the threshold decides integer counts.
* ``round_down``: count -> align * floor(count / align) (the printed routine).
  ``exact``: after rounding down, +align on the heads with the largest
  remainders (ties: lower flat head index), repeated until the total equals
  align * floor((1 - s/100) * heads * 128 / align + 1/2); a head never
  exceeds 128.
* A head keeps its n channels of largest alpha; equal alphas go to the lower
  channel index.  Ineligible heads (not FULL policy) get all channels.
"""
from __future__ import annotations

import math

import numpy as np


def percentile_fp32(values, pct: float) -> np.float32:
    v = np.sort(np.asarray(values, dtype=np.float32).ravel())
    n = len(v)
    pos = pct / 100.0 * (n - 1)
    i = int(math.floor(pos))
    j = min(i + 1, n - 1)
    frac = np.float32(pos - i)
    d = np.float32(v[j] - v[i])
    t = np.float32(frac * d)
    return np.float32(v[i] + t)


def aligned_counts(alpha, prune_pct: float, align: int, budget: str, eligible=None):
    """Per-head kept channel counts [L, H] (ineligible heads: 128)."""
    a = np.asarray(alpha, dtype=np.float32)
    L, H, D = a.shape
    elig = np.ones((L, H), dtype=bool) if eligible is None else np.asarray(eligible, dtype=bool)
    if not elig.any():                      # nothing to prune: every head keeps all channels
        return np.full((L, H), D, dtype=np.int64)
    thr = percentile_fp32(a[elig], prune_pct)
    above = (a >= thr).sum(axis=-1)
    keep = (above // align) * align
    if budget == "exact":
        n_heads = int(elig.sum())
        target = align * int(math.floor((1.0 - prune_pct / 100.0) * n_heads * D / align + 0.5))
        deficit = target - int(keep[elig].sum())
        rem = (above - keep).reshape(-1)
        order = sorted(range(L * H), key=lambda i: (-rem[i], i))
        flat = keep.reshape(-1)
        el = elig.reshape(-1)
        while deficit > 0:
            given = False
            for i in order:
                if deficit <= 0:
                    break
                if el[i] and flat[i] + align <= D:
                    flat[i] += align
                    deficit -= align
                    given = True
            if not given:
                break
        keep = flat.reshape(L, H)
    elif budget != "round_down":
        raise ValueError(budget)
    return np.where(elig, keep, D)


def top_s_prune(alpha, prune_pct: float, align: int = 32, budget: str = "round_down", eligible=None):
    """uint8 mask beta [L, H, 128]."""
    a = np.asarray(alpha, dtype=np.float32)
    L, H, D = a.shape
    keep = aligned_counts(a, prune_pct, align, budget, eligible)
    mask = np.zeros((L, H, D), dtype=np.uint8)
    for l in range(L):
        for h in range(H):
            order = np.argsort(-a[l, h], kind="stable")     # largest first, ties by index
            mask[l, h, order[: int(keep[l, h])]] = 1
    return mask
