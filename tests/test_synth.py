"""Checks of the seeded input generator (host only)."""
import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import synth as S
from helpers import workload_masks


@pytest.mark.parametrize("w", S.WORKLOADS, ids=[w.name for w in S.WORKLOADS])
def test_workload_masks_are_aligned_and_deterministic(w):
    # the masks every test and the bench use: stage 2 on the drawn
    # importances (pruned workloads) or the drawn counts (the tiny case)
    pol = S.make_policies(w)
    m1 = workload_masks(w, pol)
    m2 = workload_masks(w, pol)
    assert m1.shape == (w.num_layers, w.num_kv_heads, w.head_dim)
    assert np.array_equal(m1, m2)
    counts = m1.sum(-1)
    assert np.all(counts % 32 == 0)
    assert set(np.unique(m1)) <= {0, 1}
    if w.prune_pct is not None:
        alpha, elig = S.stage2_inputs(w, pol)
        assert alpha.dtype == np.float32 and np.array_equal(elig, pol == S.POLICY_FULL)


def test_drawn_counts_of_the_tiny_case():
    w = S.WORKLOADS[0]
    c = S.drawn_counts(w)
    assert c.shape == (1, 2) and set(np.unique(c)) <= {0, 64}
    with pytest.raises(ValueError):
        S.drawn_counts(S.WORKLOADS[1])


def test_exact_budget_hits_the_aligned_target():
    for w in (S.WORKLOAD_BY_NAME["qwen25_7b_long"], S.WORKLOAD_BY_NAME["fastgen_mix"]):
        pol = S.make_policies(w)
        m = workload_masks(w, pol)
        full = pol == S.POLICY_FULL
        target = 32 * int(np.floor((1 - w.prune_pct / 100) * full.sum() * 128 / 32 + 0.5))
        assert m.sum(-1)[full].sum() == target


def test_round_down_never_exceeds_threshold_count():
    w = S.WORKLOAD_BY_NAME["serving_b64"]
    alpha, _ = S.stage2_inputs(w)
    thr = np.percentile(alpha.astype(np.float64).reshape(-1), w.prune_pct)
    above = (alpha >= thr).sum(-1)
    m = workload_masks(w)
    assert np.all(m.sum(-1) == (above // 32) * 32)
    # kept channels are the head's largest alphas
    for l, h in [(0, 0), (5, 3), (31, 7)]:
        k = int(m[l, h].sum())
        if k:
            kept = np.nonzero(m[l, h])[0]
            assert alpha[l, h, kept].min() >= np.sort(alpha[l, h])[::-1][k - 1]


def test_policy_counts_exact():
    w = S.WORKLOAD_BY_NAME["fastgen_mix"]
    pol = S.make_policies(w)
    assert (pol == S.POLICY_LOCAL).sum() == 102
    assert (pol == S.POLICY_SPECIAL).sum() == 51
    assert (pol == S.POLICY_FULL).sum() == 103


def test_special_table_and_ids():
    w = S.WORKLOAD_BY_NAME["fastgen_mix"].scaled(batch=2)
    t = S.make_special_table(w)
    assert t.shape == (32000,) and t.sum() == 1600
    ids = S.make_token_ids(w, 1000)
    assert ids.shape == (2, 1000) and ids.min() >= 0 and ids.max() < 32000
    frac = t[ids].mean()
    assert 0.02 < frac < 0.08


def test_kv_shapes_outliers_and_rope():
    w = S.WORKLOAD_BY_NAME["llama31_8b_layer"].scaled(context=64)
    k, v = S.make_kv(w, 0, 64)
    assert k.shape == (1, 64, 8, 128) and k.dtype == torch.bfloat16
    # 4 pairs (i, i+64) per head have ~8x larger magnitude
    mags = k.float().abs().mean(dim=(0, 1))          # [H, 128]
    big = (mags > 4).sum(dim=1)
    assert torch.all(big == 8)
    wr = S.WORKLOAD_BY_NAME["qwen25_7b_long"].scaled(context=32, batch=1)
    kr, _ = S.make_kv(wr, 0, 32)
    plain = S._normal(wr, 0, S.STREAM_K, (1, 32, 4, 128), None)
    # rotation preserves each pair's norm
    a = kr.float()[..., :64] ** 2 + kr.float()[..., 64:] ** 2
    b = plain[..., :64] ** 2 + plain[..., 64:] ** 2
    assert torch.allclose(a, b, rtol=2e-2, atol=2e-2)
    # position 0 is unrotated
    assert torch.allclose(kr.float()[:, 0], plain[:, 0].to(torch.bfloat16).float())


def test_mask_stats_report():
    w = S.WORKLOAD_BY_NAME["serving_b64"]
    pol = S.make_policies(w)
    st = S.mask_stats(w, workload_masks(w, pol), pol)
    assert 0.7 <= st["prune_ratio"] <= 0.85
    assert 0.05 <= st["zero_head_fraction"] <= 0.35
