"""Pins for the fp64 oracle: each check compares it with something other than
itself -- a library attention routine, brute force with explicit channel
masks, closed forms, or numbers the pages print (``tests/golden/``).

The mutation test at the end plants plausible mistakes in the oracle (on the
CPU) and requires at least one pin to catch each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import footprint as F
from oracle import layout as LY

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FULL, LOCAL, SPECIAL = 0, 1, 2
D = 128


def _bf16_values(shape, seed, scale=1.0):
    """fp64 arrays holding exact bf16 values (what the cache stores)."""
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)
    return x.to(torch.float64).numpy()


def _sdpa(q, K, V):
    """torch fp64 scaled_dot_product_attention of one query over rows K, V.
    q [G, d]; K, V [n, d] -> [G, d]."""
    qt = torch.from_numpy(np.ascontiguousarray(q))[None, :, None, :]       # [1, G, 1, d]
    G = q.shape[0]
    Kt = torch.from_numpy(np.ascontiguousarray(K))[None, None].expand(1, G, -1, -1)
    Vt = torch.from_numpy(np.ascontiguousarray(V))[None, None].expand(1, G, -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)[0, :, 0, :].numpy()


def _brute_force_head(q, K, V, policy, beta, N, S, W, W_loc, flags=None):
    """Pure-Python loops: an explicit per-(token, channel) weight w[t][c]
    (1 at full width, beta[c] for a middle token, token excluded when the
    head keeps no channel), an inclusion flag per token, then softmax."""
    G = q.shape[0]
    k = int(sum(beta))
    out = np.zeros((G, D))
    for g in range(G):
        scores, rows = [], []
        for t in range(N):
            if policy == FULL:
                in_sink, in_win = t < S, t >= N - W
                if k == 0 and not (in_sink or in_win):
                    continue
                w = [1.0] * D if (in_sink or in_win) else [float(b) for b in beta]
            elif policy == LOCAL:
                if t < N - W_loc:
                    continue
                w = [1.0] * D
            else:
                if not flags[t]:
                    continue
                w = [1.0] * D
            s = 0.0
            for c in range(D):
                s += w[c] * q[g][c] * K[t][c]
            scores.append(s / math.sqrt(D))
            rows.append(t)
        if not rows:
            continue
        mx = max(scores)
        ex = [math.exp(s - mx) for s in scores]
        tot = sum(ex)
        for e, t in zip(ex, rows):
            for c in range(D):
                out[g][c] += e / tot * V[t][c]
    return out


# ---------------------------------------------------------------------------
# pin checks (plain functions so the mutation test can run them all)
# ---------------------------------------------------------------------------

def check_dense_equals_sdpa():
    """k = 128 FULL heads are plain softmax attention (library routine)."""
    for N, G, seed in [(1, 2, 1), (37, 4, 2), (300, 7, 3)]:
        q = _bf16_values((G, D), seed)
        K = _bf16_values((N, D), seed + 10)
        V = _bf16_values((N, D), seed + 20)
        got = A.decode_head(q, K, V, FULL, np.arange(D), N, S=4, W=16, W_loc=0)
        ref = _sdpa(q, K, V)
        assert np.max(np.abs(got - ref)) < 1e-12


def check_zero_head_equals_sink_local_sdpa():
    """A head with no kept channel attends to sinks + window only (LeanK §3.2)."""
    S, W = 4, 16
    for N in [1, 3, S, S + 1, S + W - 1, S + W, S + W + 1, 97]:
        q = _bf16_values((2, D), N)
        K = _bf16_values((N, D), N + 1)
        V = _bf16_values((N, D), N + 2)
        idx = sorted(set(range(min(S, N))) | set(range(max(S, N - W), N)))
        got = A.decode_head(q, K, V, FULL, np.arange(0), N, S, W, 0)
        ref = _sdpa(q, K[idx], V[idx])
        assert np.max(np.abs(got - ref)) < 1e-12


def check_local_equals_sdpa():
    """LOCAL heads read the last W_loc tokens (FastGen §3.2)."""
    for N, W_loc in [(5, 8), (8, 8), (9, 8), (100, 32)]:
        q = _bf16_values((4, D), N)
        K = _bf16_values((N, D), N + 3)
        V = _bf16_values((N, D), N + 4)
        got = A.decode_head(q, K, V, LOCAL, np.arange(0), N, 4, 16, W_loc)
        lo = max(0, N - W_loc)
        assert np.max(np.abs(got - _sdpa(q, K[lo:], V[lo:]))) < 1e-12


def check_special_equals_sdpa():
    """SPECIAL heads read only special tokens; none gives o = 0 (FastGen §3.2)."""
    rs = np.random.default_rng(5)
    N = 60
    q = _bf16_values((4, D), 7)
    K = _bf16_values((N, D), 8)
    V = _bf16_values((N, D), 9)
    flags = rs.random(N) < 0.2
    idx = np.nonzero(flags)[0]
    got = A.decode_head(q, K, V, SPECIAL, np.arange(0), N, 4, 16, 0, flags)
    assert np.max(np.abs(got - _sdpa(q, K[idx], V[idx]))) < 1e-12
    none = A.decode_head(q, K, V, SPECIAL, np.arange(0), N, 4, 16, 0, np.zeros(N, bool))
    assert np.all(none == 0.0)


def check_pruned_equals_brute_force():
    """0 < k < 128: brute force with explicit beta-weighted channels."""
    S, W = 4, 8
    rs = np.random.default_rng(11)
    for N in [3, S, S + W, S + W + 1, 29]:
        for k in [32, 64, 96]:
            beta = np.zeros(D, dtype=np.uint8)
            beta[rs.choice(D, size=k, replace=False)] = 1
            q = _bf16_values((2, D), 100 + N + k)
            K = _bf16_values((N, D), 200 + N + k, scale=2.0)
            V = _bf16_values((N, D), 300 + N + k)
            got = A.decode_head(q, K, V, FULL, np.nonzero(beta)[0], N, S, W, 0)
            ref = _brute_force_head(q, K, V, FULL, beta, N, S, W, 0)
            assert np.max(np.abs(got - ref)) < 1e-12, (N, k)
    for policy in (LOCAL, SPECIAL):
        N = 23
        flags = rs.random(N) < 0.3
        q = _bf16_values((2, D), 41)
        K = _bf16_values((N, D), 42)
        V = _bf16_values((N, D), 43)
        got = A.decode_head(q, K, V, policy, np.arange(0), N, S, W, 6, flags)
        ref = _brute_force_head(q, K, V, policy, np.zeros(D), N, S, W, 6, flags)
        assert np.max(np.abs(got - ref)) < 1e-12


def check_uniform_scores_give_region_means():
    """q = 0 makes every score equal, so o is the mean V over exactly the
    included tokens: pins each region boundary (closed form)."""
    S, W, W_loc = 4, 8, 5
    for N in [1, 3, 4, 5, 11, 12, 13, 40]:
        V = _bf16_values((N, D), 500 + N)
        K = _bf16_values((N, D), 600 + N)
        q = np.zeros((2, D))
        cases = {
            (FULL, 128): list(range(N)),
            (FULL, 32): list(range(N)),
            (FULL, 0): sorted(set(range(min(S, N))) | set(range(max(S, N - W), N))),
            (LOCAL, 0): list(range(max(0, N - W_loc), N)),
        }
        for (pol, k), idx in cases.items():
            got = A.decode_head(q, K, V, pol, np.arange(k), N, S, W, W_loc)
            assert np.max(np.abs(got - V[idx].mean(axis=0))) < 1e-12, (pol, k, N)


def check_two_token_closed_form():
    """Two included tokens: o = (e^s1 v1 + e^s2 v2) / (e^s1 + e^s2), with
    s = q.k / sqrt(128); one scored at full width, one through a kept channel."""
    S, W, N = 1, 1, 3          # token 0 sink, token 1 middle, token 2 window
    q = np.zeros((1, D)); q[0, 5] = 2.0; q[0, 9] = 3.0
    K = np.zeros((N, D)); K[0, 5] = 1.5; K[1, 5] = 4.0; K[1, 9] = 1.0; K[2, 9] = -1.0
    V = np.zeros((N, D)); V[0, 0] = 1.0; V[1, 1] = 1.0; V[2, 2] = 1.0
    kept = np.array([9])       # channel 5 pruned in the middle
    got = A.decode_head(q, K, V, FULL, kept, N, S, W, 0)
    r = 1.0 / math.sqrt(128.0)
    s = np.array([2.0 * 1.5, 3.0 * 1.0, 3.0 * -1.0]) * r   # middle token loses 2*4
    e = np.exp(s - s.max())
    want = e / e.sum()
    assert np.max(np.abs(got[0, :3] - want)) < 1e-15
    assert np.all(got[0, 3:] == 0.0)


def check_single_token_returns_its_v():
    V = _bf16_values((1, D), 77)
    K = _bf16_values((1, D), 78)
    q = _bf16_values((3, D), 79)
    for pol, k in [(FULL, 0), (FULL, 64), (LOCAL, 0)]:
        got = A.decode_head(q, K, V, pol, np.arange(k), 1, 4, 8, 4)
        assert np.max(np.abs(got - V[0])) < 1e-15


def check_decode_layer_gqa_mapping():
    """Query head j uses KV head j // G (contiguous groups)."""
    B, Hkv, G, N = 2, 3, 2, 9
    q = _bf16_values((B, Hkv * G, D), 1)
    K = _bf16_values((B, N, Hkv, D), 2)
    V = _bf16_values((B, N, Hkv, D), 3)
    masks = np.ones((Hkv, D), dtype=np.uint8)
    out = A.decode_layer(q, K, V, masks, [FULL] * Hkv, N, 2, 4, 0)
    for b in range(B):
        for j in range(Hkv * G):
            ref = _sdpa(q[b, j:j + 1], K[b, :, j // G], V[b, :, j // G])
            assert np.max(np.abs(out[b, j] - ref[0])) < 1e-12


def _simulate_appends(policy, n_kept, N, S, W, W_loc, flags, cap=None):
    """Independent formulation of the cache editing: push tokens one by one
    into explicit Python containers, evicting from the window as it fills."""
    a = {}                     # row -> token, full-width region
    b = {}                     # row -> token, kept-channel region
    window = []                # tokens currently in the window, oldest first
    spec = []
    for t in range(N):
        if policy == FULL:
            if t < S:
                a[t] = t
                continue
            if len(window) == W:
                old = window.pop(0)
                if n_kept > 0:
                    b[old - S] = old
                del a[[r for r, tok in a.items() if tok == old][0]]
            used = {r for r, tok in a.items() if tok >= S}
            free = [S + (t - S) % W]
            assert free[0] not in used
            a[free[0]] = t
            window.append(t)
        elif policy == LOCAL:
            for r in [r for r, tok in a.items() if tok <= t - W_loc]:
                del a[r]
            a[t % W_loc] = t
        else:
            if flags[t] and (cap is None or len(spec) < cap):
                a[len(spec)] = t
                spec.append(t)
    return a, b


def check_layout_matches_simulation():
    S, W, W_loc = 3, 5, 4
    rs = np.random.default_rng(3)
    flags = rs.random(40) < 0.4
    for N in range(0, 40):
        for pol, k in [(FULL, 32), (FULL, 0), (FULL, 128), (LOCAL, 0), (SPECIAL, 0)]:
            a, b = _simulate_appends(pol, k, N, S, W, W_loc, flags, cap=7)
            ra, ta = LY.region_a(pol, N, S, W, W_loc, flags, special_capacity=7)
            rb, tb = LY.region_b(pol, k, N, S, W)
            assert dict(zip(ra.tolist(), ta.tolist())) == a, (pol, k, N)
            assert dict(zip(rb.tolist(), tb.tolist())) == b, (pol, k, N)


def check_footprint_fastgen_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_footprint_fastgen_s2_2.json")))
    i, p = g["inputs"], g["printed"]
    assert F.dense_kv_bytes(1, 1, i["head_dim"], 1, i["elem_bytes"]) == p["bytes_per_token_per_head_per_layer"]
    assert F.dense_kv_bytes(1, i["heads"], i["head_dim"], 1, i["elem_bytes"]) == p["bytes_per_token_per_layer_all_heads"]
    assert F.dense_kv_bytes(i["layers"], i["heads"], i["head_dim"], 1, i["elem_bytes"]) == p["bytes_per_token_all_layers"]
    total = F.dense_kv_bytes(i["layers"], i["heads"], i["head_dim"], i["tokens"], i["elem_bytes"])
    assert total == p["kilobytes_whole_sequence"] * 1024 == 2 ** 30


def check_footprint_leank_llama_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_footprint_leank_s1.json")))
    i, a = g["inputs"], g["architecture_not_printed_on_page"]
    n = i["input_tokens"] + i["output_tokens"]
    total = F.dense_kv_bytes(a["layers"], a["kv_heads"], a["head_dim"], n, i["elem_bytes"], i["batch"])
    assert total == 40 * 2 ** 30
    assert abs(total / 1e9 - g["printed"]["approx_gigabytes"]) / g["printed"]["approx_gigabytes"] < 0.08


def check_footprint_pruned_rules():
    # k = 128 reads the dense per-head bytes
    for N in [1, 50, 5000]:
        assert F.resident_bytes(FULL, 128, N, 16, 512, 0) == F.dense_kv_bytes(1, 1, D, N)
    # sliding window of 512 at 2048 keeps 25 % (FastGen §4.1 table)
    g = json.load(open(os.path.join(GOLDEN, "window_fraction_fastgen_s4_1.json")))
    frac = F.resident_bytes(LOCAL, 0, g["inputs"]["sequence"], 0, 0, g["inputs"]["window"]) / \
        F.dense_kv_bytes(1, 1, D, g["inputs"]["sequence"])
    assert round(100 * frac) == g["printed"]["fraction_percent_approx"]
    # V memory falls by about the zero-head fraction (LeanK §3.2) at long context
    g = json.load(open(os.path.join(GOLDEN, "v_drop_leank_s3_2.json")))
    lo, hi = g["printed"]["v_reduction_range"]
    N, S, W, H = 32768, 16, 1024, 100
    for f in (g["printed"]["zero_head_fraction_qwen"], g["printed"]["zero_head_fraction_llama"]):
        n0 = int(round(f * H))
        v_dense = H * N * D * 2
        v_kept = (H - n0) * N * D * 2 + n0 * (S + W) * D * 2
        red = 1 - v_kept / v_dense
        assert lo - 0.01 <= red <= hi + 0.005
    # explicit per-token costs
    assert F.resident_bytes(FULL, 32, 100, 4, 16, 0) == 20 * 512 + 80 * (32 + 128) * 2
    assert F.resident_bytes(FULL, 0, 100, 4, 16, 0) == 20 * 512
    assert F.resident_bytes(SPECIAL, 0, 100, 4, 16, 0, n_special=7) == 7 * 512


PINS = [
    check_dense_equals_sdpa, check_zero_head_equals_sink_local_sdpa, check_local_equals_sdpa,
    check_special_equals_sdpa, check_pruned_equals_brute_force,
    check_uniform_scores_give_region_means, check_two_token_closed_form,
    check_single_token_returns_its_v, check_decode_layer_gqa_mapping,
    check_layout_matches_simulation, check_footprint_fastgen_worked_example,
    check_footprint_leank_llama_example, check_footprint_pruned_rules,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

def _mut_scale_sqrt_k(mp):
    # middle region scaled by 1/sqrt(k) instead of 1/sqrt(d)
    orig = A.decode_head

    def wrong(q, K, V, policy, kept, N, S, W, W_loc, special_flags=None):
        o = orig(q, K, V, policy, kept, N, S, W, W_loc, special_flags)
        if policy == FULL and 0 < len(kept) < 128 and N > S + W:
            K2 = np.array(K[:N], dtype=np.float64)
            K2[S:N - W] *= math.sqrt(128 / len(kept))
            return orig(q, K2, V, policy, kept, N, S, W, W_loc, special_flags)
        return o
    mp.setattr(A, "decode_head", wrong)


MUTATIONS = {
    "no_scale": lambda mp: mp.setattr(A, "score_scale", lambda d: 1.0),
    "scale_sqrt_k": _mut_scale_sqrt_k,
    "window_off_by_one": lambda mp: mp.setattr(
        A, "full_width_tokens",
        (lambda f: (lambda p, k, N, S, W, Wl, fl=None:
                    f(p, k, N, S, W - 1 if p == FULL else W, Wl, fl)))(A.full_width_tokens)),
    "middle_all_channels": lambda mp: mp.setattr(
        A, "kept_channel_tokens", lambda p, k, N, S, W: np.arange(0)),
    "zero_head_scored_as_zero": lambda mp: mp.setattr(
        A, "full_width_tokens",
        (lambda f: (lambda p, k, N, S, W, Wl, fl=None:
                    np.arange(N) if (p == FULL and k == 0) else f(p, k, N, S, W, Wl, fl)))(A.full_width_tokens)),
    "local_includes_one_more": lambda mp: mp.setattr(
        A, "full_width_tokens",
        (lambda f: (lambda p, k, N, S, W, Wl, fl=None:
                    f(p, k, N, S, W, Wl + 1 if p == LOCAL else Wl, fl)))(A.full_width_tokens)),
    "ring_slot_without_sink_offset": lambda mp: mp.setattr(
        LY, "region_a",
        (lambda f: (lambda p, N, S, W, Wl, fl=None, special_capacity=None:
                    (lambda r: ((r[0] - (S if p == FULL else 0)) % max(1, S + W) if p == FULL else r[0], r[1]))(
                        f(p, N, S, W, Wl, fl, special_capacity))))(LY.region_a)),
    "dense_formula_missing_factor_2": lambda mp: mp.setattr(
        F, "dense_kv_elements", lambda L, H, d, N: L * H * d * N),
    "mid_row_missing_v": lambda mp: mp.setattr(
        F, "resident_bytes",
        (lambda f: (lambda p, k, N, S, W, Wl, n_special=0, head_dim=128, elem_bytes=2:
                    f(p, k, N, S, W, Wl, n_special, head_dim, elem_bytes)
                    - F.resident_tokens(p, k, N, S, W, Wl, n_special)[1] * head_dim * elem_bytes))(F.resident_bytes)),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    MUTATIONS[name](monkeypatch)
    failures = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin catches mutation {name}"
