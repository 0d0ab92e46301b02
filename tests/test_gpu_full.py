"""Parity at the workloads' full sizes, in the launch configuration bench.py
times: lk_step / lk_step_layers in the library's automatic mode (one fused
launch for the single-layer 32K and 128K-token workloads and for the
32-layer FastGen step, append + decode launches over all 32 layers for the
64-sequence serving step),
after a prefill of N-1 tokens.  The oracle recomputes sampled (sequence, kv
head) outputs one by one from the same seeded history; the layout check
reads sampled heads' cache rows byte for byte."""
import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import synth as S
from helpers import DECODE_TOL, Case

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_pairs(w, layer, k, rng):
    pairs = [(int(rng.integers(w.batch)), int(rng.integers(w.num_kv_heads))) for _ in range(k)]
    return sorted(set(pairs))


def _token(case, layer, t):
    k, v = case.history(layer)
    ids = case.ids[:, t].contiguous() if len(case.is_special) else None
    return k[:, t].contiguous(), v[:, t].contiguous(), ids


def _check(case, layer, N, o, q, pairs, layout_pairs):
    ref = case.expected(layer, q, N, heads=pairs)
    G = case.w.group
    worst = 0.0
    for (b, h), r in ref.items():
        err = float(np.abs(o[b, h * G:(h + 1) * G].double().cpu().numpy() - r).max())
        worst = max(worst, err)
        assert err <= DECODE_TOL, (layer, b, h, err)
    case.check_layout(layer, N, heads=layout_pairs)
    return worst


def _check_layer(case, layer, N, pairs, layout_pairs, fused=None):
    """One layer: prefill N-1 tokens, then one lk_step with token N-1."""
    case.prefill(layer, N - 1)
    if fused is not None:
        assert case.cache.step_is_fused(layer, 1) == fused
    q = case.q(layer, N)
    k, v, ids = _token(case, layer, N - 1)
    o = case.cache.step(layer, q, k, v, ids)
    case.cache.check()
    worst = _check(case, layer, N, o, q, pairs, layout_pairs)
    case.drop_history(layer)
    return worst


def _check_all_layers(case, N, pick, fused):
    """Every layer prefilled to N-1 tokens, then one lk_step_layers over all
    of them (the bench's step); pick(layer) -> (pairs, layout_pairs)."""
    w = case.w
    L = w.num_layers
    ks, vs = [], []
    for layer in range(L):
        case.prefill(layer, N - 1)
        k, v, _ = _token(case, layer, N - 1)
        ks.append(k)
        vs.append(v)
        case.drop_history(layer)
    assert case.cache.step_is_fused(0, L) == fused
    ids = case.ids[:, N - 1].contiguous() if len(case.is_special) else None
    qs = torch.stack([case.q(layer, N) for layer in range(L)]).contiguous()
    o = case.cache.step_layers(0, qs, torch.stack(ks).contiguous(), torch.stack(vs).contiguous(), ids)
    case.cache.check()
    del ks, vs
    for layer in range(L):
        pairs, layout_pairs = pick(layer)
        _check(case, layer, N, o[layer], qs[layer], pairs, layout_pairs)
        case.drop_history(layer)


def test_full_llama31_8b_layer(cuda):
    w = S.WORKLOADS[1]
    case = Case(w, total=w.context, gen_device=cuda)
    pairs = [(0, h) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, pairs, fused=True)


def test_full_qwen25_7b_long(cuda):
    w = S.WORKLOADS[3]
    case = Case(w, total=w.context, gen_device=cuda)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, [(0, h) for h in range(w.num_kv_heads)], fused=True)


def test_full_serving_b64_all_layers(cuda):
    w = S.WORKLOADS[2]
    case = Case(w, total=w.context, gen_device=cuda)
    rng = np.random.default_rng(7)

    def pick(layer):
        pairs = _sample_pairs(w, layer, 4, rng)
        return pairs, pairs[:1]

    _check_all_layers(case, w.context, pick, fused=False)


def test_full_serving_b64_three_ctas(cuda):
    """The 32-layer serving cache (19.7 GB) decoded on three CTAs: each CTA's
    range of the line is ~6.5 GB, so the row ranges and the owners of the
    split entries are computed from offsets past 2^32 bytes.  Every output
    agrees with the default grid's (a different split, so within rounding of
    the partial merges), and sampled heads agree with the oracle."""
    w = S.WORKLOADS[2]
    N = w.context
    L = w.num_layers
    case = Case(w, total=N, gen_device=cuda)
    for layer in range(L):
        case.prefill(layer, N)
        case.drop_history(layer)
    assert sum(case.cache.resident_bytes(layer) for layer in range(L)) > 3 * (1 << 32)
    qs = torch.stack([case.q(layer, N) for layer in range(L)]).contiguous()
    o_def = case.cache.decode_layers(0, qs)
    case.cache.set_decode_ctas(3)
    o_3 = case.cache.decode_layers(0, qs)
    case.cache.check()
    case.cache.set_decode_ctas(0)
    assert float((o_3 - o_def).abs().max()) <= 2e-4
    rng = np.random.default_rng(5)
    for layer in (0, L // 2, L - 1):
        _check(case, layer, N, o_3[layer], qs[layer], _sample_pairs(w, layer, 3, rng), [])
        case.drop_history(layer)


def test_full_fastgen_mix_all_layers(cuda):
    w = S.WORKLOADS[4]
    case = Case(w, total=w.context, gen_device=cuda)
    rng = np.random.default_rng(11)

    def pick(layer):
        # one head of each policy present in the layer, plus a random one
        pairs = set(_sample_pairs(w, layer, 1, rng))
        for pol in (S.POLICY_FULL, S.POLICY_LOCAL, S.POLICY_SPECIAL):
            hs = np.nonzero(case.policies[layer] == pol)[0]
            if len(hs):
                pairs.add((int(rng.integers(w.batch)), int(hs[0])))
        pairs = sorted(pairs)
        return pairs, pairs[:2]

    _check_all_layers(case, w.context, pick, fused=True)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_full_fastgen_mix_quantized_all_layers(cuda, fmt):
    """The 32-layer FastGen step with INT8 / FP8 middles (append + decode
    launches, as the bench runs it).  Its FULL heads keep 32 or 64
    channels (stages of three 21 or 25 KB sealed blocks): each layer checks
    one FULL head of every width it has, one LOCAL and one SPECIAL head
    against the oracle."""
    from decode_attention_pruned_gb300 import binding as lkb
    w = S.WORKLOADS[4]
    case = Case(w, total=w.context, gen_device=cuda, kv_format=lkb.KV_INT8 if fmt == "int8" else lkb.KV_FP8)
    rng = np.random.default_rng(19)
    widths_seen = set()

    def pick(layer):
        pairs = set()
        by_width = {}
        for h in np.nonzero(case.policies[layer] == S.POLICY_FULL)[0]:
            by_width.setdefault(int(case.masks[layer, h].sum()), int(h))
        widths_seen.update(by_width)
        for h in by_width.values():
            pairs.add((int(rng.integers(w.batch)), h))
        for pol in (S.POLICY_LOCAL, S.POLICY_SPECIAL):
            hs = np.nonzero(case.policies[layer] == pol)[0]
            if len(hs):
                pairs.add((int(rng.integers(w.batch)), int(hs[0])))
        pairs = sorted(pairs)
        return pairs, pairs[:2]

    _check_all_layers(case, w.context, pick, fused=False)
    assert widths_seen == {32, 64}


def test_full_qwen25_7b_long_int8(cuda):
    from decode_attention_pruned_gb300 import binding as lkb
    w = S.WORKLOADS[3]
    case = Case(w, total=w.context, gen_device=cuda, kv_format=lkb.KV_INT8)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, [(1, h) for h in range(w.num_kv_heads)])


def test_full_qwen25_7b_long_fp8(cuda):
    from decode_attention_pruned_gb300 import binding as lkb
    w = S.WORKLOADS[3]
    case = Case(w, total=w.context, gen_device=cuda, kv_format=lkb.KV_FP8)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, [(2, h) for h in range(w.num_kv_heads)])


def test_full_serving_b64_fp8_all_layers(cuda):
    from decode_attention_pruned_gb300 import binding as lkb
    w = S.WORKLOADS[2]
    case = Case(w, total=w.context, gen_device=cuda, kv_format=lkb.KV_FP8)
    rng = np.random.default_rng(17)

    def pick(layer):
        pairs = _sample_pairs(w, layer, 3, rng)
        return pairs, pairs[:1]

    _check_all_layers(case, w.context, pick, fused=False)


def test_full_llama31_8b_layer_int8_paged(cuda):
    from decode_attention_pruned_gb300 import binding as lkb
    w = S.WORKLOADS[1]
    case = Case(w, total=w.context, gen_device=cuda, kv_format=lkb.KV_INT8, middle_tokens=w.context)
    pairs = [(0, h) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, pairs)


def test_full_llama31_8b_layer_paged(cuda):
    # bf16 middle rows in 128-row pages: each entry's ~248 pages are split
    # over 16 CTAs, most of which start inside a page (a short first tile,
    # then page ids loaded four tiles ahead)
    w = S.WORKLOADS[1]
    case = Case(w, total=w.context, gen_device=cuda, middle_tokens=w.context)
    pairs = [(0, h) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, pairs, fused=True)


def test_full_serving_b64_paged_all_layers(cuda):
    # the 32-layer serving step on a paged cache (24 pages per entry, every
    # CTA range crossing entries), as the bench's --layout paged runs it
    w = S.WORKLOADS[2]
    case = Case(w, total=w.context, gen_device=cuda, middle_tokens=w.batch * w.context)
    rng = np.random.default_rng(13)

    def pick(layer):
        pairs = _sample_pairs(w, layer, 3, rng)
        return pairs, pairs[:1]

    _check_all_layers(case, w.context, pick, fused=False)
