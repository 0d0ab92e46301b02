"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (one CTA per SM, append then decode).  The oracle recomputes sampled
(sequence, kv head) outputs one by one from the same seeded history; the
layout check reads sampled heads' cache rows byte for byte."""
import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import synth as S
from helpers import DECODE_TOL, Case

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_pairs(w, layer, k, rng):
    pairs = [(int(rng.integers(w.batch)), int(rng.integers(w.num_kv_heads))) for _ in range(k)]
    return sorted(set(pairs))


def _check_layer(case, layer, N, pairs, layout_pairs):
    case.prefill(layer, N - 1)
    case.append(layer, N - 1)
    q = case.q(layer, N)
    o = case.cache.decode(layer, q)
    case.cache.check()
    ref = case.expected(layer, q, N, heads=pairs)
    G = case.w.group
    worst = 0.0
    for (b, h), r in ref.items():
        err = float(np.abs(o[b, h * G:(h + 1) * G].double().cpu().numpy() - r).max())
        worst = max(worst, err)
        assert err <= DECODE_TOL, (layer, b, h, err)
    case.check_layout(layer, N, heads=layout_pairs)
    case.drop_history(layer)
    return worst


def test_full_llama31_8b_layer(cuda):
    w = S.WORKLOADS[1]
    case = Case(w, total=w.context, gen_device=cuda)
    pairs = [(0, h) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, pairs)


def test_full_qwen25_7b_long(cuda):
    w = S.WORKLOADS[3]
    case = Case(w, total=w.context, gen_device=cuda)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, [(0, h) for h in range(w.num_kv_heads)])


def test_full_serving_b64_all_layers(cuda):
    w = S.WORKLOADS[2]
    case = Case(w, total=w.context, gen_device=cuda)
    rng = np.random.default_rng(7)
    for layer in range(w.num_layers):
        pairs = _sample_pairs(w, layer, 4, rng)
        _check_layer(case, layer, w.context, pairs, pairs[:1])


def test_full_fastgen_mix_all_layers(cuda):
    w = S.WORKLOADS[4]
    case = Case(w, total=w.context, gen_device=cuda)
    rng = np.random.default_rng(11)
    for layer in range(w.num_layers):
        # one head of each policy present in the layer, plus a random one
        pairs = set(_sample_pairs(w, layer, 1, rng))
        for pol in (S.POLICY_FULL, S.POLICY_LOCAL, S.POLICY_SPECIAL):
            hs = np.nonzero(case.policies[layer] == pol)[0]
            if len(hs):
                pairs.add((int(rng.integers(w.batch)), int(hs[0])))
        pairs = sorted(pairs)
        _check_layer(case, layer, w.context, pairs, pairs[:2])


def test_full_qwen25_7b_long_int8(cuda):
    from decode_attention_pruned_gb300 import binding as lkb
    w = S.WORKLOADS[3]
    case = Case(w, total=w.context, gen_device=cuda, kv_format=lkb.KV_INT8)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, [(1, h) for h in range(w.num_kv_heads)])


def test_full_llama31_8b_layer_int8_paged(cuda):
    from decode_attention_pruned_gb300 import binding as lkb
    w = S.WORKLOADS[1]
    case = Case(w, total=w.context, gen_device=cuda, kv_format=lkb.KV_INT8, middle_tokens=w.context)
    pairs = [(0, h) for h in range(w.num_kv_heads)]
    _check_layer(case, 0, w.context, pairs, pairs)
