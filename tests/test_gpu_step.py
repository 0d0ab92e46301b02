"""The fused decode step (lk_step): the append of token t and attention with
the query of step t in one launch, against the fp64 oracle over tokens
0..t and against the split path (lk_append, then lk_decode_attn).

The order is the method's: the new K, V enter the cache, then the query
attends to everything resident (FastGen article, mhpn.cn, section 2.1; the
LeanK article, framerc.cn, section 3.1 for the split cache the token goes
into).  The fused launch scores the new token from its inputs, leaves out
the window slot it replaces, scores the token that slot sends to the middle
on the kept channels, and only then writes the cache; so its output must
match the oracle, and the cache it leaves must equal the split path's byte
for byte (contiguous caches) or row for row through the page table (paged
caches, whose free pages may be handed out in another order)."""
import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from helpers import DECODE_TOL, Case

pytestmark = pytest.mark.gpu

TINY = S.WORKLOADS[0]
LLAMA = S.WORKLOADS[1]
SERVING = S.WORKLOADS[2]
FASTGEN = S.WORKLOADS[4]


def _max_err(o, ref):
    return float(np.abs(o.double().cpu().numpy() - ref).max())


def _token(case, layer, pos):
    """k, v [B, Hkv, 128] and ids [B] of the token at position pos[b] of each
    sequence (pos an int or one position per sequence)."""
    k, v = case.history(layer)
    B = case.w.batch
    p = torch.as_tensor(np.broadcast_to(np.asarray(pos, dtype=np.int64), (B,)).copy(), device=k.device)
    bi = torch.arange(B, device=k.device)
    ids = case.ids[bi, p].contiguous() if len(case.is_special) else None
    return k[bi, p].contiguous(), v[bi, p].contiguous(), ids


def _fused(case):
    """The case's cache runs lk_step as one launch whatever its size."""
    case.cache.set_step_mode(lkb.STEP_FUSED)
    return case


def _twins(w, total, **kw):
    return _fused(Case(w, total=total, **kw)), Case(w, total=total, **kw)


def _step_both(fused, split, layer, pos, q):
    """One step on both caches: fused on one, append + decode on the other."""
    k, v, ids = _token(fused, layer, pos)
    of = fused.cache.step(layer, q, k, v, ids)
    split.cache.append(layer, k, v, ids)
    os_ = split.cache.decode(layer, q)
    return of, os_


@pytest.mark.parametrize("counts", [(0, 64), (64, 64), None], ids=["k0-64", "k64-64", "seeded"])
def test_tiny_steps_from_an_empty_cache(cuda, counts):
    # S = 4, W = 64: the steps fill the sinks (entries without resident
    # tokens at t = 0), the window, and wrap the ring into the middle
    masks = None if counts is None else S.masks_with_counts(TINY, counts)
    fused, split = _twins(TINY, 200, masks=masks)
    for t in range(200):
        q = fused.q(0, t + 1, step=t)
        of, os_ = _step_both(fused, split, 0, t, q)
        if t % 9 == 0 or t in (3, 4, 67, 68, 69, 131, 132, 199):
            fused.cache.check()
            assert _max_err(of, fused.expected(0, q, t + 1)) <= DECODE_TOL, t
            assert float((of - os_).abs().max()) <= 1e-4, t
    fused.cache.check()
    split.cache.check()
    assert list(fused.cache.lengths(0)) == [200]
    torch.cuda.synchronize()
    assert torch.equal(fused.cache.buffer, split.cache.buffer)
    fused.check_layout(0, 200)


@pytest.mark.parametrize("paged", [False, True], ids=["contiguous", "paged"])
@pytest.mark.parametrize("ctas", [1, 7, 0])
def test_llama_layer_all_widths(cuda, paged, ctas):
    w = LLAMA.scaled(context=3100, batch=2)
    masks = S.masks_with_counts(w, [0, 32, 64, 96, 128, 32, 0, 64])
    mt = 2 * 3100 if paged else None
    fused, split = _twins(w, 3100, masks=masks, middle_tokens=mt)
    # S + W = 1040: the token appended at n = 3088 evicts middle row 2048,
    # the first row of page 16
    fused.prefill(0, 3075)
    split.prefill(0, 3075)
    fused.cache.set_decode_ctas(ctas)
    split.cache.set_decode_ctas(ctas)
    for t in range(3075, 3100):
        q = fused.q(0, t + 1, step=t)
        of, os_ = _step_both(fused, split, 0, t, q)
        if t % 6 == 0 or t in (3087, 3088, 3089, 3099):
            fused.cache.check()
            assert _max_err(of, fused.expected(0, q, t + 1)) <= DECODE_TOL, t
            assert float((of - os_).abs().max()) <= 1e-4, t
    fused.cache.check()
    split.cache.check()
    torch.cuda.synchronize()
    if paged:
        assert {c: fused.cache.pages(c) for c in (32, 64, 96, 128)} == \
            {c: split.cache.pages(c) for c in (32, 64, 96, 128)}
    else:
        assert torch.equal(fused.cache.buffer, split.cache.buffer)
    fused.check_layout(0, 3100)


def test_fastgen_policies_two_layers_in_one_launch(cuda):
    # LOCAL heads wrap their W_loc = 256 ring; SPECIAL heads take a token only
    # when its id is special; FULL heads evict into the middle
    w = FASTGEN.scaled(num_layers=2, batch=3, context=600, policy_counts=(6, 4, 6))
    fused, split = _twins(w, 640)
    L = w.num_layers
    for layer in range(L):
        fused.prefill(layer, 600)
        split.prefill(layer, 600)
    for t in range(600, 640):
        qs = torch.stack([fused.q(l, t + 1, step=t) for l in range(L)]).contiguous()
        ks = torch.stack([_token(fused, l, t)[0] for l in range(L)]).contiguous()
        vs = torch.stack([_token(fused, l, t)[1] for l in range(L)]).contiguous()
        ids = _token(fused, 0, t)[2]
        of = fused.cache.step_layers(0, qs, ks, vs, ids)
        split.cache.append_layers(0, ks, vs, ids)
        os_ = split.cache.decode_layers(0, qs)
        if t % 8 == 0 or t == 639:
            fused.cache.check()
            for layer in range(L):
                assert _max_err(of[layer], fused.expected(layer, qs[layer], t + 1)) <= DECODE_TOL, (t, layer)
            assert float((of - os_).abs().max()) <= 1e-4, t
    fused.cache.check()
    torch.cuda.synchronize()
    assert torch.equal(fused.cache.buffer, split.cache.buffer)
    for layer in range(L):
        fused.check_layout(layer, 640)


def test_fastgen_from_empty_special_rows(cuda):
    # SPECIAL heads start with no rows: entries with nothing resident take
    # the new token alone when it is special and give o = 0 otherwise
    w = FASTGEN.scaled(num_layers=1, batch=4, context=64, policy_counts=(2, 4, 2))
    fused, split = _twins(w, 64)
    assert fused.flags[:, :40].any()
    for t in range(40):
        q = fused.q(0, t + 1, step=t)
        of, os_ = _step_both(fused, split, 0, t, q)
        fused.cache.check()
        assert _max_err(of, fused.expected(0, q, t + 1)) <= DECODE_TOL, t
        assert float((of - os_).abs().max()) <= 1e-4, t
    torch.cuda.synchronize()
    assert torch.equal(fused.cache.buffer, split.cache.buffer)
    fused.check_layout(0, 40)


def test_ragged_released_and_refilled_slots(cuda):
    w = SERVING.scaled(num_layers=1, batch=3, context=1400)
    fused, split = _twins(w, 1500, middle_tokens=3 * 1500)
    lens = np.array([1400, 1100, 700], dtype=np.int32)
    for c in (fused, split):
        k, v = c.history(0)
        c.cache.prefill_ragged(0, k[:, :1400].contiguous(), v[:, :1400].contiguous(), lens)
        c.cache.release(1)
    lens[1] = 0
    for step in range(12):
        q = fused.q(0, int(lens.max()) + 1, step=step)
        of, os_ = _step_both(fused, split, 0, lens, q)
        lens = lens + np.array([1, 0, 1], dtype=np.int32)
        assert list(fused.cache.lengths(0)) == list(lens)
        fused.cache.check()
        assert torch.all(of[1] == 0)
        assert _max_err(of, fused.expected(0, q, lens)) <= DECODE_TOL, step
        assert float((of - os_).abs().max()) <= 1e-4
    # slot 1 takes a new sequence and decodes on
    for c in (fused, split):
        k, v = c.history(0)
        c.cache.prefill_sequence(0, 1, k[1, :1290].contiguous(), v[1, :1290].contiguous())
    lens[1] = 1290
    for step in range(12):
        q = fused.q(0, int(lens.max()) + 1, step=100 + step)
        of, os_ = _step_both(fused, split, 0, lens, q)
        lens = lens + 1
        fused.cache.check()
        assert _max_err(of, fused.expected(0, q, lens)) <= DECODE_TOL, step
    split.cache.check()
    assert list(fused.cache.lengths(0)) == list(split.cache.lengths(0)) == list(lens)
    fused.check_layout(0, lens)
    split.check_layout(0, lens)


def test_int8_middle_runs_append_then_decode(cuda):
    # an append may seal a block, which changes the values decode reads: the
    # step is the two launches, so both paths agree exactly
    fused, split = _twins(TINY, 600, masks=S.masks_with_counts(TINY, (64, 32)), kv_format=lkb.KV_INT8)
    fused.prefill(0, 570)
    split.prefill(0, 570)
    for t in range(570, 590):                  # seals a block at 580 tokens
        q = fused.q(0, t + 1, step=t)
        of, os_ = _step_both(fused, split, 0, t, q)
        assert torch.equal(of, os_), t
    fused.cache.check()
    assert _max_err(of, fused.expected(0, q, 590)) <= DECODE_TOL
    torch.cuda.synchronize()
    assert torch.equal(fused.cache.buffer, split.cache.buffer)


def test_full_sequence_is_refused_before_launch(cuda):
    w = SERVING.scaled(num_layers=1, batch=2, context=600)
    case = _fused(Case(w, total=601, capacity=600))
    case.prefill(0, 600)
    q = case.q(0, 601)
    k, v, ids = _token(case, 0, 600)
    with pytest.raises(lkb.LeankError) as e:
        case.cache.step(0, q, k, v, ids)
    assert e.value.status == lkb.LK_ERR_CAPACITY
    assert list(case.cache.lengths(0)) == [600, 600]
    case.cache.check()
    o = case.cache.decode(0, q)
    assert _max_err(o, case.expected(0, q, 600)) <= DECODE_TOL


@pytest.mark.parametrize("offset", [5, -1], ids=["past_vocab", "negative"])
def test_out_of_range_id_is_reported(cuda, offset):
    w = FASTGEN.scaled(num_layers=1, batch=2, context=300, policy_counts=(2, 2, 4))
    case = _fused(Case(w, total=302))
    case.prefill(0, 300)
    k, v, ids = _token(case, 0, 300)
    bad = ids.clone()
    bad[1] = w.vocab + offset if offset > 0 else offset
    case.cache.step(0, case.q(0, 301), k, v, bad)
    with pytest.raises(lkb.LeankError) as e:
        case.cache.check()
    assert e.value.status == lkb.LK_ERR_ARG
    # the token still entered (as not special), as lk_append does
    assert list(case.cache.lengths(0)) == [301, 301]


@pytest.mark.parametrize("fused_step", [True, False], ids=["fused", "split"])
def test_one_long_head_over_many_ctas(cuda, fused_step):
    # one full-width head holds most of the bytes, so its entry spans ~100
    # CTAs and the in-launch combine merges its partials in several rounds
    w = LLAMA.scaled(context=20000)
    masks = S.masks_with_counts(w, [128, 0, 0, 0, 0, 0, 0, 0])
    case = _fused(Case(w, total=20004, masks=masks))
    case.prefill(0, 20000)
    for t in range(20000, 20004):
        q = case.q(0, t + 1, step=t)
        k, v, ids = _token(case, 0, t)
        if fused_step:
            o = case.cache.step(0, q, k, v, ids)
        else:
            case.cache.append(0, k, v, ids)
            o = case.cache.decode(0, q)
        case.cache.check()
        assert _max_err(o, case.expected(0, q, t + 1)) <= DECODE_TOL, t
    case.check_layout(0, 20004)


def test_automatic_mode_fuses_small_or_long_few_entry_launches(cuda):
    # one launch for launches of at most 32 entries (the 32K-token layer, the
    # 0.24 MB tiny layer) and for larger ones whose CTAs stream long and meet
    # few entries; two for short CTAs over more than 32 entries, for many
    # entries per CTA, and for INT8
    big = Case(LLAMA, total=LLAMA.context + 2)
    big.prefill(0, LLAMA.context)
    assert big.cache.step_is_fused(0, 1)
    small = Case(TINY, total=TINY.context + 2)
    small.prefill(0, TINY.context)
    assert small.cache.step_is_fused(0, 1)
    small.cache.set_step_mode(lkb.STEP_SPLIT)
    assert not small.cache.step_is_fused(0, 1)
    big.cache.set_step_mode(lkb.STEP_SPLIT)
    assert not big.cache.step_is_fused(0, 1)
    # 2 layers x 3 sequences x 8 heads = 48 entries, ~64 KB per CTA
    short = Case(FASTGEN.scaled(num_layers=2, batch=3, context=600, policy_counts=(6, 4, 6)), total=602)
    for layer in range(2):
        short.prefill(layer, 600)
    assert not short.cache.step_is_fused(0, 2)
    # 32 layers x 64 sequences x 8 heads: 108 entries per CTA
    many = Case(SERVING.scaled(context=600), total=602, gen_device=cuda)
    for layer in range(many.w.num_layers):
        many.prefill(layer, 600)
        many.drop_history(layer)
    assert not many.cache.step_is_fused(0, many.w.num_layers)
    q8 = Case(TINY, total=TINY.context + 2, kv_format=lkb.KV_INT8)
    q8.cache.set_step_mode(lkb.STEP_FUSED)
    assert not q8.cache.step_is_fused(0, 1)
    # either way the step gives the oracle's output
    q = big.q(0, LLAMA.context + 1)
    k, v, ids = _token(big, 0, LLAMA.context)
    o = big.cache.step(0, q, k, v, ids)
    big.cache.check()
    assert _max_err(o, big.expected(0, q, LLAMA.context + 1)) <= DECODE_TOL


@pytest.mark.parametrize("hq,hkv", [(4, 4), (32, 4), (12, 4)], ids=["G1", "G8", "G3"])
def test_fused_query_group_sizes(cuda, hq, hkv):
    # the token fold splits warp 0 as 8 heads x 4 channel quarters: G = 1,
    # the full G = 8 and an odd G = 3, on every width class (with evictions)
    w = LLAMA.scaled(num_q_heads=hq, num_kv_heads=hkv, context=1700, batch=2)
    masks = S.masks_with_counts(w, [32, 0, 96, 128])
    fused, split = _twins(w, 1706, masks=masks)
    fused.prefill(0, 1700)
    split.prefill(0, 1700)
    for t in range(1700, 1706):
        q = fused.q(0, t + 1, step=t)
        of, os_ = _step_both(fused, split, 0, t, q)
        fused.cache.check()
        assert _max_err(of, fused.expected(0, q, t + 1)) <= DECODE_TOL, t
        assert float((of - os_).abs().max()) <= 1e-4, t
    torch.cuda.synchronize()
    assert torch.equal(fused.cache.buffer, split.cache.buffer)


@pytest.mark.parametrize("layers,batch,hkv", [(1, 4, 8), (1, 3, 11), (4, 2, 4), (3, 11, 1)],
                         ids=["E32-1layer", "E33-1layer", "E32-4layers", "E33-3layers"])
def test_fused_steps_either_side_of_32_entries(cuda, layers, batch, hkv):
    # Launches of at most 32 (layer, sequence, kv head) entries keep the
    # lengths their split read in shared memory and advance them right after
    # every CTA's split; larger ones advance them at the end.  Both sides of
    # the boundary, one layer and several, with LOCAL / SPECIAL / FULL heads:
    # outputs against the oracle and the two-launch path, lengths after every
    # step, and the cache byte for byte.
    n = layers * hkv
    counts = (n // 3, n // 3, n - 2 * (n // 3))
    w = FASTGEN.scaled(num_layers=layers, batch=batch, num_q_heads=4 * hkv, num_kv_heads=hkv, context=600,
                       policy_counts=counts)
    fused, split = _twins(w, 612)
    L = w.num_layers
    for layer in range(L):
        fused.prefill(layer, 600)
        split.prefill(layer, 600)
    for t in range(600, 612):
        qs = torch.stack([fused.q(l, t + 1, step=t) for l in range(L)]).contiguous()
        ks = torch.stack([_token(fused, l, t)[0] for l in range(L)]).contiguous()
        vs = torch.stack([_token(fused, l, t)[1] for l in range(L)]).contiguous()
        ids = _token(fused, 0, t)[2]
        of = fused.cache.step_layers(0, qs, ks, vs, ids)
        split.cache.append_layers(0, ks, vs, ids)
        os_ = split.cache.decode_layers(0, qs)
        fused.cache.check()
        for layer in range(L):
            assert list(fused.cache.lengths(layer)) == [t + 1] * batch, (t, layer)
        assert float((of - os_).abs().max()) <= 1e-4, t
        if t % 4 == 3:
            for layer in range(L):
                assert _max_err(of[layer], fused.expected(layer, qs[layer], t + 1)) <= DECODE_TOL, (t, layer)
    torch.cuda.synchronize()
    assert torch.equal(fused.cache.buffer, split.cache.buffer)
    for layer in range(L):
        fused.check_layout(layer, 612)
