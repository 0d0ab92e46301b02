"""Paged middle region (continuous batching) vs the fp64 oracle.

The cache's middle rows live in 128-row pages of each width class, found
through a page table (paged KV blocks: the pruning white paper, yyx235 blog,
section 3.2 "granularity"; per-head variable allocation: FastGen article,
section 5.1).  Decode output is compared with the oracle element by element,
and every resident row is read back through the page table and compared byte
for byte with the layout the oracle expects.  Slots are released and
refilled with other sequences while the rest keep decoding."""
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
WIDTHS = (32, 64, 96, 128)


def _max_err(o, ref):
    return float(np.abs(o.double().cpu().numpy() - ref).max())


def _pages_held(case, layer, lens):
    """Pages per width class that heads of `layer` hold at lengths `lens`."""
    w = case.w
    held = {c: 0 for c in WIDTHS}
    for h in range(w.num_kv_heads):
        k = int(case.masks[layer, h].sum())
        if case.policies[layer, h] != S.POLICY_FULL or k == 0:
            continue
        for n in np.atleast_1d(lens):
            held[k] += -(-max(0, int(n) - w.sink - w.local) // 128)
    return held


def _free(case):
    return {c: case.cache.pages(c)[1] for c in WIDTHS}


@pytest.mark.parametrize("counts", [(0, 64), (64, 64), None], ids=["k0-64", "k64-64", "seeded"])
def test_tiny_paged_prefill_then_appends(cuda, counts):
    masks = None if counts is None else S.masks_with_counts(TINY, counts)
    # S + W = 68: the middle reaches 460 rows = 4 pages; appends cross into a 5th
    case = Case(TINY, total=720, masks=masks, middle_tokens=700)
    case.prefill(0, 580)
    case.check_layout(0, 580)
    for t in range(580, 720, 7):
        for u in range(t, min(t + 7, 720)):
            case.append(0, u)
        N = min(t + 7, 720)
        q = case.q(0, N, step=t)
        o = case.cache.decode(0, q)
        case.cache.check()
        assert _max_err(o, case.expected(0, q, N)) <= DECODE_TOL, N
        case.check_layout(0, N)


def test_llama_layer_all_widths_paged(cuda):
    w = LLAMA.scaled(context=3000, batch=2)
    masks = S.masks_with_counts(w, [0, 32, 64, 96, 128, 32, 0, 64])
    case = Case(w, total=3003, masks=masks, middle_tokens=2 * 3003)
    case.prefill(0, 2990)
    for t in range(2990, 3003):
        case.append(0, t)
    q = case.q(0, 3003)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 3003)) <= DECODE_TOL
    case.check_layout(0, 3003)


@pytest.mark.parametrize("ctas", [1, 7, 0])
def test_paged_matches_contiguous(cuda, ctas):
    w = LLAMA.scaled(context=2300, batch=2)
    masks = S.masks_with_counts(w, [32, 64, 0, 96, 128, 32, 32, 64])
    a = Case(w, total=2300, masks=masks)
    b = Case(w, total=2300, masks=masks, middle_tokens=4600)
    a.prefill(0, 2300)
    b.prefill(0, 2300)
    a.cache.set_decode_ctas(ctas)
    b.cache.set_decode_ctas(ctas)
    q = a.q(0, 2300)
    oa = a.cache.decode(0, q)
    ob = b.cache.decode(0, q)
    a.cache.check()
    b.cache.check()
    ref = a.expected(0, q, 2300)
    assert _max_err(oa, ref) <= DECODE_TOL
    assert _max_err(ob, ref) <= DECODE_TOL
    # only the tile boundaries (page-aligned vs range-aligned) differ
    assert float((oa - ob).abs().max()) <= 1e-4


def test_release_and_refill_slots(cuda):
    w = FASTGEN.scaled(num_layers=2, batch=4, context=1500, policy_counts=(4, 2, 10))
    case = Case(w, total=1600, middle_tokens=4 * 1600)
    L, B = w.num_layers, w.batch
    lens = np.array([1500, 1210, 700, 90], dtype=np.int32)
    for layer in range(L):
        k, v = case.history(layer)
        n_max = int(lens.max())
        case.cache.prefill_ragged(layer, k[:, :n_max].contiguous(), v[:, :n_max].contiguous(), lens,
                                  case.ids[:, :n_max].contiguous())
    total = {c: case.cache.pages(c)[0] for c in WIDTHS}
    held = {c: sum(_pages_held(case, l, lens)[c] for l in range(L)) for c in WIDTHS}
    assert _free(case) == {c: total[c] - held[c] for c in WIDTHS}

    def step(lens, tag):
        for layer in range(L):
            k, v = case.history(layer)
            pos = torch.from_numpy(lens.astype(np.int64)).to(k.device)
            bi = torch.arange(B, device=k.device)
            case.cache.append(layer, k[bi, pos].contiguous(), v[bi, pos].contiguous(),
                              case.ids[bi, pos].contiguous())
        lens = lens + 1
        for layer in range(L):
            q = case.q(layer, int(lens.max()), step=int(lens.sum()))
            o = case.cache.decode(layer, q)
            case.cache.check()
            assert _max_err(o, case.expected(layer, q, lens)) <= DECODE_TOL, (tag, layer)
            case.check_layout(layer, lens)
        return lens

    lens = step(lens, "before")
    # slot 1 finishes: its pages return, the slot is skipped by appends
    before = _free(case)
    back = {c: sum(_pages_held(case, l, lens[1])[c] for l in range(L)) for c in WIDTHS}
    case.cache.release(1)
    assert _free(case) == {c: before[c] + back[c] for c in WIDTHS}
    assert all(case.cache.lengths(l)[1] == 0 for l in range(L))
    # a new request takes slot 1: sequence 0's tokens at another length
    n_new = 1333
    for layer in range(L):
        k, v = case.history(layer)
        k[1].copy_(k[0])
        v[1].copy_(v[0])
    case.ids[1].copy_(case.ids[0])
    case.flags[1] = case.flags[0]
    for layer in range(L):
        k, v = case.history(layer)
        case.cache.prefill_sequence(layer, 1, k[1, :n_new].contiguous(), v[1, :n_new].contiguous(),
                                    case.ids[1, :n_new].contiguous())
    lens[1] = n_new
    assert list(case.cache.lengths(0)) == list(lens)
    for _ in range(3):
        lens = step(lens, "after")


def test_released_slot_is_skipped(cuda):
    w = SERVING.scaled(num_layers=1, batch=3, context=800)
    case = Case(w, total=802)
    case.prefill(0, 800)
    case.cache.release(2)
    case.append(0, 800)
    assert list(case.cache.lengths(0)) == [801, 801, 0]
    q = case.q(0, 801)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert torch.all(o[2] == 0)
    ref = case.expected(0, q, np.array([801, 801, 0]))
    assert _max_err(o, ref) <= DECODE_TOL
    # the slot cannot be refilled while it holds tokens, and refills at 0 tokens
    with pytest.raises(lkb.LeankError) as e:
        k, v = case.history(0)
        case.cache.prefill_sequence(0, 0, k[0, :5].contiguous(), v[0, :5].contiguous())
    assert e.value.status == lkb.LK_ERR_STATE
    k, v = case.history(0)
    case.cache.prefill_sequence(0, 2, k[2, :801].contiguous(), v[2, :801].contiguous())
    case.append(0, 801)
    assert list(case.cache.lengths(0)) == [802, 802, 802]
    q = case.q(0, 802)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 802)) <= DECODE_TOL
    case.check_layout(0, 802)


def test_page_exhaustion_is_refused_before_launch(cuda):
    w = SERVING.scaled(num_layers=1, batch=2, context=900)
    masks = S.masks_with_counts(w, [32] * 8)
    # S + W = 528; 256 middle tokens in all: 2 + 2 pages per head
    case = Case(w, total=1200, masks=masks, middle_tokens=256)
    total = case.cache.pages(32)[0]
    assert total == 8 * 4
    case.prefill(0, 528 + 200)               # 2 pages per head and sequence
    assert case.cache.pages(32)[1] == 0
    for t in range(728, 528 + 256):
        case.append(0, t)                    # fills the second pages
    with pytest.raises(lkb.LeankError) as e:
        case.append(0, 528 + 256)            # would open a third page
    assert e.value.status == lkb.LK_ERR_CAPACITY
    assert list(case.cache.lengths(0)) == [784, 784]
    case.cache.check()
    q = case.q(0, 784)
    o = case.cache.decode(0, q)
    assert _max_err(o, case.expected(0, q, 784)) <= DECODE_TOL
    # releasing one sequence frees its pages; the other grows into them
    case.cache.release(0)
    assert case.cache.pages(32)[1] == 16
    case.append(0, 784)
    assert list(case.cache.lengths(0)) == [0, 785]
    q = case.q(0, 785)
    o = case.cache.decode(0, q)
    case.cache.check()
    ref = case.expected(0, q, np.array([0, 785]))
    assert _max_err(o, ref) <= DECODE_TOL
    case.check_layout(0, np.array([0, 785]), heads=[(1, h) for h in range(8)])


def test_paged_all_layers_in_one_launch(cuda):
    w = FASTGEN.scaled(num_layers=4, batch=3, context=900, policy_counts=(4, 4, 24))
    case = Case(w, total=1030, middle_tokens=3 * 1030)
    L = w.num_layers
    for layer in range(L):
        case.prefill(layer, 900)
    for t in range(900, 1030):
        ks = torch.stack([case.history(l)[0][:, t] for l in range(L)]).contiguous()
        vs = torch.stack([case.history(l)[1][:, t] for l in range(L)]).contiguous()
        case.cache.append_layers(0, ks, vs, case.ids[:, t].contiguous())
    qs = torch.stack([case.q(l, 1030, step=3) for l in range(L)]).contiguous()
    o = case.cache.decode_layers(0, qs)
    case.cache.check()
    for layer in range(L):
        assert _max_err(o[layer], case.expected(layer, qs[layer], 1030)) <= DECODE_TOL, layer
        case.check_layout(layer, 1030)
