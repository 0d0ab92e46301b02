"""Quantised middle region (KIVI-style quantisation after LeanK pruning),
INT8 and FP8 (e4m3), vs the fp64 oracle over the dequantised cache.

Complete 128-row blocks of each head's middle are stored as one-byte codes
with per-channel K scales and per-token V scales (LeanK article §4.2 and
§5.2 problem 3; the pruning white paper §5.2.1); the open block stays bf16.
The codes and scales of every sealed block must equal the oracle's byte for
byte, the tail rows must equal the inputs, and decode must match the oracle
evaluated on the dequantised values element by element.  Every test runs
for both formats."""
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


@pytest.fixture(params=[lkb.KV_INT8, lkb.KV_FP8], ids=["int8", "fp8"])
def Q8(request):
    return request.param


def _max_err(o, ref):
    return float(np.abs(o.double().cpu().numpy() - ref).max())


@pytest.mark.parametrize("counts", [(0, 64), (64, 64), None], ids=["k0-64", "k64-64", "seeded"])
def test_tiny_seal_during_appends(cuda, Q8, counts):
    # S + W = 68: prefill 560 leaves 3 sealed blocks + 108 tail rows; the
    # appends seal a fourth block at 580 tokens
    masks = None if counts is None else S.masks_with_counts(TINY, counts)
    case = Case(TINY, total=600, masks=masks, kv_format=Q8)
    case.prefill(0, 560)
    case.check_layout(0, 560)
    for t in range(560, 600):
        case.append(0, t)
        if t % 8 == 7 or t in (579, 580, 581):
            N = t + 1
            q = case.q(0, N, step=t)
            o = case.cache.decode(0, q)
            case.cache.check()
            assert _max_err(o, case.expected(0, q, N)) <= DECODE_TOL, N
            case.check_layout(0, N)


def test_llama_layer_all_widths(cuda, Q8):
    w = LLAMA.scaled(context=3000, batch=2)
    masks = S.masks_with_counts(w, [0, 32, 64, 96, 128, 32, 0, 64])
    case = Case(w, total=3003, masks=masks, kv_format=Q8)
    case.prefill(0, 2990)
    for t in range(2990, 3003):
        case.append(0, t)
    q = case.q(0, 3003)
    o = case.cache.decode(0, q)
    case.cache.check()
    ref = case.expected(0, q, 3003)
    assert _max_err(o, ref) <= DECODE_TOL
    case.check_layout(0, 3003)
    # the kernel reads the quantised values: the bf16 oracle is measurably off
    exact = Case(w, total=3003, masks=masks)
    ref_bf16 = exact.expected(0, q, 3003)
    assert np.abs(ref - ref_bf16).max() > 10 * np.abs(o.double().cpu().numpy() - ref).max()


@pytest.mark.parametrize("ctas", [1, 7, 0])
def test_split_invariance(cuda, Q8, ctas):
    w = LLAMA.scaled(context=2300, batch=2)
    masks = S.masks_with_counts(w, [32, 64, 0, 96, 128, 32, 32, 64])
    case = Case(w, total=2300, masks=masks, kv_format=Q8)
    case.prefill(0, 2300)
    case.cache.set_decode_ctas(ctas)
    q = case.q(0, 2300)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 2300)) <= DECODE_TOL


def test_prefill_equals_appends_byte_for_byte(cuda, Q8):
    w = FASTGEN.scaled(num_layers=1, batch=2, context=900, policy_counts=(2, 2, 4))
    a = Case(w, total=930, kv_format=Q8)
    b = Case(w, total=930, kv_format=Q8)
    a.prefill(0, 930)
    b.prefill(0, 850)                       # S + W = 528: 2 sealed + 66 tail rows
    for t in range(850, 930):               # seals the third block at 912 tokens
        b.append(0, t)
    a.cache.check()
    b.cache.check()
    torch.cuda.synchronize()
    assert torch.equal(a.cache.buffer, b.cache.buffer)
    a.check_layout(0, 930)


def test_fastgen_policy_mix_two_layers(cuda, Q8):
    w = FASTGEN.scaled(num_layers=2, batch=3, context=1200, policy_counts=(6, 4, 6))
    case = Case(w, total=1203, kv_format=Q8)
    for layer in range(2):
        case.prefill(layer, 1200)
        for t in range(1200, 1203):
            case.append(layer, t)
        q = case.q(layer, 1203)
        o = case.cache.decode(layer, q)
        case.cache.check()
        assert _max_err(o, case.expected(layer, q, 1203)) <= DECODE_TOL, layer
        case.check_layout(layer, 1203)


def test_paged_release_and_refill(cuda, Q8):
    w = SERVING.scaled(num_layers=1, batch=3, context=1400)
    case = Case(w, total=1500, kv_format=Q8, middle_tokens=3 * 1000)
    k, v = case.history(0)
    lens = np.array([1400, 1100, 700], dtype=np.int32)
    case.cache.prefill_ragged(0, k[:, :1400].contiguous(), v[:, :1400].contiguous(), lens)
    # sealed blocks per head: 6 + 4 + 1
    heads = [h for h in range(8) if case.masks[0, h].sum() > 0]
    used = {}
    for h in heads:
        c = int(case.masks[0, h].sum())
        used[c] = used.get(c, 0) + 11
    for c, n in used.items():
        total, free = case.cache.pages(c)
        assert total - free == n, (c, total, free, n)
    case.check_layout(0, lens)
    case.cache.release(1)
    k[1].copy_(k[0])
    v[1].copy_(v[0])
    case.cache.prefill_sequence(0, 1, k[1, :1290].contiguous(), v[1, :1290].contiguous())
    lens[1] = 1290
    for step in range(40):                  # sequence 1 seals a block at 1296
        pos = torch.from_numpy(lens.astype(np.int64)).to(k.device)
        bi = torch.arange(3, device=k.device)
        case.cache.append(0, k[bi, pos].contiguous(), v[bi, pos].contiguous())
        lens = lens + 1
    q = case.q(0, int(lens.max()))
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, lens)) <= DECODE_TOL
    case.check_layout(0, lens)


def test_all_layers_in_one_launch(cuda, Q8):
    w = FASTGEN.scaled(num_layers=3, batch=2, context=800, policy_counts=(2, 2, 20))
    case = Case(w, total=802, kv_format=Q8)
    L = w.num_layers
    for layer in range(L):
        case.prefill(layer, 800)
    ks = torch.stack([case.history(l)[0][:, 800] for l in range(L)]).contiguous()
    vs = torch.stack([case.history(l)[1][:, 800] for l in range(L)]).contiguous()
    case.cache.append_layers(0, ks, vs, case.ids[:, 800].contiguous())
    qs = torch.stack([case.q(l, 801) for l in range(L)]).contiguous()
    o = case.cache.decode_layers(0, qs)
    case.cache.check()
    for layer in range(L):
        assert _max_err(o[layer], case.expected(layer, qs[layer], 801)) <= DECODE_TOL, layer


def test_sealing_edge_values_match_the_oracle_bit_for_bit(cuda, Q8):
    # Values planted on the quantiser's decision edges, in units of a scale
    # that is a power of two (so x / scale is exact in fp32): exact ties
    # (INT8 .5 steps; FP8 midpoints between neighbouring e4m3 values),
    # values one fp32 ulp either side of a tie, tiny negatives that round to
    # a zero code, zeros of both signs, and the absmax itself.  Every sealed
    # byte and scale must equal the oracle's (the same fp32 decisions).
    from oracle import quant as OQ
    w = TINY.scaled(num_q_heads=2, num_kv_heads=1, context=4 + 64 + 256)
    masks = S.masks_with_counts(w, [32])
    N = w.context
    case = Case(w, total=N, masks=masks, kv_format=Q8)
    kept = np.nonzero(masks[0, 0])[0]
    rs = np.random.default_rng(5)
    if Q8 == lkb.KV_FP8:
        qmax, scale = 448.0, 2.0 ** -6
        grid = OQ.e4m3_value(np.arange(0x7F))
        mids = (grid[:-1] + grid[1:]) / 2
        ties = np.concatenate([mids, -mids])
    else:
        qmax, scale = 127.0, 2.0 ** -4
        ties = np.concatenate([np.arange(126) + 0.5, -(np.arange(126) + 0.5)])
    edge = np.concatenate([ties, np.nextafter(ties, np.inf), np.nextafter(ties, -np.inf),
                           [0.0, -0.0, -2.0 ** -12, 2.0 ** -12, -1e-7, qmax, -qmax]])
    vals = (edge * scale).astype(np.float32)
    # bf16 holds only 8 significant bits: keep the values bf16 represents
    # exactly, so the cache's inputs are these very numbers
    vals = vals[torch.from_numpy(vals).to(torch.bfloat16).float().numpy() == vals]
    k = torch.randn((1, N, 1, 128), dtype=torch.float64, generator=torch.Generator().manual_seed(3))
    v = torch.randn((1, N, 1, 128), dtype=torch.float64, generator=torch.Generator().manual_seed(4))
    mid = slice(w.sink, w.sink + 256)           # the first two middle blocks (sealed)
    kb = rs.choice(vals, size=(256, len(kept)))
    vb = rs.choice(vals, size=(256, 128))
    kb[0, :] = qmax * scale                      # every K channel of block 0 reaches the absmax
    kb[128, :] = -qmax * scale
    vb[:, 0] = qmax * scale                      # every V token reaches it
    kk = k[0, mid, 0].numpy().copy()
    kk[:, kept] = kb
    k[0, mid, 0] = torch.from_numpy(kk)
    v[0, mid, 0] = torch.from_numpy(vb)
    case.hist[0] = (k.to(torch.bfloat16).to(cuda), v.to(torch.bfloat16).to(cuda))
    case.prefill(0, N)
    case.cache.check()
    case.check_layout(0, N)                      # codes and scales byte for byte
    q = case.q(0, N)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, N)) <= DECODE_TOL
