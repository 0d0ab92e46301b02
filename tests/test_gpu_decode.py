"""GPU decode attention vs the fp64 oracle, element by element, at sizes the
oracle finishes in seconds (several 64-row tiles and ragged tails).  Every
call goes through the C ABI (libleank.so)."""
import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from helpers import DECODE_TOL, Case
from oracle import masks as OM

pytestmark = pytest.mark.gpu

TINY = S.WORKLOADS[0]
LLAMA = S.WORKLOADS[1]
SERVING = S.WORKLOADS[2]
QWEN = S.WORKLOADS[3]
FASTGEN = S.WORKLOADS[4]


def _max_err(o, ref):
    return float(np.abs(o.double().cpu().numpy() - ref).max())


def _decode_steps(case, layer, n0, n_steps, layout=False):
    case.prefill(layer, n0)
    if layout:
        case.check_layout(layer, n0)
    worst = 0.0
    for t in range(n0, n0 + n_steps):
        case.append(layer, t)
        N = t + 1
        q = case.q(layer, N, step=t)
        o = case.cache.decode(layer, q)
        case.cache.check()
        err = _max_err(o, case.expected(layer, q, N))
        assert err <= DECODE_TOL, (layer, N, err)
        worst = max(worst, err)
        if layout:
            case.check_layout(layer, N)
    return worst


@pytest.mark.parametrize("counts", [(0, 0), (0, 64), (64, 0), (64, 64), None],
                         ids=["k0-0", "k0-64", "k64-0", "k64-64", "seeded"])
def test_tiny_prefill_then_16_appends(cuda, counts):
    masks = None if counts is None else S.masks_with_counts(TINY, counts)
    case = Case(TINY, total=528, masks=masks)
    _decode_steps(case, 0, 512, 16, layout=True)


def test_llama_layer_shape_all_widths(cuda):
    w = LLAMA.scaled(context=3000)
    masks = S.masks_with_counts(w, [0, 32, 64, 96, 128, 32, 0, 64])
    case = Case(w, total=3003, masks=masks)
    _decode_steps(case, 0, 3000, 3, layout=True)


def test_llama_layer_seeded_masks_outliers(cuda):
    w = LLAMA.scaled(context=2600)
    case = Case(w, total=2601)
    _decode_steps(case, 0, 2600, 1, layout=True)


def test_serving_shape_two_layers(cuda):
    w = SERVING.scaled(num_layers=2, batch=3, context=700)
    case = Case(w, total=702)
    for layer in range(2):
        _decode_steps(case, layer, 700, 2, layout=True)


def test_qwen_shape_group7_rope(cuda):
    w = QWEN.scaled(batch=2, context=2500)
    masks = S.masks_with_counts(w, [32, 0, 96, 64])
    case = Case(w, total=2501, masks=masks)
    _decode_steps(case, 0, 2500, 1, layout=True)


def test_fastgen_policy_mix(cuda):
    w = FASTGEN.scaled(num_layers=2, batch=3, context=900, policy_counts=(6, 4, 6))
    case = Case(w, total=903)
    for layer in range(2):
        _decode_steps(case, layer, 880, 23, layout=(layer == 0))


@pytest.mark.parametrize("ctas", [1, 2, 7, 0])
def test_split_invariance(cuda, ctas):
    w = LLAMA.scaled(context=2300, batch=2)
    masks = S.masks_with_counts(w, [32, 64, 0, 96, 128, 32, 32, 64])
    case = Case(w, total=2300, masks=masks)
    case.prefill(0, 2300)
    case.cache.set_decode_ctas(ctas)
    q = case.q(0, 2300)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 2300)) <= DECODE_TOL


@pytest.mark.parametrize("N", [1, 3, 16, 17, 1039, 1040, 1041, 1105])
def test_region_boundaries(cuda, N):
    # S = 16, W = 1024: below the sinks, inside the window fill, at the first
    # eviction, and one ragged tile past it
    w = LLAMA.scaled(context=N)
    masks = S.masks_with_counts(w, [0, 32, 64, 96, 128, 32, 0, 64])
    case = Case(w, total=N, masks=masks)
    case.prefill(0, N - 1)
    case.append(0, N - 1)
    q = case.q(0, N)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, N)) <= DECODE_TOL
    case.check_layout(0, N)


def test_all_heads_dropped(cuda):
    w = SERVING.scaled(num_layers=1, batch=2, context=1500)
    masks = np.zeros((1, 8, 128), dtype=np.uint8)
    case = Case(w, total=1500, masks=masks)
    case.prefill(0, 1500)
    q = case.q(0, 1500)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 1500)) <= DECODE_TOL


def test_special_head_without_special_tokens_gives_zero(cuda):
    w = FASTGEN.scaled(num_layers=1, batch=2, context=300, policy_counts=(2, 4, 2))
    case = Case(w, total=300)
    case.flags[:] = False
    case.is_special[:] = 0
    case.plan = lkb.Plan.for_workload(w, case.masks, case.policies, case.is_special)
    case.cache = lkb.Cache(case.plan, w.batch, 300)
    case.prefill(0, 300)
    q = case.q(0, 300)
    o = case.cache.decode(0, q)
    case.cache.check()
    ref = case.expected(0, q, 300)
    assert _max_err(o, ref) <= DECODE_TOL
    G = w.group
    for h in range(8):
        if case.policies[0, h] == S.POLICY_SPECIAL:
            assert torch.all(o[:, h * G:(h + 1) * G] == 0)


def test_empty_layer_decodes_to_zero(cuda):
    w = TINY
    case = Case(w, total=4)
    q = case.q(0, 1)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert torch.all(o == 0)


def test_prefill_equals_appends_byte_for_byte(cuda):
    w = FASTGEN.scaled(num_layers=1, batch=2, context=700, policy_counts=(3, 2, 3))
    a = Case(w, total=716)
    b = Case(w, total=716)
    a.prefill(0, 716)
    b.prefill(0, 700)
    for t in range(700, 716):
        b.append(0, t)
    a.cache.check()
    b.cache.check()
    torch.cuda.synchronize()
    assert torch.equal(a.cache.buffer, b.cache.buffer)
    a.check_layout(0, 716)


def test_step_host_matches_device_path(cuda):
    w = SERVING.scaled(num_layers=1, batch=2, context=600)
    a = Case(w, total=601)
    b = Case(w, total=601)
    a.prefill(0, 600)
    b.prefill(0, 600)
    k, v = a.history(0)
    q = a.q(0, 601)
    # pinned buffers: the host entry point reads them in place with the append
    # and decode launches (no bulk copies from host memory), so the device
    # call runs as those two launches too -- the same launches on the same
    # values
    a.cache.set_step_mode(lkb.STEP_SPLIT)
    o_dev = a.cache.step(0, q, k[:, 600].contiguous(), v[:, 600].contiguous())
    pin = lambda t: t.cpu().pin_memory()
    o_host = torch.empty(o_dev.shape, dtype=torch.float32).pin_memory()
    b.cache.step_host(0, pin(q), pin(k[:, 600].contiguous()), pin(v[:, 600].contiguous()), None, o_host)
    torch.cuda.synchronize()
    b.cache.check()
    assert torch.equal(o_host, o_dev.cpu())
    assert float(np.abs(o_host.double().numpy() - a.expected(0, q, 601)).max()) <= DECODE_TOL
    assert torch.equal(a.cache.buffer, b.cache.buffer)


def test_step_host_pageable_buffers_are_copied(cuda):
    # pageable host memory cannot be read by the kernels: the step stages
    # the inputs through the workspace and copies o back, with the same result
    w = SERVING.scaled(num_layers=1, batch=2, context=600)
    a = Case(w, total=601)
    b = Case(w, total=601)
    a.prefill(0, 600)
    b.prefill(0, 600)
    k, v = a.history(0)
    q = a.q(0, 601)
    o_dev = a.cache.step(0, q, k[:, 600].contiguous(), v[:, 600].contiguous())
    o_host = torch.empty(o_dev.shape, dtype=torch.float32)
    b.cache.step_host(0, q.cpu(), k[:, 600].contiguous().cpu(), v[:, 600].contiguous().cpu(), None, o_host)
    torch.cuda.synchronize()
    b.cache.check()
    assert torch.equal(o_host, o_dev.cpu())
    assert torch.equal(a.cache.buffer, b.cache.buffer)


def test_step_host_packed_matches_device_path(cuda):
    # one pinned block q | k | v, read in place by the append and decode
    # launches (o written into the mapped host buffer): the device call run
    # as those two launches gives identical o and cache bytes
    w = SERVING.scaled(num_layers=1, batch=2, context=600)
    a = Case(w, total=601)
    b = Case(w, total=601)
    for case in (a, b):
        case.prefill(0, 600)
    a.cache.set_step_mode(lkb.STEP_SPLIT)
    k, v = a.history(0)
    q = a.q(0, 601)
    kn, vn = k[:, 600].contiguous(), v[:, 600].contiguous()
    o_dev = a.cache.step(0, q, kn, vn)
    blk = torch.cat([t.cpu().contiguous().view(torch.uint8).reshape(-1) for t in (q, kn, vn)]).pin_memory()
    o_host = torch.full(o_dev.shape, float("nan"), dtype=torch.float32).pin_memory()
    b.cache.step_host_packed(0, blk, False, o_host)
    torch.cuda.synchronize()
    b.cache.check()
    assert torch.equal(o_host, o_dev.cpu())
    assert float(np.abs(o_host.double().numpy() - a.expected(0, q, 601)).max()) <= DECODE_TOL
    assert torch.equal(a.cache.buffer, b.cache.buffer)


def test_capacity_is_enforced(cuda):
    w = TINY
    case = Case(w, total=10, capacity=10)
    case.prefill(0, 10)
    with pytest.raises(lkb.LeankError) as e:
        case.append(0, 9)
    assert e.value.status == lkb.LK_ERR_CAPACITY
    with pytest.raises(lkb.LeankError) as e:
        case.prefill(0, 5)
    assert e.value.status == lkb.LK_ERR_STATE


def test_special_overflow_is_reported_on_device(cuda):
    w = FASTGEN.scaled(num_layers=1, batch=1, context=400, policy_counts=(2, 4, 2))
    case = Case(w, total=400, special_capacity=4)
    case.prefill(0, 400)
    with pytest.raises(lkb.LeankError) as e:
        case.cache.check()
    assert e.value.status == lkb.LK_ERR_CAPACITY
    case.cache.check()   # cleared


def test_all_layers_in_one_append_and_one_decode(cuda):
    w = FASTGEN.scaled(num_layers=4, batch=3, context=700, policy_counts=(10, 6, 16))
    case = Case(w, total=702)
    L = w.num_layers
    for layer in range(L):
        case.prefill(layer, 700)
    for t in (700, 701):
        ks = torch.stack([case.history(l)[0][:, t] for l in range(L)]).contiguous()
        vs = torch.stack([case.history(l)[1][:, t] for l in range(L)]).contiguous()
        case.cache.append_layers(0, ks, vs, case.ids[:, t].contiguous())
        qs = torch.stack([case.q(l, t + 1, step=t) for l in range(L)]).contiguous()
        o = case.cache.decode_layers(0, qs)
        case.cache.check()
        for layer in range(L):
            assert case.cache.length(layer) == t + 1
            assert _max_err(o[layer], case.expected(layer, qs[layer], t + 1)) <= DECODE_TOL, (layer, t)
    for layer in range(L):
        case.check_layout(layer, 702)
    # a sub-range of layers
    q2 = torch.stack([case.q(l, 702, step=9) for l in (1, 2)]).contiguous()
    o2 = case.cache.decode_layers(1, q2)
    for i, layer in enumerate((1, 2)):
        assert _max_err(o2[i], case.expected(layer, q2[i], 702)) <= DECODE_TOL


def test_ragged_lengths(cuda):
    # four sequences at different lengths: past the window, inside the window
    # fill, and below the sinks; then appends advance each at its own position
    w = FASTGEN.scaled(num_layers=1, batch=4, context=1300, policy_counts=(3, 2, 3))
    case = Case(w, total=1304)
    k, v = case.history(0)
    lens = np.array([1300, 1163, 700, 9], dtype=np.int32)
    n_max = int(lens.max())
    case.cache.prefill_ragged(0, k[:, :n_max].contiguous(), v[:, :n_max].contiguous(), lens,
                              case.ids[:, :n_max].contiguous())
    assert list(case.cache.lengths(0)) == list(lens)
    case.check_layout(0, lens)
    B = w.batch
    for step in range(3):
        pos = torch.from_numpy(lens.astype(np.int64)).to(k.device)
        bi = torch.arange(B, device=k.device)
        case.cache.append(0, k[bi, pos].contiguous(), v[bi, pos].contiguous(), case.ids[bi, pos].contiguous())
        lens = lens + 1
        q = case.q(0, int(lens.max()), step=step)
        o = case.cache.decode(0, q)
        case.cache.check()
        assert _max_err(o, case.expected(0, q, lens)) <= DECODE_TOL, step
        case.check_layout(0, lens)


def test_alignment_64_masks(cuda):
    # per-head kept counts rounded to multiples of 64 (the H100 setting of the
    # LeanK article's troubleshooting notes): widths 0, 64 and 128 only
    w = SERVING.scaled(num_layers=2, batch=2, context=900, tau=0.5)
    alpha = S.draw_alpha(w).astype(np.float32)
    masks = OM.top_s_prune(alpha, 60.0, align=64, budget="exact")
    counts = masks.sum(-1)
    assert set(np.unique(counts)) <= {0, 64, 128} and len(set(np.unique(counts))) >= 2
    case = Case(w, total=901, masks=masks)
    for layer in range(2):
        _decode_steps(case, layer, 900, 1, layout=True)


def test_device_status_bits_reach_the_host(cuda):
    # the kernels report a timed-out wait, a full layer and a bad token id
    # through sticky bits in the cache header; lk_check maps and clears them
    # (set here directly: no kernel is made to time out)
    case = Case(TINY, total=8)
    for bit, status in ((1, lkb.LK_ERR_TIMEOUT), (2, lkb.LK_ERR_CAPACITY), (4, lkb.LK_ERR_ARG)):
        case.cache.buffer[0:4].copy_(torch.tensor([bit], dtype=torch.int32).view(torch.uint8))
        with pytest.raises(lkb.LeankError) as e:
            case.cache.check()
        assert e.value.status == status
        case.cache.check()                   # cleared
    # the cache keeps working afterwards
    case.prefill(0, 8)
    q = case.q(0, 8)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 8)) <= DECODE_TOL


@pytest.mark.parametrize("hq,hkv", [(4, 4), (32, 4), (12, 4)], ids=["G1", "G8", "G3"])
@pytest.mark.parametrize("kv", [lkb.KV_BF16, lkb.KV_INT8, lkb.KV_FP8], ids=["bf16", "int8", "fp8"])
def test_query_group_sizes(cuda, hq, hkv, kv):
    # G = 1 (one query head per kv head), G = 8 (the largest group, all of the
    # mma's N) and an odd G = 3
    w = LLAMA.scaled(num_q_heads=hq, num_kv_heads=hkv, context=1700, batch=2)
    masks = S.masks_with_counts(w, [32, 0, 96, 128])
    case = Case(w, total=1701, masks=masks, kv_format=kv)
    case.prefill(0, 1700)
    case.append(0, 1700)
    q = case.q(0, 1701)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 1701)) <= DECODE_TOL


def test_step_layers_host_packed_matches_device_path(cuda):
    # every layer's step from one mapped pinned block (q of all layers | k |
    # v | ids): the append and decode launches of the device path, read and
    # written in place, so outputs and cache bytes are identical
    w = FASTGEN.scaled(num_layers=3, batch=2, context=500, policy_counts=(6, 4, 14))
    a = Case(w, total=502)
    b = Case(w, total=502)
    a.cache.set_step_mode(lkb.STEP_SPLIT)
    L, N = w.num_layers, 500
    for case in (a, b):
        for layer in range(L):
            case.prefill(layer, N)
    qs = torch.stack([a.q(layer, N + 1) for layer in range(L)]).contiguous()
    ks = torch.stack([a.history(layer)[0][:, N] for layer in range(L)]).contiguous()
    vs = torch.stack([a.history(layer)[1][:, N] for layer in range(L)]).contiguous()
    ids = a.ids[:, N].contiguous()
    o_dev = a.cache.step_layers(0, qs, ks, vs, ids)
    blk = torch.cat([t.cpu().contiguous().view(torch.uint8).reshape(-1) for t in (qs, ks, vs, ids)]).pin_memory()
    o_host = torch.empty(o_dev.shape, dtype=torch.float32).pin_memory()
    b.cache.step_layers_host_packed(0, L, blk, True, o_host)
    torch.cuda.synchronize()
    b.cache.check()
    assert torch.equal(o_host, o_dev.cpu())
    for layer in range(L):
        assert float(np.abs(o_host[layer].double().numpy() - a.expected(layer, qs[layer], N + 1)).max()) <= DECODE_TOL
    assert torch.equal(a.cache.buffer, b.cache.buffer)
    # pageable buffers are refused before anything is launched
    with pytest.raises(lkb.LeankError) as e:
        b.cache.step_layers_host_packed(0, L, blk.clone(), True, torch.empty_like(o_host))
    assert e.value.status == lkb.LK_ERR_ARG
    assert list(b.cache.lengths(0)) == [N + 1, N + 1]


def test_bounded_wait_runs_out_and_the_cache_recovers(cuda):
    # Failure path of the decode kernel, with no fault: a wait limit of 0
    # makes every ring and segment wait that is not already complete run out
    # (a CTA of 4 streams ~40 tiles through a ring of 3 to 5 stages, so the
    # producer's first slot wait finds its oldest stage still in use).  The
    # launch records LK_ERR_TIMEOUT; the producer still waits (bounded) for
    # its own copies to land before its CTA exits.  With the limit back and
    # the workspace zeroed, the next decode matches the oracle.
    w = LLAMA.scaled(context=3000, batch=2)
    masks = S.masks_with_counts(w, [32, 64, 0, 96, 128, 32, 32, 64])
    case = Case(w, total=3000, masks=masks)
    case.prefill(0, 3000)
    case.cache.set_decode_ctas(4)
    q = case.q(0, 3000)
    case.cache.set_wait_limit(0)
    case.cache.decode(0, q)
    with pytest.raises(lkb.LeankError) as e:
        case.cache.check()
    assert e.value.status == lkb.LK_ERR_TIMEOUT
    case.cache.check()                        # the status word was cleared
    case.cache.set_wait_limit(10 ** 9)
    case.cache.workspace_init()
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, 3000)) <= DECODE_TOL
    with pytest.raises(lkb.LeankError) as e:
        case.cache.set_wait_limit(11 * 10 ** 9)
    assert e.value.status == lkb.LK_ERR_ARG


def test_host_step_is_refused_before_the_append(cuda):
    # a workspace too small for the decode is refused before the append, so
    # no token is committed (lengths and cache bytes unchanged)
    import ctypes
    w = FASTGEN.scaled(num_layers=2, batch=2, context=300, policy_counts=(1, 1, 14))
    case = Case(w, total=301)
    L, N = w.num_layers, 300
    for layer in range(L):
        case.prefill(layer, N)
    qs = torch.stack([case.q(layer, N + 1) for layer in range(L)]).contiguous()
    ks = torch.stack([case.history(layer)[0][:, N] for layer in range(L)]).contiguous()
    vs = torch.stack([case.history(layer)[1][:, N] for layer in range(L)]).contiguous()
    ids = case.ids[:, N].contiguous()
    blk = torch.cat([t.cpu().contiguous().view(torch.uint8).reshape(-1) for t in (qs, ks, vs, ids)]).pin_memory()
    o_host = torch.empty((L, w.batch, w.num_q_heads, 128), dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    before = case.cache.buffer.clone()
    lib = lkb.load()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.lk_step_layers_host_packed(case.cache._h, 0, L, blk.data_ptr(), 1, o_host.data_ptr(),
                                        case.cache.workspace.data_ptr(), 256, s)
    assert st == lkb.LK_ERR_CAPACITY
    # one layer from mapped host buffers, with a misaligned o
    o1 = torch.empty(w.batch * w.num_q_heads * 128 + 4, dtype=torch.float32).pin_memory()
    st = lib.lk_step_host_packed(case.cache._h, 0, blk.data_ptr(), 0, o1.data_ptr() + 4,
                                 case.cache.workspace.data_ptr(), case.cache.workspace.numel(), s)
    assert st == lkb.LK_ERR_ALIGN
    torch.cuda.synchronize()
    case.cache.check()
    for layer in range(L):
        assert list(case.cache.lengths(layer)) == [N] * w.batch
    assert torch.equal(case.cache.buffer, before)
