"""The decode entry point that allocates nothing (lk_decode_attn_static).

It exists for callers that cannot call cudaMalloc themselves, such as a
plugin inside a host runtime that owns the device allocator, or a loop where
an allocation would synchronise the device: they still pass q and o, and the
split scratch comes from an array built into the library.  This file runs
last so that a failure here never hides the other tests; it passes alone in a
fresh process as well as after them.
"""
import ctypes

import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from helpers import DECODE_TOL, Case

pytestmark = pytest.mark.gpu


def test_static_scratch_first_call_on_a_side_stream_and_a_later_layer(cuda):
    # Kept first in this file, so that in a run of the whole suite (and in a
    # fresh process) it makes the process's first call of this entry point:
    # on a non-blocking stream (nothing orders it after work on the legacy
    # default stream) and on layer 1 of a two-layer cache (entries and split
    # slots of a launch count from its first layer).  Two calls in a row.
    w = S.WORKLOADS[2].scaled(num_layers=2, batch=3, context=900)
    case = Case(w, total=902)
    for layer in range(2):
        case.prefill(layer, 900)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    for t in (900, 901):
        for layer in range(2):
            case.append(layer, t)
        q = case.q(1, t + 1, step=t)
        o_ws = case.cache.decode(1, q)
        torch.cuda.synchronize()
        o_st = torch.full_like(o_ws, float("nan"))
        with torch.cuda.stream(side):
            case.cache.decode_static(1, q, o_st, stream=side)
        side.synchronize()
        case.cache.check(stream=side)
        err = float((o_st.double() - o_ws.double()).abs().max())
        assert err <= DECODE_TOL, err
        ref = case.expected(1, q, t + 1)
        assert float(np.abs(o_st.double().cpu().numpy() - ref).max()) <= DECODE_TOL


def test_static_scratch_matches_workspace_path_twice(cuda):
    w = S.WORKLOADS[1].scaled(context=2600, batch=2)
    masks = S.masks_with_counts(w, [0, 32, 64, 96, 128, 32, 0, 64])
    case = Case(w, total=2602, masks=masks)
    case.prefill(0, 2600)
    lib = lkb.load()
    for t in (2600, 2601):                   # two calls in a row, the cache growing
        case.append(0, t)
        q = case.q(0, t + 1, step=t)
        o_ws = case.cache.decode(0, q)
        o_st = torch.full_like(o_ws, float("nan"))
        st = lib.lk_decode_attn_static(case.cache._h, 0, q.data_ptr(), o_st.data_ptr(),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == lkb.LK_OK, lib.lk_last_error()
        case.cache.check()
        err = float((o_st.double() - o_ws.double()).abs().max())
        assert err <= DECODE_TOL, err
        ref = case.expected(0, q, t + 1)
        assert float(np.abs(o_st.double().cpu().numpy() - ref).max()) <= DECODE_TOL


def test_static_scratch_rejects_caches_beyond_its_size(cuda):
    w = S.WORKLOADS[2].scaled(num_layers=1, batch=2048, context=8)
    case = Case(w, total=8)
    o = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device=cuda)
    q = torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.bfloat16, device=cuda)
    with pytest.raises(lkb.LeankError) as e:
        case.cache.decode_static(0, q, o)
    assert e.value.status == lkb.LK_ERR_CAPACITY


@pytest.mark.parametrize("kv,paged", [(lkb.KV_BF16, True), (lkb.KV_INT8, False), (lkb.KV_FP8, True)],
                         ids=["bf16-paged", "int8", "fp8-paged"])
def test_static_scratch_on_paged_and_quantized_caches(cuda, kv, paged):
    # the same launch as lk_decode_attn over the other cache layouts: region B
    # through the page table, and sealed INT8 / FP8 blocks beside a bf16 tail
    w = S.WORKLOADS[1].scaled(context=1500, batch=2)
    masks = S.masks_with_counts(w, [32, 0, 64, 128, 96, 32, 64, 0])
    case = Case(w, total=1501, masks=masks, kv_format=kv, middle_tokens=2 * 1501 if paged else None)
    case.prefill(0, 1500)
    case.append(0, 1500)
    q = case.q(0, 1501, step=1500)
    o_ws = case.cache.decode(0, q)
    o_st = torch.full_like(o_ws, float("nan"))
    case.cache.decode_static(0, q, o_st)
    case.cache.check()
    assert torch.equal(o_st, o_ws)
    ref = case.expected(0, q, 1501)
    assert float(np.abs(o_st.double().cpu().numpy() - ref).max()) <= DECODE_TOL
