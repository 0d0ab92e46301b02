"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and the host-only calls validate their arguments."""
import ctypes
import os
import re

import numpy as np
import pytest

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from helpers import workload_masks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "leank.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lk_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lkb.SIGNATURES), set(names) ^ set(lkb.SIGNATURES)


def _plan(masks, policies=None, **kw):
    L, H, _ = masks.shape
    args = dict(num_layers=L, num_q_heads=4 * H, num_kv_heads=H, sink=4, local=16)
    args.update(kw)
    return lkb.Plan(args.pop("num_layers"), args.pop("num_q_heads"), args.pop("num_kv_heads"),
                    args.pop("sink"), args.pop("local"), masks, policies, **args)


def test_plan_rejects_unaligned_mask_count(lib):
    m = np.zeros((1, 2, 128), dtype=np.uint8)
    m[0, 0, :33] = 1
    with pytest.raises(lkb.LeankError) as e:
        _plan(m)
    assert e.value.status == lkb.LK_ERR_ARG
    assert "multiple of 32" in str(e.value)


def test_plan_rejects_bad_values(lib):
    m = np.ones((1, 2, 128), dtype=np.uint8)
    m2 = m.copy(); m2[0, 1, 5] = 2
    with pytest.raises(lkb.LeankError) as e:
        _plan(m2)
    assert e.value.status == lkb.LK_ERR_ARG
    with pytest.raises(lkb.LeankError) as e:
        _plan(m, policies=np.array([[0, 7]], dtype=np.int32))
    assert e.value.status == lkb.LK_ERR_ARG
    with pytest.raises(lkb.LeankError) as e:                 # SPECIAL without a table
        _plan(m, policies=np.array([[0, 2]], dtype=np.int32))
    assert e.value.status == lkb.LK_ERR_ARG
    with pytest.raises(lkb.LeankError) as e:                 # LOCAL without a window
        _plan(m, policies=np.array([[1, 0]], dtype=np.int32))
    assert e.value.status == lkb.LK_ERR_ARG
    with pytest.raises(lkb.LeankError) as e:
        _plan(m, num_q_heads=5)
    assert e.value.status == lkb.LK_ERR_ARG


def test_plan_rejects_unsupported_shapes(lib):
    m = np.ones((1, 2, 128), dtype=np.uint8)
    with pytest.raises(lkb.LeankError) as e:
        _plan(m, num_q_heads=18)                              # G = 9 > 8
    assert e.value.status == lkb.LK_ERR_UNSUPPORTED
    desc = lkb.PlanDesc(1, 2, 2, 64, 4, 16, 0, 0, 0)
    h = ctypes.c_void_p()
    pol = np.zeros((1, 2), np.int32)
    st = lib.lk_build_plan(ctypes.byref(desc), np.ones((1, 2, 64), np.uint8).ctypes.data, pol.ctypes.data,
                           None, ctypes.byref(h))
    assert st == lkb.LK_ERR_UNSUPPORTED
    st = lib.lk_build_plan(None, None, None, None, ctypes.byref(h))
    assert st == lkb.LK_ERR_ARG
    assert b"null" in lib.lk_last_error()


def test_plan_groups_heads_and_orders_kept_channels(lib):
    w = S.WORKLOADS[2]
    pol = S.make_policies(w)
    masks = workload_masks(w, pol)
    plan = lkb.Plan.for_workload(w, masks, pol)
    for l, h in [(0, 0), (3, 5), (31, 7)]:
        p, k, kept = plan.head(l, h)
        assert p == S.POLICY_FULL
        assert k == int(masks[l, h].sum())
        assert np.array_equal(kept, np.nonzero(masks[l, h])[0])


def test_cache_bytes_grow_with_capacity_and_width(lib):
    w = S.WORKLOADS[1]
    m32 = S.masks_with_counts(w, [32] * 8)
    m128 = S.masks_with_counts(w, [128] * 8)
    m0 = S.masks_with_counts(w, [0] * 8)
    sizes = {}
    for name, m in [("k0", m0), ("k32", m32), ("k128", m128)]:
        plan = lkb.Plan.for_workload(w, m, S.make_policies(w))
        sizes[name] = plan.cache_bytes(1, 32768)
        assert plan.cache_bytes(1, 40000) > sizes[name] or name == "k0"
    # dense K+V of 8 heads x 32768 tokens is 128 MiB; the k=128 layout holds it
    dense = 2 * 8 * 32768 * 128 * 2
    assert dense <= sizes["k128"] < dense + (4 << 20)
    mid = 32768 - 16 - 1024
    # (less the 128-row minimum every pool keeps for its tensor map box)
    assert sizes["k32"] - sizes["k0"] >= 8 * mid * (32 + 128) * 2 - 128 * 32 * 2
    assert sizes["k0"] < 8 * (16 + 1024) * 512 + (8 << 20)
    with pytest.raises(lkb.LeankError):
        plan.cache_bytes(0, 10)
    with pytest.raises(lkb.LeankError):
        plan.cache_bytes(1, 0)


def test_workspace_bytes(lib):
    w = S.WORKLOADS[3]
    plan = lkb.Plan.for_workload(w, workload_masks(w), S.make_policies(w))
    n = plan.workspace_bytes(w.batch)
    E, G = w.batch * w.num_kv_heads, w.group
    assert n >= (256 + E) * G * 128 * 4


def test_cache_init_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    w = S.WORKLOADS[0]
    plan = lkb.Plan.for_workload(w, workload_masks(w), S.make_policies(w))
    buf = np.zeros(plan.cache_bytes(1, 64) + 256, dtype=np.uint8)
    addr = (buf.ctypes.data + 255) // 256 * 256
    h = ctypes.c_void_p()
    st = lib.lk_cache_init(plan._h, addr, plan.cache_bytes(1, 64), 1, 64, None, ctypes.byref(h))
    assert st in (lkb.LK_ERR_CUDA,)
    assert h.value is None
    st = lib.lk_cache_init(plan._h, addr + 8, 1 << 20, 1, 64, None, ctypes.byref(h))
    assert st == lkb.LK_ERR_ALIGN


def test_paged_cache_bytes(lib):
    w = S.WORKLOADS[1]
    plan = lkb.Plan.for_workload(w, S.masks_with_counts(w, [32] * 8), S.make_policies(w))
    B, cap = 4, 32768
    mid = cap - w.sink - w.local
    contiguous = plan.cache_bytes(B, cap)
    # room for every sequence's whole middle: the contiguous size plus the
    # rounding of each sequence's last page and the page tables
    full = plan.cache_bytes(B, cap, middle_tokens=B * mid)
    assert contiguous <= full <= contiguous + (1 << 20)
    # a quarter of that: about a quarter of the middle bytes
    small = plan.cache_bytes(B, cap, middle_tokens=mid)
    middle_bytes = 8 * B * mid * (32 + 128) * 2
    assert abs((contiguous - small) - 0.75 * middle_bytes) < 0.01 * middle_bytes
    assert plan.cache_bytes(B, cap, middle_tokens=0) < contiguous - middle_bytes + (8 << 20)
    with pytest.raises(lkb.LeankError) as e:
        plan.cache_bytes(B, cap, middle_tokens=-1)
    assert e.value.status == lkb.LK_ERR_ARG


def test_int8_cache_bytes(lib):
    w = S.WORKLOADS[1]
    plan = lkb.Plan.for_workload(w, S.masks_with_counts(w, [32] * 8), S.make_policies(w))
    B, cap = 2, 32768
    mid = cap - w.sink - w.local
    bf16 = plan.cache_bytes(B, cap)
    q8 = plan.cache_bytes(B, cap, kv_format=lkb.KV_INT8)
    # middle rows: 320 B in bf16, 165 B per row in sealed blocks (+ a 128-row bf16 tail)
    blocks = mid // 128
    expect = bf16 - 8 * B * mid * 320 + 8 * B * (blocks * 132 * 160 + 128 * 320)
    assert abs(q8 - expect) < (1 << 20)
    paged = plan.cache_bytes(B, cap, middle_tokens=B * mid, kv_format=lkb.KV_INT8)
    assert abs(paged - q8) < (1 << 20)
    with pytest.raises(lkb.LeankError) as e:
        plan.cache_bytes(B, cap, kv_format=7)
    assert e.value.status == lkb.LK_ERR_ARG


_LAYOUT_PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "leank.h"
#define SIZE(T) printf(#T " %zu\n", sizeof(T));
#define OFF(T, m) printf(#T "." #m " %zu\n", offsetof(T, m));
#define VAL(e) printf(#e " %d\n", (int)(e));
int main(void) {
  SIZE(lk_plan_desc) SIZE(lk_region_info) SIZE(lk_cache_options)
  OFF(lk_plan_desc, num_layers) OFF(lk_plan_desc, num_q_heads) OFF(lk_plan_desc, num_kv_heads)
  OFF(lk_plan_desc, head_dim) OFF(lk_plan_desc, sink) OFF(lk_plan_desc, local)
  OFF(lk_plan_desc, local_only_window) OFF(lk_plan_desc, vocab) OFF(lk_plan_desc, special_capacity)
  OFF(lk_region_info, policy) OFF(lk_region_info, n_kept) OFF(lk_region_info, rows_a)
  OFF(lk_region_info, rows_b) OFF(lk_region_info, k_a_offset) OFF(lk_region_info, v_a_offset)
  OFF(lk_region_info, k_b_offset) OFF(lk_region_info, v_b_offset) OFF(lk_region_info, page_rows)
  OFF(lk_region_info, max_pages) OFF(lk_region_info, page_table_offset) OFF(lk_region_info, kv_format)
  OFF(lk_region_info, sealed_blocks)
  OFF(lk_cache_options, middle_tokens) OFF(lk_cache_options, kv_format) OFF(lk_cache_options, reserved)
  VAL(LK_OK) VAL(LK_ERR_ARG) VAL(LK_ERR_ALIGN) VAL(LK_ERR_CAPACITY) VAL(LK_ERR_STATE) VAL(LK_ERR_CUDA)
  VAL(LK_ERR_TIMEOUT) VAL(LK_ERR_UNSUPPORTED)
  VAL(LK_POLICY_FULL) VAL(LK_POLICY_LOCAL) VAL(LK_POLICY_SPECIAL)
  VAL(LK_KV_BF16) VAL(LK_KV_INT8) VAL(LK_KV_FP8)
  VAL(LK_STEP_AUTO) VAL(LK_STEP_FUSED) VAL(LK_STEP_SPLIT)
  return 0;
}
"""


def test_header_compiles_as_c_and_cxx_and_matches_the_binding(tmp_path):
    """The public header stands alone in C99 and C++17 with every warning an
    error, and the binding's structures and constants have the header's
    sizes, field offsets and values (a mismatch would pass garbage through
    ctypes without an error)."""
    import shutil
    import subprocess
    gcc, gxx = shutil.which("gcc"), shutil.which("g++")
    if gcc is None or gxx is None:
        pytest.skip("no host C / C++ compiler")
    inc = os.path.join(ROOT, "include")
    src = tmp_path / "layout.c"
    src.write_text(_LAYOUT_PROBE)
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src), "-o", str(exe)],
                   check=True)
    cxx = tmp_path / "header.cc"
    cxx.write_text('#include "leank.h"\nint main() { return LK_OK; }\n')
    subprocess.run([gxx, "-std=c++17", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I", inc,
                    str(cxx)], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                              text=True).stdout.splitlines())
    got = {k: int(v) for k, v in got.items()}
    structs = {"lk_plan_desc": lkb.PlanDesc, "lk_region_info": lkb.RegionInfo,
               "lk_cache_options": lkb.CacheOptions}
    for cname, ct in structs.items():
        assert ctypes.sizeof(ct) == got[cname], cname
        for field, _ in ct._fields_:
            assert getattr(ct, field).offset == got[f"{cname}.{field}"], (cname, field)
    assert len([k for k in got if "." in k]) == sum(len(ct._fields_) for ct in structs.values())
    for i, name in enumerate(lkb.STATUS_NAMES):
        assert got[name] == i
    assert (got["LK_POLICY_FULL"], got["LK_POLICY_LOCAL"], got["LK_POLICY_SPECIAL"]) == \
        (lkb.POLICY_FULL, lkb.POLICY_LOCAL, lkb.POLICY_SPECIAL)
    assert (got["LK_KV_BF16"], got["LK_KV_INT8"], got["LK_KV_FP8"]) == (lkb.KV_BF16, lkb.KV_INT8, lkb.KV_FP8)
    assert (got["LK_STEP_AUTO"], got["LK_STEP_FUSED"], got["LK_STEP_SPLIT"]) == \
        (lkb.STEP_AUTO, lkb.STEP_FUSED, lkb.STEP_SPLIT)
