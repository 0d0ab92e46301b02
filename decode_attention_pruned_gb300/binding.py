"""Thin Python binding of the C ABI in include/leank.h (ctypes).

Argument marshalling only: torch tensors are passed as raw device pointers
and the current CUDA stream as a handle.  Every step of prefill, append and
decode runs in the library's CUDA kernels; there is no CPU path, and a
missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libleank.so")

LK_OK, LK_ERR_ARG, LK_ERR_ALIGN, LK_ERR_CAPACITY, LK_ERR_STATE, LK_ERR_CUDA, LK_ERR_TIMEOUT, \
    LK_ERR_UNSUPPORTED = range(8)
STATUS_NAMES = ["LK_OK", "LK_ERR_ARG", "LK_ERR_ALIGN", "LK_ERR_CAPACITY", "LK_ERR_STATE", "LK_ERR_CUDA",
                "LK_ERR_TIMEOUT", "LK_ERR_UNSUPPORTED"]
POLICY_FULL, POLICY_LOCAL, POLICY_SPECIAL = 0, 1, 2

# Every symbol include/leank.h declares, with (restype, argtypes).
_vp, _i32, _sz, _u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_uint64


class PlanDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "num_q_heads", "num_kv_heads", "head_dim", "sink", "local",
        "local_only_window", "vocab", "special_capacity")]


class RegionInfo(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int32), ("n_kept", ctypes.c_int32), ("rows_a", ctypes.c_int32),
                ("rows_b", ctypes.c_int32), ("k_a_offset", ctypes.c_uint64), ("v_a_offset", ctypes.c_uint64),
                ("k_b_offset", ctypes.c_uint64), ("v_b_offset", ctypes.c_uint64),
                ("page_rows", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("page_table_offset", ctypes.c_uint64), ("kv_format", ctypes.c_int32),
                ("sealed_blocks", ctypes.c_int32)]


KV_BF16, KV_INT8, KV_FP8 = 0, 1, 2
KV_FORMAT_NAMES = {KV_BF16: "bf16", KV_INT8: "int8", KV_FP8: "fp8"}
STEP_AUTO, STEP_FUSED, STEP_SPLIT = 0, 1, 2


class CacheOptions(ctypes.Structure):
    _fields_ = [("middle_tokens", ctypes.c_int64), ("kv_format", ctypes.c_int32), ("reserved", ctypes.c_int32)]


SIGNATURES = {
    "lk_build_plan": (ctypes.c_int, [ctypes.POINTER(PlanDesc), _vp, _vp, _vp, ctypes.POINTER(_vp)]),
    "lk_plan_destroy": (None, [_vp]),
    "lk_build_masks": (ctypes.c_int, [_vp, _vp, _i32, _i32, ctypes.c_double, _i32, _i32, _vp, _vp]),
    "lk_plan_head": (ctypes.c_int, [_vp, _i32, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32), _vp]),
    "lk_cache_bytes": (ctypes.c_int, [_vp, _i32, _i32, ctypes.POINTER(_sz)]),
    "lk_cache_bytes_paged": (ctypes.c_int, [_vp, _i32, _i32, ctypes.c_int64, ctypes.POINTER(_sz)]),
    "lk_workspace_bytes": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(_sz)]),
    "lk_cache_init": (ctypes.c_int, [_vp, _vp, _sz, _i32, _i32, _vp, ctypes.POINTER(_vp)]),
    "lk_cache_init_paged": (ctypes.c_int, [_vp, _vp, _sz, _i32, _i32, ctypes.c_int64, _vp, ctypes.POINTER(_vp)]),
    "lk_cache_bytes_ex": (ctypes.c_int, [_vp, _i32, _i32, ctypes.POINTER(CacheOptions), ctypes.POINTER(_sz)]),
    "lk_cache_init_ex": (ctypes.c_int, [_vp, _vp, _sz, _i32, _i32, ctypes.POINTER(CacheOptions), _vp,
                                        ctypes.POINTER(_vp)]),
    "lk_cache_block": (ctypes.c_int, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "lk_cache_destroy": (None, [_vp]),
    "lk_workspace_init": (ctypes.c_int, [_vp, _vp, _sz, _vp]),
    "lk_prefill": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _i32, _vp]),
    "lk_prefill_ragged": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp]),
    "lk_prefill_sequence": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _i32, _vp]),
    "lk_release_sequence": (ctypes.c_int, [_vp, _i32, _vp]),
    "lk_cache_pages": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "lk_append": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp]),
    "lk_append_layers": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp]),
    "lk_decode_attn": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "lk_decode_attn_layers": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "lk_step": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lk_set_step_mode": (ctypes.c_int, [_vp, _i32]),
    "lk_step_is_fused": (ctypes.c_int, [_vp, _i32, _i32, ctypes.POINTER(_i32)]),
    "lk_step_layers": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lk_decode_attn_static": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp]),
    "lk_step_host": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lk_step_host_packed": (ctypes.c_int, [_vp, _i32, _vp, _i32, _vp, _vp, _sz, _vp]),
    "lk_step_layers_host_packed": (ctypes.c_int, [_vp, _i32, _i32, _vp, _i32, _vp, _vp, _sz, _vp]),
    "lk_cache_length": (ctypes.c_int, [_vp, _i32, ctypes.POINTER(_i32)]),
    "lk_cache_lengths": (ctypes.c_int, [_vp, _i32, _vp]),
    "lk_cache_region": (ctypes.c_int, [_vp, _i32, _i32, _i32, ctypes.POINTER(RegionInfo)]),
    "lk_resident_bytes": (ctypes.c_int, [_vp, _i32, _vp, ctypes.POINTER(_u64)]),
    "lk_set_decode_ctas": (ctypes.c_int, [_vp, _i32]),
    "lk_set_wait_limit": (ctypes.c_int, [_vp, _u64]),
    "lk_check": (ctypes.c_int, [_vp, _vp]),
    "lk_last_error": (ctypes.c_char_p, []),
}

_lib = None


class LeankError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{name}: {message}")


def load(build_if_missing: bool = False):
    """Load libleank.so (raises if it is missing and not built here)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        if not build_if_missing:
            raise RuntimeError(f"libleank.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        from . import build as _build
        _build.build()
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != LK_OK:
        raise LeankError(status, _lib.lk_last_error().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, shape, what, device_kind="cuda"):
    try:
        if t.dtype is dtype and t.shape == shape and t.device.type == device_kind and t.is_contiguous():
            return
    except AttributeError:
        raise TypeError(f"{what} must be a torch tensor") from None
    raise ValueError(f"{what}: expected contiguous {dtype} {tuple(shape)} on {device_kind}, got "
                     f"{t.dtype} {tuple(t.shape)} on {t.device.type}")


def build_masks(alpha, prune_pct, align=32, exact=False, eligible=None, stream=None):
    """lk_build_masks: alpha device fp32 [L, Hkv, 128] -> device uint8 masks."""
    import torch
    load()
    L, H = alpha.shape[0], alpha.shape[1]
    _need(alpha, torch.float32, (L, H, 128), "alpha")
    if eligible is not None:
        _need(eligible, torch.uint8, (L, H), "eligible")
    out = torch.empty((L, H, 128), dtype=torch.uint8, device=alpha.device)
    _check(_lib.lk_build_masks(alpha.data_ptr(), _ptr(eligible), L, H, float(prune_pct), align, 1 if exact else 0,
                               out.data_ptr(), _stream(stream)))
    return out


class Plan:
    """lk_build_plan: masks [L, Hkv, 128] uint8, policies [L, Hkv] int32."""

    def __init__(self, num_layers, num_q_heads, num_kv_heads, sink, local, masks, policies=None,
                 local_only_window=0, is_special=None, special_capacity=0, head_dim=128):
        lib = load()
        masks = np.ascontiguousarray(masks, dtype=np.uint8)
        if policies is None:
            policies = np.zeros((num_layers, num_kv_heads), dtype=np.int32)
        policies = np.ascontiguousarray(policies, dtype=np.int32)
        spec = None if is_special is None else np.ascontiguousarray(is_special, dtype=np.uint8)
        self.desc = PlanDesc(num_layers, num_q_heads, num_kv_heads, head_dim, sink, local,
                             local_only_window, 0 if spec is None else len(spec), special_capacity)
        if masks.shape != (num_layers, num_kv_heads, head_dim):
            raise ValueError(f"masks shape {masks.shape}")
        if policies.shape != (num_layers, num_kv_heads):
            raise ValueError(f"policies shape {policies.shape}")
        h = ctypes.c_void_p()
        _check(lib.lk_build_plan(ctypes.byref(self.desc), masks.ctypes.data, policies.ctypes.data,
                                 None if spec is None else spec.ctypes.data, ctypes.byref(h)))
        self._h = h
        self.num_layers, self.num_q_heads, self.num_kv_heads = num_layers, num_q_heads, num_kv_heads
        self.group = num_q_heads // num_kv_heads
        self.sink, self.local, self.local_only_window = sink, local, local_only_window

    @classmethod
    def for_workload(cls, w, masks, policies, is_special=None, special_capacity=0):
        return cls(w.num_layers, w.num_q_heads, w.num_kv_heads, w.sink, w.local, masks, policies,
                   local_only_window=w.local_only_window,
                   is_special=is_special if (is_special is not None and len(is_special)) else None,
                   special_capacity=special_capacity)

    def head(self, layer, kv_head):
        pol, nk = ctypes.c_int32(), ctypes.c_int32()
        kept = np.zeros(128, dtype=np.int16)
        _check(_lib.lk_plan_head(self._h, layer, kv_head, ctypes.byref(pol), ctypes.byref(nk), kept.ctypes.data))
        return pol.value, nk.value, kept[: nk.value].copy()

    def cache_bytes(self, batch, capacity, middle_tokens=None, kv_format=KV_BF16):
        """Cache buffer bytes; paged layout when middle_tokens is given."""
        n = ctypes.c_size_t()
        if kv_format != KV_BF16:
            opt = CacheOptions(-1 if middle_tokens is None else int(middle_tokens), kv_format, 0)
            _check(_lib.lk_cache_bytes_ex(self._h, batch, capacity, ctypes.byref(opt), ctypes.byref(n)))
        elif middle_tokens is None:
            _check(_lib.lk_cache_bytes(self._h, batch, capacity, ctypes.byref(n)))
        else:
            _check(_lib.lk_cache_bytes_paged(self._h, batch, capacity, int(middle_tokens), ctypes.byref(n)))
        return n.value

    def workspace_bytes(self, batch):
        n = ctypes.c_size_t()
        _check(_lib.lk_workspace_bytes(self._h, batch, ctypes.byref(n)))
        return n.value

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.lk_plan_destroy(self._h)
            self._h = None


class Cache:
    """A cache bound to a torch-allocated device buffer, plus its workspace.

    With ``middle_tokens`` the cache is paged (lk_cache_init_paged): the
    middle rows of all sequences share page pools sized for that many middle
    tokens in total.  ``kv_format=KV_INT8`` quantises complete 128-row
    blocks of the middle (lk_cache_init_ex); ``KV_FP8`` stores them as e4m3
    codes."""

    def __init__(self, plan: Plan, batch: int, capacity: int, device=None, stream=None, middle_tokens=None,
                 kv_format=KV_BF16):
        import torch
        self.plan, self.batch, self.capacity = plan, batch, capacity
        self.paged = middle_tokens is not None
        self.kv_format = kv_format
        dev = torch.device(device if device is not None else "cuda")
        self.device = dev
        nbytes = plan.cache_bytes(batch, capacity, middle_tokens, kv_format)
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.workspace = torch.empty(plan.workspace_bytes(batch), dtype=torch.uint8, device=dev)
        h = ctypes.c_void_p()
        s = _stream(stream)
        if kv_format != KV_BF16:
            opt = CacheOptions(-1 if middle_tokens is None else int(middle_tokens), kv_format, 0)
            _check(_lib.lk_cache_init_ex(plan._h, self.buffer.data_ptr(), nbytes, batch, capacity,
                                         ctypes.byref(opt), s, ctypes.byref(h)))
        elif self.paged:
            _check(_lib.lk_cache_init_paged(plan._h, self.buffer.data_ptr(), nbytes, batch, capacity,
                                            int(middle_tokens), s, ctypes.byref(h)))
        else:
            _check(_lib.lk_cache_init(plan._h, self.buffer.data_ptr(), nbytes, batch, capacity, s,
                                      ctypes.byref(h)))
        self._h = h
        _check(_lib.lk_workspace_init(self._h, self.workspace.data_ptr(), self.workspace.numel(), s))

    # -- the hot path
    def prefill(self, layer, k, v, ids=None, stream=None):
        import torch
        B, H = self.batch, self.plan.num_kv_heads
        n = k.shape[1]
        _need(k, torch.bfloat16, (B, n, H, 128), "k")
        _need(v, torch.bfloat16, (B, n, H, 128), "v")
        if ids is not None:
            _need(ids, torch.int32, (B, n), "ids")
        _check(_lib.lk_prefill(self._h, layer, k.data_ptr(), v.data_ptr(), _ptr(ids), n, _stream(stream)))

    def prefill_ragged(self, layer, k, v, lens, ids=None, stream=None):
        """lk_prefill_ragged: k, v [B, n_max, Hkv, 128]; lens: B host ints."""
        import torch
        B, H = self.batch, self.plan.num_kv_heads
        n = k.shape[1]
        _need(k, torch.bfloat16, (B, n, H, 128), "k")
        _need(v, torch.bfloat16, (B, n, H, 128), "v")
        if ids is not None:
            _need(ids, torch.int32, (B, n), "ids")
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        if lens.shape != (B,):
            raise ValueError(f"lens shape {lens.shape}")
        _check(_lib.lk_prefill_ragged(self._h, layer, k.data_ptr(), v.data_ptr(), _ptr(ids), lens.ctypes.data, n,
                                      _stream(stream)))

    def prefill_sequence(self, layer, b, k, v, ids=None, stream=None):
        """lk_prefill_sequence: k, v [n, Hkv, 128] bf16 into empty slot b."""
        import torch
        H = self.plan.num_kv_heads
        n = k.shape[0]
        _need(k, torch.bfloat16, (n, H, 128), "k")
        _need(v, torch.bfloat16, (n, H, 128), "v")
        if ids is not None:
            _need(ids, torch.int32, (n,), "ids")
        _check(_lib.lk_prefill_sequence(self._h, layer, b, k.data_ptr() if n else None, v.data_ptr() if n else None,
                                        _ptr(ids) if n else None, n, _stream(stream)))

    def release(self, b, stream=None):
        """lk_release_sequence: empty slot b in every layer."""
        _check(_lib.lk_release_sequence(self._h, b, _stream(stream)))

    def pages(self, width):
        """(total, free) pages of a width class of a paged cache."""
        total, free = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.lk_cache_pages(self._h, width, ctypes.byref(total), ctypes.byref(free)))
        return total.value, free.value

    def page_table(self, r: RegionInfo):
        """The int32 page-table row of a paged head (a view of the buffer)."""
        import torch
        o = r.page_table_offset
        return self.buffer[o: o + 4 * r.max_pages].view(torch.int32)

    def middle_rows(self, r: RegionInfo, width_offset, width, m):
        """Rows of middle positions m (int64 tensor) of region B: K (width_offset
        = r.k_b_offset, width = n_kept) or V (r.v_b_offset, 128)."""
        import torch
        if r.page_rows == 0:
            return self.rows(width_offset, r.rows_b, width)[m]
        pt = self.page_table(r).to(torch.int64)
        rows = pt[m // r.page_rows] * r.page_rows + m % r.page_rows
        return self.rows(width_offset, r.rows_b, width)[rows]

    def block(self, layer, b, kv_head, j, stream=None):
        """lk_cache_block: (k_codes [128, k], k_scales [k], v_codes [128, 128],
        v_scales [128]) of sealed block j, logical order; codes int8 (INT8)
        or uint8 e4m3 bit patterns (FP8)."""
        k = self.plan.head(layer, kv_head)[1]
        kc = np.zeros((128, k), np.int8)
        ks = np.zeros(k, np.float32)
        vc = np.zeros((128, 128), np.int8)
        vs = np.zeros(128, np.float32)
        _check(_lib.lk_cache_block(self._h, layer, b, kv_head, j, kc.ctypes.data, ks.ctypes.data, vc.ctypes.data,
                                   vs.ctypes.data, _stream(stream)))
        if self.kv_format == KV_FP8:
            kc, vc = kc.view(np.uint8), vc.view(np.uint8)
        return kc, ks, vc, vs

    def lengths(self, layer):
        out = np.zeros(self.batch, dtype=np.int32)
        _check(_lib.lk_cache_lengths(self._h, layer, out.ctypes.data))
        return out

    def append_layers(self, layer0, k, v, ids=None, stream=None):
        """lk_append_layers: k, v [nlayers, B, Hkv, 128] bf16 (one token, every layer)."""
        import torch
        nl = k.shape[0]
        B, H = self.batch, self.plan.num_kv_heads
        _need(k, torch.bfloat16, (nl, B, H, 128), "k")
        _need(v, torch.bfloat16, (nl, B, H, 128), "v")
        if ids is not None:
            _need(ids, torch.int32, (B,), "ids")
        _check(_lib.lk_append_layers(self._h, layer0, nl, k.data_ptr(), v.data_ptr(), _ptr(ids), _stream(stream)))

    def decode_layers(self, layer0, q, o=None, stream=None):
        """lk_decode_attn_layers: q [nlayers, B, Hq, 128] bf16 -> o fp32."""
        import torch
        nl = q.shape[0]
        B, Hq = self.batch, self.plan.num_q_heads
        _need(q, torch.bfloat16, (nl, B, Hq, 128), "q")
        if o is None:
            o = torch.empty((nl, B, Hq, 128), dtype=torch.float32, device=q.device)
        _need(o, torch.float32, (nl, B, Hq, 128), "o")
        _check(_lib.lk_decode_attn_layers(self._h, layer0, nl, q.data_ptr(), o.data_ptr(), self.workspace.data_ptr(),
                                          self.workspace.numel(), _stream(stream)))
        return o

    def append(self, layer, k, v, ids=None, stream=None):
        import torch
        B, H = self.batch, self.plan.num_kv_heads
        _need(k, torch.bfloat16, (B, H, 128), "k")
        _need(v, torch.bfloat16, (B, H, 128), "v")
        if ids is not None:
            _need(ids, torch.int32, (B,), "ids")
        _check(_lib.lk_append(self._h, layer, k.data_ptr(), v.data_ptr(), _ptr(ids), _stream(stream)))

    def decode(self, layer, q, o=None, stream=None):
        import torch
        B, Hq = self.batch, self.plan.num_q_heads
        _need(q, torch.bfloat16, (B, Hq, 128), "q")
        if o is None:
            o = torch.empty((B, Hq, 128), dtype=torch.float32, device=q.device)
        _need(o, torch.float32, (B, Hq, 128), "o")
        _check(_lib.lk_decode_attn(self._h, layer, q.data_ptr(), o.data_ptr(), self.workspace.data_ptr(),
                                   self.workspace.numel(), _stream(stream)))
        return o

    def set_step_mode(self, mode):
        """lk_set_step_mode: STEP_AUTO, STEP_FUSED or STEP_SPLIT."""
        _check(_lib.lk_set_step_mode(self._h, mode))

    def step_is_fused(self, layer0=0, nlayers=1):
        f = _i32(0)
        _check(_lib.lk_step_is_fused(self._h, layer0, nlayers, ctypes.byref(f)))
        return bool(f.value)

    def step(self, layer, q, k, v, ids=None, o=None, stream=None):
        """lk_step: append k, v (ids) to `layer`, then attend with q, in one
        launch for a bf16 middle.  q [B, Hq, 128] bf16 -> o fp32."""
        import torch
        B, Hq, H = self.batch, self.plan.num_q_heads, self.plan.num_kv_heads
        _need(q, torch.bfloat16, (B, Hq, 128), "q")
        _need(k, torch.bfloat16, (B, H, 128), "k")
        _need(v, torch.bfloat16, (B, H, 128), "v")
        if ids is not None:
            _need(ids, torch.int32, (B,), "ids")
        if o is None:
            o = torch.empty((B, Hq, 128), dtype=torch.float32, device=q.device)
        _need(o, torch.float32, (B, Hq, 128), "o")
        _check(_lib.lk_step(self._h, layer, q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(ids), o.data_ptr(),
                            self.workspace.data_ptr(), self.workspace.numel(), _stream(stream)))
        return o

    def step_layers(self, layer0, q, k, v, ids=None, o=None, stream=None):
        """lk_step_layers: q [nlayers, B, Hq, 128], k, v [nlayers, B, Hkv, 128]."""
        import torch
        nl = q.shape[0]
        B, Hq, H = self.batch, self.plan.num_q_heads, self.plan.num_kv_heads
        _need(q, torch.bfloat16, (nl, B, Hq, 128), "q")
        _need(k, torch.bfloat16, (nl, B, H, 128), "k")
        _need(v, torch.bfloat16, (nl, B, H, 128), "v")
        if ids is not None:
            _need(ids, torch.int32, (B,), "ids")
        if o is None:
            o = torch.empty((nl, B, Hq, 128), dtype=torch.float32, device=q.device)
        _need(o, torch.float32, (nl, B, Hq, 128), "o")
        _check(_lib.lk_step_layers(self._h, layer0, nl, q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(ids),
                                   o.data_ptr(), self.workspace.data_ptr(), self.workspace.numel(),
                                   _stream(stream)))
        return o

    def decode_static(self, layer, q, o, stream=None):
        """lk_decode_attn_static: decode with the library's built-in split
        scratch instead of this cache's workspace (no allocation in the call;
        `o` must be given).  Calls must not overlap on the GPU."""
        import torch
        B, Hq = self.batch, self.plan.num_q_heads
        _need(q, torch.bfloat16, (B, Hq, 128), "q")
        _need(o, torch.float32, (B, Hq, 128), "o")
        _check(_lib.lk_decode_attn_static(self._h, layer, q.data_ptr(), o.data_ptr(), _stream(stream)))
        return o

    def step_host(self, layer, q, k, v, ids, o, stream=None):
        """q/k/v/ids/o are host tensors (pinned ones are read and written in
        place by the kernels, others are copied); o is valid after the stream
        syncs."""
        import torch
        B, Hq, H = self.batch, self.plan.num_q_heads, self.plan.num_kv_heads
        _need(q, torch.bfloat16, (B, Hq, 128), "q", "cpu")
        _need(k, torch.bfloat16, (B, H, 128), "k", "cpu")
        _need(v, torch.bfloat16, (B, H, 128), "v", "cpu")
        _need(o, torch.float32, (B, Hq, 128), "o", "cpu")
        if ids is not None:
            _need(ids, torch.int32, (B,), "ids", "cpu")
        _check(_lib.lk_step_host(self._h, layer, q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(ids),
                                 o.data_ptr(), self.workspace.data_ptr(), self.workspace.numel(),
                                 _stream(stream)))

    def packed_input_bytes(self, with_ids):
        B, Hq, H = self.batch, self.plan.num_q_heads, self.plan.num_kv_heads
        return B * (Hq + 2 * H) * 256 + (B * 4 if with_ids else 0)

    def step_host_packed(self, layer, host_in, with_ids, o, stream=None):
        """lk_step_host_packed: host_in is one pinned uint8 block q|k|v|ids."""
        import torch
        _need(host_in, torch.uint8, (self.packed_input_bytes(with_ids),), "host_in", "cpu")
        _need(o, torch.float32, (self.batch, self.plan.num_q_heads, 128), "o", "cpu")
        _check(_lib.lk_step_host_packed(self._h, layer, host_in.data_ptr(), 1 if with_ids else 0, o.data_ptr(),
                                        self.workspace.data_ptr(), self.workspace.numel(), _stream(stream)))

    def layers_packed_input_bytes(self, nlayers, with_ids):
        B, Hq, H = self.batch, self.plan.num_q_heads, self.plan.num_kv_heads
        return nlayers * B * (Hq + 2 * H) * 256 + (B * 4 if with_ids else 0)

    def step_layers_host_packed(self, layer0, nlayers, host_in, with_ids, o, stream=None):
        """lk_step_layers_host_packed: host_in is one pinned uint8 block
        q (all layers) | k | v | ids; o pinned fp32 [nlayers, B, Hq, 128]."""
        import torch
        _need(host_in, torch.uint8, (self.layers_packed_input_bytes(nlayers, with_ids),), "host_in", "cpu")
        _need(o, torch.float32, (nlayers, self.batch, self.plan.num_q_heads, 128), "o", "cpu")
        _check(_lib.lk_step_layers_host_packed(self._h, layer0, nlayers, host_in.data_ptr(), 1 if with_ids else 0,
                                               o.data_ptr(), self.workspace.data_ptr(), self.workspace.numel(),
                                               _stream(stream)))

    # -- queries
    def length(self, layer):
        n = ctypes.c_int32()
        _check(_lib.lk_cache_length(self._h, layer, ctypes.byref(n)))
        return n.value

    def region(self, layer, b, kv_head) -> RegionInfo:
        r = RegionInfo()
        _check(_lib.lk_cache_region(self._h, layer, b, kv_head, ctypes.byref(r)))
        return r

    def resident_bytes(self, layer, stream=None):
        n = ctypes.c_uint64()
        _check(_lib.lk_resident_bytes(self._h, layer, _stream(stream), ctypes.byref(n)))
        return n.value

    def set_decode_ctas(self, ctas):
        _check(_lib.lk_set_decode_ctas(self._h, ctas))

    def workspace_init(self, stream=None):
        """lk_workspace_init: zero this cache's workspace (after LK_ERR_TIMEOUT)."""
        _check(_lib.lk_workspace_init(self._h, self.workspace.data_ptr(), self.workspace.numel(), _stream(stream)))

    def set_wait_limit(self, ns):
        """lk_set_wait_limit: bound of the decode kernel's waits (ns)."""
        _check(_lib.lk_set_wait_limit(self._h, int(ns)))

    def check(self, stream=None):
        _check(_lib.lk_check(self._h, _stream(stream)))

    def rows(self, offset, nrows, width):
        """View of `nrows` bf16 rows of `width` channels at a byte offset of the buffer."""
        import torch
        nb = nrows * width * 2
        return self.buffer[offset: offset + nb].view(torch.bfloat16).view(nrows, width)

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.lk_cache_destroy(self._h)
            self._h = None
