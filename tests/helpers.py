"""Shared test plumbing: build a cache for a workload on the GPU and compute
what the oracle expects from the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from oracle import attention as OA
from oracle import layout as OL
from oracle import masks as OM
from oracle import quant as OQ

# max |err| bound of the decode output against the fp64 oracle (bf16 inputs,
# fp32 accumulation), as stated for this method's GPU path
DECODE_TOL = 2e-3


def workload_masks(w: S.Workload, policies=None) -> np.ndarray:
    """The workload's kept-channel masks [L, Hkv, 128]: LeanK stage 2 (the
    oracle's construction) on the seeded importances for a pruned workload,
    else the drawn per-head counts (top channels by importance)."""
    if w.prune_pct is None or w.budget == "choice64":
        return S.masks_with_counts(w, S.drawn_counts(w))
    alpha, elig = S.stage2_inputs(w, policies)
    return OM.top_s_prune(alpha, w.prune_pct, w.align, w.budget, elig)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class Case:
    """One workload instance: plan + cache on the GPU and its dense history.

    The dense history holds ``total`` tokens per layer; ``prefill`` of the
    first n0 of them followed by appends of the rest reproduces a decode loop.
    """

    def __init__(self, w: S.Workload, total: int, masks=None, policies=None, capacity=None,
                 special_capacity=0, device="cuda", layers=None, gen_device=None, middle_tokens=None,
                 kv_format=lkb.KV_BF16):
        self.w = w
        self.total = total
        self.policies = S.make_policies(w) if policies is None else np.asarray(policies, np.int32)
        self.masks = workload_masks(w, self.policies) if masks is None else np.asarray(masks, np.uint8)
        self.is_special = S.make_special_table(w)
        self.plan = lkb.Plan.for_workload(w, self.masks, self.policies, self.is_special,
                                          special_capacity=special_capacity)
        self.capacity = capacity or total
        self.kv_format = kv_format
        self.cache = lkb.Cache(self.plan, w.batch, self.capacity, device=device, middle_tokens=middle_tokens,
                               kv_format=kv_format)
        self.device = device
        self.layers = list(range(w.num_layers)) if layers is None else layers
        self.ids = torch.from_numpy(S.make_token_ids(w, total)).to(device)
        self.flags = self.is_special[S.make_token_ids(w, total)].astype(bool) if len(self.is_special) \
            else np.zeros((w.batch, total), dtype=bool)
        self.hist = {}
        self.gen_device = gen_device

    def history(self, layer):
        if layer not in self.hist:
            self.hist[layer] = S.make_kv(self.w, layer, self.total, device=self.gen_device)
            self.hist[layer] = tuple(t.to(self.device) for t in self.hist[layer])
        return self.hist[layer]

    def drop_history(self, layer):
        self.hist.pop(layer, None)

    def prefill(self, layer, n0):
        k, v = self.history(layer)
        ids = self.ids[:, :n0].contiguous() if len(self.is_special) else None
        self.cache.prefill(layer, k[:, :n0].contiguous(), v[:, :n0].contiguous(), ids)

    def append(self, layer, t):
        k, v = self.history(layer)
        ids = self.ids[:, t].contiguous() if len(self.is_special) else None
        self.cache.append(layer, k[:, t].contiguous(), v[:, t].contiguous(), ids)

    def q(self, layer, N, step=0):
        return S.make_q(self.w, layer, N - 1, device=self.gen_device, step=step).to(self.device)

    def expected(self, layer, q, N, heads=None):
        """fp64 oracle output for the first N tokens of the history (N an int,
        or one length per sequence)."""
        k, v = self.history(layer)
        w = self.w
        ragged = not np.isscalar(N)
        quant = self.kv_format != lkb.KV_BF16
        fmt = lkb.KV_FORMAT_NAMES[self.kv_format]
        if heads is None and not ragged and not quant:
            K, V = f64(k[:, :N]), f64(v[:, :N])
            return OA.decode_layer(f64(q), K, V, self.masks[layer], self.policies[layer], N, w.sink,
                                   w.local, w.local_only_window, self.flags)
        pairs = heads if heads is not None else [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
        out = {}
        G = w.group
        for b, h in pairs:
            Nb = int(N[b]) if ragged else N
            K, V = f64(k[b, :Nb, h]), f64(v[b, :Nb, h])
            kept = np.nonzero(self.masks[layer, h])[0]
            args = (f64(q[b, h * G:(h + 1) * G]), K, V, int(self.policies[layer, h]), kept, Nb, w.sink, w.local,
                    w.local_only_window, self.flags[b])
            out[(b, h)] = OQ.decode_head_quantized(*args, fmt=fmt) if quant else OA.decode_head(*args)
        if heads is None:
            full = np.zeros((w.batch, w.num_q_heads, 128))
            for (b, h), r in out.items():
                full[b, h * G:(h + 1) * G] = r
            return full
        return out

    def check_layout(self, layer, N, heads=None):
        """Every resident row of the cache equals the oracle's expected row."""
        k, v = self.history(layer)
        w = self.w
        B, H = w.batch, w.num_kv_heads
        pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
        for b, h in pairs:
            Nb = N if np.isscalar(N) else int(N[b])
            r = self.cache.region(layer, b, h)
            pol = int(self.policies[layer, h])
            kept = np.nonzero(self.masks[layer, h])[0] if pol == S.POLICY_FULL else np.arange(0)
            rows, toks = OL.region_a(pol, Nb, w.sink, w.local, w.local_only_window, self.flags[b],
                                     special_capacity=r.rows_a)
            if len(rows):
                ka = self.cache.rows(r.k_a_offset, r.rows_a, 128)
                va = self.cache.rows(r.v_a_offset, r.rows_a, 128)
                ri = torch.from_numpy(rows).to(self.device)
                ti = torch.from_numpy(toks).to(self.device)
                assert torch.equal(ka[ri], k[b, ti, h]), (layer, b, h, "K region A")
                assert torch.equal(va[ri], v[b, ti, h]), (layer, b, h, "V region A")
            rows, toks = OL.region_b(pol, len(kept), Nb, w.sink, w.local)
            if len(rows) and self.kv_format != lkb.KV_BF16:
                # complete blocks: codes and scales exactly as the oracle
                # quantises them; the open block: bf16 tail rows
                blocks = OQ.middle_blocks(f64(k[b, :, h]).astype(np.float32), f64(v[b, :, h]).astype(np.float32),
                                          kept, Nb, w.sink, w.local, fmt=lkb.KV_FORMAT_NAMES[self.kv_format])
                assert r.sealed_blocks == len(blocks), (layer, b, h, r.sealed_blocks, len(blocks))
                for j, (kc, ks, vc, vs) in enumerate(blocks):
                    gk, gks, gv, gvs = self.cache.block(layer, b, h, j)
                    assert np.array_equal(gk, kc) and np.array_equal(gks.view(np.uint32), ks.view(np.uint32)), \
                        (layer, b, h, j, "K block")
                    assert np.array_equal(gv, vc) and np.array_equal(gvs.view(np.uint32), vs.view(np.uint32)), \
                        (layer, b, h, j, "V block")
                keep = rows >= 128 * len(blocks)
                rows, toks = rows[keep] - 128 * len(blocks), toks[keep]
            if len(rows):
                ri = torch.from_numpy(rows).to(self.device)
                ti = torch.from_numpy(toks).to(self.device)
                ki = torch.from_numpy(kept).to(self.device)
                kb = self.cache.middle_rows(r, r.k_b_offset, r.n_kept, ri)
                vb = self.cache.middle_rows(r, r.v_b_offset, 128, ri)
                assert torch.equal(kb, k[b, ti, h][:, ki]), (layer, b, h, "K_prun")
                assert torch.equal(vb, v[b, ti, h]), (layer, b, h, "V middle")
