"""lk_resident_bytes -- the numerator of every GB/s and roofline figure the
bench reports -- against the oracle's byte counts, at the five workloads'
full sizes: contiguous and paged bf16 caches, INT8 and paged FP8 middles.

The oracle counts per (sequence, kv head) from the method's rules alone
(LeanK article, framerc.cn, sections 3.1-3.2: sinks and window at full
width, middle tokens on the kept channels plus their V row, nothing in the
middle for a head with no kept channel; FastGen article, mhpn.cn, section
3.2: the last W_loc tokens of a LOCAL head, the special tokens of a SPECIAL
head up to its row capacity; INT8 / FP8: complete 128-row middle blocks as
one-byte codes plus fp32 scales).  The cache contents do not matter for the
count, so the histories are zeros; the token ids are the workload's."""
import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from helpers import workload_masks
from oracle import footprint as F
from oracle import quant as OQ

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _oracle_bytes(w, masks, pol, N, flags, spec_cap, kv):
    per_layer = []
    fn = OQ.resident_bytes_quantized if kv != lkb.KV_BF16 else F.resident_bytes
    n_special = np.minimum(flags[:, :N].sum(axis=1), spec_cap) if flags is not None else np.zeros(w.batch, int)
    for l in range(w.num_layers):
        tot = 0
        for b in range(w.batch):
            for h in range(w.num_kv_heads):
                tot += fn(int(pol[l, h]), int(masks[l, h].sum()), N, w.sink, w.local, w.local_only_window,
                          n_special=int(n_special[b]))
        per_layer.append(tot)
    return per_layer


@pytest.mark.parametrize("layout,kv", [("contiguous", lkb.KV_BF16), ("paged", lkb.KV_BF16),
                                       ("contiguous", lkb.KV_INT8), ("paged", lkb.KV_FP8)],
                         ids=["bf16", "bf16-paged", "int8", "fp8-paged"])
@pytest.mark.parametrize("w", S.WORKLOADS, ids=[w.name for w in S.WORKLOADS])
def test_resident_bytes_match_the_oracle(cuda, w, layout, kv):
    N = w.context
    pol = S.make_policies(w)
    masks = workload_masks(w, pol)
    spec = S.make_special_table(w)
    plan = lkb.Plan.for_workload(w, masks, pol, spec if len(spec) else None)
    middle = w.batch * max(0, N - w.sink - w.local) if layout == "paged" else None
    cache = lkb.Cache(plan, w.batch, N, device=cuda, middle_tokens=middle, kv_format=kv)
    k = torch.zeros((w.batch, N, w.num_kv_heads, 128), dtype=torch.bfloat16, device=cuda)
    ids_np = S.make_token_ids(w, N) if len(spec) else None
    ids = torch.from_numpy(ids_np).to(cuda) if ids_np is not None else None
    for l in range(w.num_layers):
        cache.prefill(l, k, k, ids)
    cache.check()
    flags = spec[ids_np].astype(bool) if ids_np is not None else None
    want = _oracle_bytes(w, masks, pol, N, flags, N, kv)
    got = [cache.resident_bytes(l) for l in range(w.num_layers)]
    assert got == want
    del cache, k
    torch.cuda.empty_cache()
