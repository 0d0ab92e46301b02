"""The device mask builder (lk_build_masks) against the oracle's stage-2
mask construction: bit-exact (the output is integer)."""
import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from oracle import masks as OM

pytestmark = pytest.mark.gpu


def _device_masks(alpha, s, align, exact, eligible, cuda):
    a = torch.from_numpy(np.ascontiguousarray(alpha, dtype=np.float32)).to(cuda)
    e = None if eligible is None else torch.from_numpy(eligible.astype(np.uint8)).to(cuda)
    out = lkb.build_masks(a, s, align=align, exact=exact, eligible=e)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("trial", range(8))
def test_random_importances(cuda, trial):
    rs = np.random.default_rng(100 + trial)
    L, H = int(rs.integers(1, 9)), int(rs.integers(1, 17))
    a = np.exp(rs.standard_normal((L, H, 128)) + 0.4 * rs.standard_normal((L, H, 1))).astype(np.float32)
    if trial % 3 == 1:
        a = np.round(a, 1).astype(np.float32)                 # many ties
    elig = None if trial % 2 == 0 else (rs.random((L, H)) < 0.7)
    if elig is not None:
        elig[0, 0] = True
    for s in (float(rs.uniform(30, 90)), 70.0):
        for align in (32, 64):
            for exact in (False, True):
                got = _device_masks(a, s, align, exact, elig, cuda)
                want = OM.top_s_prune(a, s, align, "exact" if exact else "round_down", elig)
                assert np.array_equal(got, want), (trial, s, align, exact)


@pytest.mark.parametrize("name", ["llama31_8b_layer", "serving_b64", "qwen25_7b_long", "fastgen_mix"])
def test_workload_importances(cuda, name):
    w = S.WORKLOAD_BY_NAME[name]
    pol = S.make_policies(w)
    alpha = S.draw_alpha(w).astype(np.float32)
    elig = pol == S.POLICY_FULL
    budget = w.budget
    got = _device_masks(alpha, w.prune_pct, 32, budget == "exact", None if elig.all() else elig, cuda)
    want = OM.top_s_prune(alpha, w.prune_pct, 32, budget, elig)
    assert np.array_equal(got, want)
    assert np.all(got.sum(-1) % 32 == 0)


def test_edge_cases(cuda):
    a = np.zeros((1, 2, 128), dtype=np.float32)
    a[0, 0] = np.arange(1, 129)
    a[0, 1] = np.arange(129, 257)
    for s in (0.0, 65.0, 100.0):
        for exact in (False, True):
            got = _device_masks(a, s, 32, exact, None, cuda)
            assert np.array_equal(got, OM.top_s_prune(a, s, 32, "exact" if exact else "round_down"))
    got = _device_masks(a, 65.0, 32, True, np.zeros((1, 2), bool), cuda)     # no eligible head
    assert np.all(got == 1)
    with pytest.raises(lkb.LeankError):
        _device_masks(a, 65.0, 48, False, None, cuda)
    with pytest.raises(lkb.LeankError):
        _device_masks(a, 101.0, 32, False, None, cuda)
