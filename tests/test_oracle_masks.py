"""Pins for the oracle's stage-2 mask builder (oracle/masks.py): a hand-worked
example, brute-force properties on random importances, the library
percentile, and planted mistakes that must be caught."""
import numpy as np
import pytest

from oracle import masks as OM


def _ladder():
    # head 0 holds alpha 1..128, head 1 holds 129..256 (channel c -> value)
    a = np.zeros((1, 2, 128), dtype=np.float32)
    a[0, 0] = np.arange(1, 129)
    a[0, 1] = np.arange(129, 257)
    return a


def check_hand_example():
    a = _ladder()
    # s = 70: p = 0.7 * 255 = 178.5 -> threshold 179 + 0.5 = 179.5; head 1 has
    # 77 values >= 179.5 (180..256) -> 64 after rounding down; head 0 none.
    assert OM.percentile_fp32(a, 70.0) == np.float32(179.5)
    assert OM.aligned_counts(a, 70.0, 32, "round_down").tolist() == [[0, 64]]
    m = OM.top_s_prune(a, 70.0, 32, "round_down")
    assert np.nonzero(m[0, 1])[0].tolist() == list(range(64, 128))      # values 193..256
    assert m[0, 0].sum() == 0
    # s = 65: threshold 166 + 0.75 = 166.75 -> 90 above -> 64, remainder 26;
    # exact budget 32 * floor(0.35 * 256 / 32 + 0.5) = 96 -> head 1 gets 96.
    assert OM.percentile_fp32(a, 65.0) == np.float32(166.75)
    assert OM.aligned_counts(a, 65.0, 32, "exact").tolist() == [[0, 96]]
    m = OM.top_s_prune(a, 65.0, 32, "exact")
    assert np.nonzero(m[0, 1])[0].tolist() == list(range(32, 128))
    # alignment 64 rounds 90 down to 64
    assert OM.aligned_counts(a, 65.0, 64, "round_down").tolist() == [[0, 64]]


def check_properties_random():
    rs = np.random.default_rng(4)
    for trial in range(6):
        L, H = int(rs.integers(1, 5)), int(rs.integers(1, 9))
        a = np.exp(rs.standard_normal((L, H, 128)) + 0.3 * rs.standard_normal((L, H, 1))).astype(np.float32)
        if trial % 2:
            a = np.round(a, 1).astype(np.float32)          # many ties
        elig = rs.random((L, H)) < 0.8
        elig[0, 0] = True
        for budget in ("round_down", "exact"):
            for align in (32, 64):
                s = float(rs.uniform(40, 85))
                m = OM.top_s_prune(a, s, align, budget, elig)
                thr = OM.percentile_fp32(a[elig], s)
                counts = m.sum(-1)
                for l in range(L):
                    for h in range(H):
                        if not elig[l, h]:
                            assert counts[l, h] == 128
                            continue
                        assert counts[l, h] % align == 0
                        above = int((a[l, h] >= thr).sum())
                        if budget == "round_down":
                            assert counts[l, h] == above // align * align
                        else:
                            assert above // align * align <= counts[l, h] <= 128
                        kept = np.nonzero(m[l, h])[0]
                        dropped = np.nonzero(m[l, h] == 0)[0]
                        if len(kept) and len(dropped):
                            lo = a[l, h, kept].min()
                            assert lo >= a[l, h, dropped].max()
                            for c in dropped:          # ties go to the lower index
                                if a[l, h, c] == lo:
                                    assert c > kept[a[l, h, kept] == lo].max()
                if budget == "exact":
                    n = int(elig.sum())
                    target = align * int(np.floor((1 - s / 100) * n * 128 / align + 0.5))
                    assert counts[elig].sum() == min(target, 128 * n) or counts[elig].sum() <= target


def check_percentile_matches_library():
    rs = np.random.default_rng(9)
    for n in (7, 128, 3000):
        v = rs.standard_normal(n).astype(np.float32)
        for s in (0.0, 12.5, 70.0, 99.9, 100.0):
            got = float(OM.percentile_fp32(v, s))
            ref = float(np.percentile(v.astype(np.float64), s))
            assert abs(got - ref) <= 1e-6 * max(1.0, abs(ref))


PINS = [check_hand_example, check_properties_random, check_percentile_matches_library]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


MUTATIONS = {
    "round_up": lambda mp: mp.setattr(
        OM, "aligned_counts",
        (lambda f: (lambda a, s, al, b, e=None: np.minimum(128, -(-f(a, s, 1, "round_down", e) // al) * al)))(
            OM.aligned_counts)),
    "keep_above_threshold_share": lambda mp: mp.setattr(
        OM, "percentile_fp32", (lambda f: (lambda v, s: f(v, 100.0 - s)))(OM.percentile_fp32)),
    "no_interpolation": lambda mp: mp.setattr(
        OM, "percentile_fp32",
        lambda v, s: np.float32(np.sort(np.asarray(v, np.float32).ravel())[int(s / 100.0 * (np.size(v) - 1))])),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    MUTATIONS[name](monkeypatch)
    failures = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, name
