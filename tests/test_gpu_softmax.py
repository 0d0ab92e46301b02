"""GPU parity on inputs built to drive every branch of the online softmax.

The method runs one softmax over the full-width rows and the kept-channel
middle rows (LeanK article, framerc.cn, section 3.1, "fused computation"),
split over CTAs and merged by log-sum-exp.  The kernel moves a column's
running max only when a tile beats it by more than 2^8 (lazy rescaling) and
splits p into bf16 hi + lo halves for P.V.  Seeded N(0,1) caches almost never
reach either case, so these tests build K, V and q to reach them:

* climbing scores: a per-128-token offset of the scores (a random walk in
  log2 units with steps in [-6, 14]) makes later tiles beat the running max
  by more and by less than 2^8, across the full-width and middle regions and
  across CTA splits (1, 7 and the library's count), for bf16, INT8 and FP8
  middles and for fused and two-launch steps;
* peaky P: three dominant tokens (a sink, a middle and a window token) with
  near-equal scores and V rows of magnitude 6-8, beside a head with no kept
  channel (whose middle token must leave the softmax);
* special-token overflow (FastGen article, mhpn.cn, section 3.2 stage 2): a
  SPECIAL head keeps its first `special_capacity` special tokens and decode
  attends to exactly those.

Expected values are the fp64 oracle on the same inputs."""
import math

import numpy as np
import pytest
import torch

from decode_attention_pruned_gb300 import binding as lkb
from decode_attention_pruned_gb300 import synth as S
from helpers import DECODE_TOL, Case, f64
from oracle import attention as OA
from oracle import layout as OL

pytestmark = pytest.mark.gpu

LLAMA = S.WORKLOADS[1]
FASTGEN = S.WORKLOADS[4]
LOG2E_OVER_SQRT_D = math.log2(math.e) / math.sqrt(128)


def _max_err(o, ref):
    return float(np.abs(o.double().cpu().numpy() - ref).max())


def _unit(x):
    return x / x.norm(dim=-1, keepdim=True)


def _planted_case(w, counts, total, kv_format, target_fn, v_fn=None, seed=0, exact=()):
    """A Case whose history has K[t] = z_t + beta_t u_t, where u_t is a unit
    direction shared by the G query heads of the kv head (restricted to the
    kept channels for middle tokens, which are scored on those only) and
    beta_t puts the score of token t near target_fn(b, h, t) log2 units; q_g =
    d + 0.1 noise.  Tokens in `exact` have z_t = 0 (their scores then sit
    within ~1 % of the target).  v_fn(b, h, t) optionally overrides V rows."""
    masks = S.masks_with_counts(w, counts)
    case = Case(w, total=total, masks=masks, kv_format=kv_format)
    B, H, G, N = w.batch, w.num_kv_heads, w.group, total
    gen = torch.Generator().manual_seed(seed)
    d = torch.randn(B, H, 128, generator=gen, dtype=torch.float64)
    q = (d.repeat_interleave(G, dim=1) + 0.1 * torch.randn(B, H * G, 128, generator=gen, dtype=torch.float64))
    k = torch.randn(B, N, H, 128, generator=gen, dtype=torch.float64)
    v = torch.randn(B, N, H, 128, generator=gen, dtype=torch.float64)
    t = np.arange(N)
    mid = (t >= w.sink) & (t < N - w.local)
    for x in exact:
        k[:, x] = 0.0
    for h in range(H):
        kept = torch.from_numpy(masks[0, h].astype(np.float64))
        for b in range(B):
            u_full = _unit(d[b, h])
            dk = d[b, h] * kept
            u_mid = _unit(dk) if float(dk.norm()) > 0 else u_full
            # score of beta u against q_g ~ beta (d . u) / sqrt(128) in nats
            gain_full = float(d[b, h] @ u_full) * LOG2E_OVER_SQRT_D
            gain_mid = float(d[b, h] @ u_mid) * LOG2E_OVER_SQRT_D
            target = np.asarray([target_fn(b, h, int(x)) for x in t], dtype=np.float64)
            beta = np.where(mid, target / gain_mid, target / gain_full)
            dirs = torch.where(torch.from_numpy(mid)[:, None], u_mid[None, :], u_full[None, :])
            k[b, :, h] += torch.from_numpy(beta)[:, None] * dirs
            if v_fn is not None:
                for x in t:
                    row = v_fn(b, h, int(x))
                    if row is not None:
                        v[b, x, h] = torch.as_tensor(row, dtype=torch.float64)
    case.hist[0] = (k.to(torch.bfloat16).cuda(), v.to(torch.bfloat16).cuda())
    return case, q.to(torch.bfloat16).cuda()


def _line_row(w, N, t):
    """Where token t of an N-token FULL head sits in the order the kernel
    streams it: region A rows (sink t at row t, window token t at ring row
    S + (t - S) mod W), then the middle rows."""
    S_, W_ = w.sink, w.local
    if t < S_:
        return t
    if t >= N - W_:
        return S_ + (t - S_) % W_
    return S_ + W_ + (t - S_)


def _climb(w, N, seed):
    """target_fn: a random walk (log2 units) over 128-row blocks of the
    kernel's row order, so that scores climb as the rows stream."""
    rs = np.random.default_rng(seed)
    nblk = (N + 127) // 128 + 1
    walk = np.cumsum(rs.uniform(-6.0, 14.0, size=(w.batch, w.num_kv_heads, nblk)), axis=-1)
    return lambda b, h, t: float(walk[b, h, _line_row(w, N, t) // 128])


CLIMB_W = LLAMA.scaled(num_q_heads=16, num_kv_heads=4, batch=2, context=3000)
CLIMB_COUNTS = [64, 0, 32, 128]


@pytest.mark.parametrize("ctas", [1, 7, 0], ids=["ctas1", "ctas7", "default"])
@pytest.mark.parametrize("kv", [lkb.KV_BF16, lkb.KV_INT8, lkb.KV_FP8], ids=["bf16", "int8", "fp8"])
def test_climbing_scores_decode(cuda, kv, ctas):
    N = CLIMB_W.context
    case, q = _planted_case(CLIMB_W, CLIMB_COUNTS, N, kv, _climb(CLIMB_W, N, 5))
    case.prefill(0, N)
    case.cache.set_decode_ctas(ctas)
    o = case.cache.decode(0, q)
    case.cache.check()
    assert _max_err(o, case.expected(0, q, N)) <= DECODE_TOL


@pytest.mark.parametrize("mode", [lkb.STEP_FUSED, lkb.STEP_SPLIT], ids=["fused", "split"])
@pytest.mark.parametrize("ctas", [7, 0], ids=["ctas7", "default"])
def test_climbing_scores_step(cuda, mode, ctas):
    # the appended token and the window row it evicts join the softmax of
    # the step (fused: folded by the CTA that holds the evicted slot)
    N = CLIMB_W.context
    case, q = _planted_case(CLIMB_W, CLIMB_COUNTS, N, lkb.KV_BF16, _climb(CLIMB_W, N, 6))
    case.prefill(0, N - 1)
    case.cache.set_step_mode(mode)
    case.cache.set_decode_ctas(ctas)
    k, v = case.history(0)
    o = case.cache.step(0, q, k[:, N - 1].contiguous(), v[:, N - 1].contiguous())
    case.cache.check()
    assert _max_err(o, case.expected(0, q, N)) <= DECODE_TOL
    case.check_layout(0, N)


def test_climbing_scores_reach_the_rescale_branch():
    # the planted offsets make some 128-row tiles beat the running max by
    # more than 2^8 and others by less, in the kernel's row order, in the
    # middle region of every head that has one
    N = CLIMB_W.context
    fn = _climb(CLIMB_W, N, 5)
    for b in range(CLIMB_W.batch):
        for h in range(CLIMB_W.num_kv_heads):
            if CLIMB_COUNTS[h] == 0:
                continue
            x = np.full(N, -np.inf)
            for t in range(N):
                x[_line_row(CLIMB_W, N, t)] = fn(b, h, t)
            a = CLIMB_W.sink + CLIMB_W.local
            jumps = [x[i:i + 128].max() - x[:i].max() for i in range(a, N, 128)]
            assert max(jumps) > 8 and min(jumps) < 8


def _peaky(w, counts, kv, seed):
    N = w.context
    planted = {2: (40.0, 7.0), w.sink + 500: (40.2, -6.0), N - 5: (39.7, 8.0)}
    signs = np.random.default_rng(seed).choice([-1.0, 1.0], size=(len(planted), 128))
    order = sorted(planted)

    def target(b, h, t):
        return planted[t][0] if t in planted else 0.0

    def vrow(b, h, t):
        if t not in planted:
            return None
        return planted[t][1] * signs[order.index(t)]

    return _planted_case(w, counts, N, kv, target, vrow, seed=seed, exact=order)


@pytest.mark.parametrize("kv", [lkb.KV_BF16, lkb.KV_INT8, lkb.KV_FP8], ids=["bf16", "int8", "fp8"])
@pytest.mark.parametrize("ctas", [1, 0], ids=["ctas1", "default"])
def test_peaky_p_near_equal_dominant_tokens(cuda, kv, ctas):
    # o is a weighted mix of three V rows of size 6-8 with weights of equal
    # size: p kept to 8 bits would miss 2e-3 here; the head with k = 0 drops
    # the middle token (only the sink and window tokens stay)
    w = LLAMA.scaled(num_q_heads=16, num_kv_heads=4, batch=2, context=2200)
    case, q = _peaky(w, [64, 0, 32, 128], kv, seed=3)
    N = w.context
    case.prefill(0, N)
    case.cache.set_decode_ctas(ctas)
    o = case.cache.decode(0, q)
    case.cache.check()
    ref = case.expected(0, q, N)
    assert _max_err(o, ref) <= DECODE_TOL
    # the planted tokens dominate: o is far from the mean of V
    assert float(np.abs(ref).max()) > 3.0


def _capped_flags(case, N, cap):
    """Special flags that keep only the first `cap` special tokens of each
    sequence: the rows a SPECIAL head holds (oracle layout)."""
    out = np.zeros_like(case.flags)
    for b in range(case.w.batch):
        _, toks = OL.region_a(S.POLICY_SPECIAL, N, 0, 0, 0, case.flags[b], special_capacity=cap)
        out[b, toks] = True
    return out


def test_special_overflow_decodes_the_kept_rows(cuda):
    w = FASTGEN.scaled(num_layers=1, batch=2, context=400, policy_counts=(2, 4, 2))
    cap = 4
    case = Case(w, total=420, special_capacity=cap)
    assert case.flags[:, :400].sum(axis=1).min() > cap          # every sequence overflows
    case.prefill(0, 400)
    with pytest.raises(lkb.LeankError) as e:
        case.cache.check()
    assert e.value.status == lkb.LK_ERR_CAPACITY
    for N in (400, 420):
        if N == 420:
            for t in range(400, 420):
                case.append(0, t)
            try:                                # a special token among them overflows again
                case.cache.check()
            except lkb.LeankError as e:
                assert e.status == lkb.LK_ERR_CAPACITY
        q = case.q(0, N, step=N)
        o = case.cache.decode(0, q)
        case.cache.check()
        k, v = case.history(0)
        flags = _capped_flags(case, N, cap)
        ref = OA.decode_layer(f64(q), f64(k[:, :N]), f64(v[:, :N]), case.masks[0], case.policies[0], N, w.sink,
                              w.local, w.local_only_window, flags)
        assert _max_err(o, ref) <= DECODE_TOL, N
        case.check_layout(0, N)
