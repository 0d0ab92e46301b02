"""Throughput of decode attention over a LeanK-pruned KV cache on one GB300.

One step = one pass of the whole hot path for one decode token of the
workload: for each layer, the append (new K/V into the window ring, eviction
into K_prun) then the split-K decode with its in-launch combine, through
lk_step_layers.  --step auto (default) lets the library choose between one
fused launch and the append + decode launches (it fuses launches over few,
long entries with a bf16 middle); --step fused / split force one.
Default workload: the batch-serving step (32 layers x 32 q / 8 kv heads,
d 128, batch 64, context 4096, sink 16, window 512, 70 % channel pruning
rounded down to multiples of 32), the largest single-GPU workload; the
channel masks come from the library's mask builder (lk_build_masks) on the
seeded importances.

Timing rules: W untimed warm-up steps (at least one use of every cache copy
and one replay of every captured graph, whatever W is); exactly K timed steps
bracketed by a barrier + synchronize; CUDA events on the launching stream;
max over ranks.  Inputs are larger than L2: the steps rotate over C copies of
the cache whose resident bytes together exceed 4x L2, and C also bounds the
context growth of the appends.  The step loop is captured in CUDA graphs
(programmatic dependent launch between consecutive kernels).  Clocks are
sampled over the loaded window: untimed decode-only replays that bring the
GPU to its load clocks, then the timed steps.

Printed: one JSON line (rank 0).  `value` = decode-attention calls/s of all
ranks (a call = one layer's decode over every sequence and kv head);
`roofline` = the step's decode kernel (the fused one when the step is one
launch): algorithmic bytes / event-timed launch duration, against the HBM
peak; `e2e` = the same metric through lk_step_host_packed (one layer) or
lk_step_layers_host_packed (several) from pinned host memory, the host
traffic inside the timed region; `cpu_baseline` = the fp64 oracle on a
bounded sample on all host cores (worker processes) and on one core.

--impl reference times the oracle (the only reference this method has) on
the host's cores, on the same workload: each step is one (sequence, kv head)
unit per worker process.
"""
from __future__ import annotations

import os

# the oracle's numpy BLAS runs on exactly one thread (reported as `cores`)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode-attn calls/s & effective HBM GB/s (% of GB300 peak) on pruned KV"
UNIT = "calls/s"
FALLBACK_HBM_GBS = 6800.0
MAX_CONTEXT_GROWTH = 0.01           # appends may lengthen the context by at most 1 %
COPY_BUDGET_BYTES = 120 << 30       # device memory the rotating copies may take
MAX_COPIES = 256                    # rotating cache copies at most

# DRAM bytes (read + write) per decode launch from one ncu capture, keyed by
# "<sha256[:16] of the decode kernel sources>:<workload>[/<layers>L][/paged]:<kv
# format>:<fused | decode>" (the bench reports null when the kernel changed
# since the capture).  The 32-layer launches are too large to capture with
# multi-pass metrics; their entries are the traffic per algorithmic byte of
# the same workload's 4-layer capture (the 2-layer one is listed beside it:
# the ratio falls as the launch grows, since the excess is mostly per CTA --
# split partials, each CTA's last box past its range end), applied to the
# full launch's algorithmic bytes.
NCU_TRAFFIC = {
    "0197f9dad46f17ec:fastgen_mix/2L:bf16:fused": 445716480,
    "0197f9dad46f17ec:fastgen_mix/2L:fp8:decode": 265465088,
    "0197f9dad46f17ec:fastgen_mix/2L:int8:decode": 265490688,
    "0197f9dad46f17ec:fastgen_mix/4L:bf16:fused": 867568128,
    "0197f9dad46f17ec:fastgen_mix/4L:fp8:decode": 514968832,
    "0197f9dad46f17ec:fastgen_mix/4L:int8:decode": 515119872,
    "0197f9dad46f17ec:llama31_8b_layer:bf16:decode": 88016128,
    "0197f9dad46f17ec:llama31_8b_layer:bf16:fused": 88024320,
    "0197f9dad46f17ec:llama31_8b_layer:fp8:decode": 46433792,
    "0197f9dad46f17ec:llama31_8b_layer:int8:decode": 46436864,
    "0197f9dad46f17ec:llama31_8b_layer/paged:bf16:fused": 87989504,
    "0197f9dad46f17ec:qwen25_7b_long:bf16:fused": 517321216,
    "0197f9dad46f17ec:qwen25_7b_long:fp8:decode": 278952960,
    "0197f9dad46f17ec:qwen25_7b_long:int8:decode": 278957056,
    "0197f9dad46f17ec:serving_b64/2L:bf16:decode": 947085056,
    "0197f9dad46f17ec:serving_b64/2L:bf16:fused": 947103232,
    "0197f9dad46f17ec:serving_b64/2L:fp8:decode": 637853952,
    "0197f9dad46f17ec:serving_b64/2L:int8:decode": 637905408,
    "0197f9dad46f17ec:serving_b64/2L/paged:bf16:decode": 946146048,
    "0197f9dad46f17ec:serving_b64/2L/paged:bf16:fused": 946523904,
    "0197f9dad46f17ec:serving_b64/2L/paged:int8:decode": 637677056,
    "0197f9dad46f17ec:serving_b64/4L:bf16:decode": 2179566080,
    "0197f9dad46f17ec:serving_b64/4L:bf16:fused": 2179599872,
    "0197f9dad46f17ec:serving_b64/4L:fp8:decode": 1425171200,
    "0197f9dad46f17ec:serving_b64/4L:int8:decode": 1425136640,
    "0197f9dad46f17ec:serving_b64/4L/paged:bf16:decode": 2178592000,
    "0197f9dad46f17ec:serving_b64/4L/paged:bf16:fused": 2178788608,
    "0197f9dad46f17ec:serving_b64/4L/paged:int8:decode": 1425398528,
    "0197f9dad46f17ec:tiny:bf16:fused": 529920,
}
# 32-layer launches: DRAM bytes per algorithmic byte of the 4-layer capture
NCU_TRAFFIC_RATIO = {
    "0197f9dad46f17ec:serving_b64:bf16:decode": 2179566080 / 2178351104,
    "0197f9dad46f17ec:serving_b64:int8:decode": 1425136640 / 1396178944,
    "0197f9dad46f17ec:serving_b64:fp8:decode": 1425171200 / 1396178944,
    "0197f9dad46f17ec:serving_b64/paged:bf16:decode": 2178592000 / 2178351104,
    "0197f9dad46f17ec:serving_b64/paged:int8:decode": 1425398528 / 1396178944,
    "0197f9dad46f17ec:fastgen_mix:bf16:fused": 867568128 / 856061952,
    "0197f9dad46f17ec:fastgen_mix:int8:decode": 515119872 / 504039424,
    "0197f9dad46f17ec:fastgen_mix:fp8:decode": 514968832 / 504039424,
}


def _rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
                if key in d:
                    return float(d[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _decode_source_hash():
    """sha256[:16] of the decode kernel's sources (the kernel file and the
    device headers it includes)."""
    h = hashlib.sha256()
    for f in ("lk_decode.cu", "lk_append.cuh", "lk_device.cuh", "lk_internal.h"):
        h.update(open(os.path.join(ROOT, "decode_attention_pruned_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(seconds: float, dist, device) -> float:
    """The slowest rank's time (the job's time for weak-scaled replicas)."""
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(steps: int, layers: int, world: int, seconds: float) -> float:
    """Calls/s of the whole job: every rank ran `steps` steps of `layers` calls."""
    return steps * layers * world / seconds


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def device_masks(w, pol, dev):
    """The workload's kept-channel masks [L, Hkv, 128] (host uint8): LeanK
    stage 2 by the library's mask builder on the seeded importances, or the
    drawn counts of a workload without a prune ratio."""
    import torch
    from decode_attention_pruned_gb300 import binding as lkb
    from decode_attention_pruned_gb300 import synth as S
    if w.prune_pct is None or w.budget == "choice64":
        return S.masks_with_counts(w, S.drawn_counts(w))
    alpha, elig = S.stage2_inputs(w, pol)
    a = torch.from_numpy(alpha).to(dev)
    e = None if elig.all() else torch.from_numpy(elig.astype(np.uint8)).to(dev)
    m = lkb.build_masks(a, w.prune_pct, align=w.align, exact=w.budget == "exact", eligible=e)
    torch.cuda.synchronize(dev)
    return m.cpu().numpy()


def run_gpu(args, rank, local_rank, world):
    import torch
    from decode_attention_pruned_gb300 import binding as lkb
    from decode_attention_pruned_gb300 import synth as S

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lkb.load()
    w = S.WORKLOAD_BY_NAME[args.workload]
    N = w.context
    pol = S.make_policies(w)
    masks = device_masks(w, pol, dev)
    spec = S.make_special_table(w)
    if args.layers:
        # a smaller case for profiling: the workload's first layers, with the
        # masks and policies they have in the whole workload
        if not 0 < args.layers <= w.num_layers:
            raise SystemExit(f"--layers must be in 1..{w.num_layers}")
        w = w.scaled(num_layers=args.layers)
        pol, masks = pol[: w.num_layers].copy(), masks[: w.num_layers].copy()
    plan = lkb.Plan.for_workload(w, masks, pol, spec if len(spec) else None)
    L, B = w.num_layers, w.batch
    W, K = args.warmup, args.steps
    e2e_steps = min(K, args.e2e_steps)
    kt_steps = min(K, args.kernel_steps)
    # appends over all copies: the warm-up, the timed steps, the end-to-end
    # steps, slack; every copy also takes up to 3 in the warm-up's first
    # rotations (eager step, graph replay, remainder graph)
    appends = W + K + 2 * e2e_steps + 8

    # one copy first, to size the rest
    prop = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(prop, "L2_cache_size", 0) or 126 << 20)
    max_growth = max(1, int(MAX_CONTEXT_GROWTH * N))
    cap_probe = N + 64
    paged = args.layout == "paged"
    kvf = {"bf16": lkb.KV_BF16, "int8": lkb.KV_INT8, "fp8": lkb.KV_FP8}[args.kv]
    # paged: page pools sized for every sequence's middle at the capacity
    middle = (lambda cap: B * max(0, cap - w.sink - w.local)) if paged else (lambda cap: None)
    copy_bytes = plan.cache_bytes(B, cap_probe, middle(cap_probe), kvf) + plan.workspace_bytes(B)

    # dense history of every layer, generated once on the device
    hist = {l: S.make_kv(w, l, N, device=dev) for l in range(L)} if L <= 2 else None
    ids_all = torch.from_numpy(S.make_token_ids(w, N)).to(dev) if len(spec) else None

    first = lkb.Cache(plan, B, cap_probe, device=dev, middle_tokens=middle(cap_probe), kv_format=kvf)
    for l in range(L):
        k, v = hist[l] if hist else S.make_kv(w, l, N, device=dev)
        first.prefill(l, k[:, : N - 1].contiguous(), v[:, : N - 1].contiguous(),
                      None if ids_all is None else ids_all[:, : N - 1].contiguous())
        first.append(l, k[:, N - 1].contiguous(), v[:, N - 1].contiguous(),
                     None if ids_all is None else ids_all[:, N - 1].contiguous())
    torch.cuda.synchronize()
    resident = [first.resident_bytes(l) for l in range(L)]
    resident_step = sum(resident)
    copies = max(1, math.ceil(4 * l2 / max(1, resident_step)), math.ceil(appends / max(1, max_growth - 3)))
    copies = int(min(copies, MAX_COPIES, max(1, COPY_BUDGET_BYTES // copy_bytes)))
    growth = math.ceil(appends / copies) + 6
    capacity = N + growth
    del first
    torch.cuda.empty_cache()

    caches = []
    for c in range(copies):
        cache = lkb.Cache(plan, B, capacity, device=dev, middle_tokens=middle(capacity), kv_format=kvf)
        if args.decode_ctas:
            cache.set_decode_ctas(args.decode_ctas)
        for l in range(L):
            k, v = hist[l] if hist else S.make_kv(w, l, N, device=dev)
            cache.prefill(l, k[:, : N - 1].contiguous(), v[:, : N - 1].contiguous(),
                          None if ids_all is None else ids_all[:, : N - 1].contiguous())
        caches.append(cache)
    hist = None
    torch.cuda.synchronize()

    # per-step inputs (a bank cycled through), resident before timing:
    # q [L, B, Hq, 128]; the new token's k, v [L, B, Hkv, 128]
    bank = 16
    gq = [torch.stack([S.make_q(w, l, N - 1, device=dev, step=s) for l in range(L)]).contiguous()
          for s in range(bank)]
    gk, gv = [], []
    for s in range(bank):
        kk, vv = S.make_kv(w.scaled(seed=w.seed + 7919 * (s + 1), num_layers=1, batch=L * B), 0, 1, device=dev)
        gk.append(kk[:, 0].reshape(L, B, w.num_kv_heads, 128).contiguous())
        gv.append(vv[:, 0].reshape(L, B, w.num_kv_heads, 128).contiguous())
    gid = [torch.zeros(B, dtype=torch.int32, device=dev) + (s * 37) % max(1, w.vocab) for s in range(bank)] \
        if len(spec) else [None] * bank
    outs = [torch.empty((L, B, w.num_q_heads, 128), dtype=torch.float32, device=dev) for _ in range(copies)]

    stream = torch.cuda.Stream(device=dev)

    # one step: the new token into every layer (one launch), then decode
    # attention of every layer (one launch; for one layer these are the plain
    # per-layer calls)
    mode = {"auto": lkb.STEP_AUTO, "fused": lkb.STEP_FUSED, "split": lkb.STEP_SPLIT}[args.step]
    for c in caches:
        c.set_step_mode(mode)
    fused = caches[0].step_is_fused(0, L)

    def enqueue_step(i):
        c = caches[i % copies]
        s = i % bank
        c.step_layers(0, gq[s], gk[s], gv[s], gid[s], outs[i % copies], stream=stream)

    # graphs of whole rotations (copies steps) plus one of the remainder
    def capture(n_steps, start):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n_steps):
                enqueue_step(start + j)
        return g

    # warm-up: one eager step on every cache copy (its first use), then one
    # replay of every captured graph (their uploads), then the rest of W
    with torch.cuda.stream(stream):
        for i in range(copies):
            enqueue_step(i)
    stream.synchronize()
    for c in caches:
        c.check(stream)
    full_graph = capture(copies, 0)
    rem = K % copies
    rem_graph = capture(rem, 0) if rem else None
    # (capture only records the steps: the kernels read the device lengths,
    # which only executed steps advance)
    with torch.cuda.stream(stream):
        full_graph.replay()
        if rem_graph is not None:
            rem_graph.replay()
        warm_done = 2 * copies + rem
        while warm_done < W:
            full_graph.replay()
            warm_done += copies
    stream.synchronize()
    for c in caches:
        c.check(stream)

    # decode-only graph: back-to-back decode launches over the rotating
    # copies (no append between; the lengths stay put).  Its replays load
    # the GPU before the timed steps (so the clock samples show it under
    # load) and, after them, time the decode kernel alone.
    n_kg = min(max(kt_steps, 1), max(copies, 8))
    kgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(kgraph, stream=stream):
        for i in range(n_kg):
            caches[i % copies].decode_layers(0, gq[i % bank], outs[i % copies], stream=stream)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        kgraph.replay()                        # upload
        k0.record(stream)
        kgraph.replay()
        k1.record(stream)
    k1.synchronize()
    t_kg = max(1e-6, k0.elapsed_time(k1) / 1e3)
    load_reps = int(min(20000, math.ceil(args.load_seconds / t_kg))) if args.load_seconds > 0 else 0
    # resident bytes of the timed steps: every copy holds the same lengths
    # (the steps rotate over them), which grow by at most one token per copy
    # and rotation; the launches' mean is the mean of the two ends
    res_before = sum(caches[0].resident_bytes(l, stream=stream) for l in range(L))

    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            for _ in range(load_reps):
                kgraph.replay()
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(K // copies):
                full_graph.replay()
            if rem_graph is not None:
                rem_graph.replay()
        ev1.record(stream)
        ev1.synchronize()
    torch.cuda.synchronize()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    if dist is not None:
        elapsed = max_over_ranks(elapsed, dist, dev)
    for c in caches:
        c.check(stream)
    res_after = sum(caches[K % copies].resident_bytes(l, stream=stream) for l in range(L))
    resident_step = (res_before + res_after) / 2

    # the decode kernel alone: kgraph replays, CUDA events around them on the
    # launching stream, divided by the launches.  Event pairs around single
    # launches are also reported: they add each launch's front-end latency,
    # so they understate the kernel's rate.
    reps = max(3, kt_steps // n_kg)
    k0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            kgraph.replay()
    k1.record(stream)
    k1.synchronize()
    kdur = k0.elapsed_time(k1) / 1e3 / (reps * n_kg)
    res_kernel = sum(caches[0].resident_bytes(l, stream=stream) for l in range(L))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(kt_steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(kt_steps)]
    with torch.cuda.stream(stream):
        for i in range(kt_steps):
            c = caches[i % copies]
            starts[i].record(stream)
            c.decode_layers(0, gq[i % bank], outs[i % copies], stream=stream)
            ends[i].record(stream)
    stream.synchronize()
    kdur_isolated = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3 if kt_steps else kdur

    # end to end from pinned host memory: each step's inputs sit in one host
    # block, read in place by the kernels (lk_step_host_packed: q | k | v |
    # ids of one layer; over several layers lk_step_layers_host_packed: q of
    # every layer | k | v | ids), and o lands in a pinned host buffer
    def packed_inputs(s):
        if L == 1:
            parts = [gq[s][0], gk[s][0], gv[s][0]]
        else:
            parts = [gq[s], gk[s], gv[s]]
        parts = [p.contiguous().view(torch.uint8).reshape(-1) for p in parts]
        if gid[s] is not None:
            parts.append(gid[s].view(torch.uint8).reshape(-1))
        return torch.cat([p.cpu() for p in parts]).pin_memory()
    packed = [packed_inputs(s) for s in range(bank)]
    with_ids = gid[0] is not None
    ho = torch.empty((L, B, w.num_q_heads, 128), dtype=torch.float32).pin_memory()
    h2d = packed[0].numel()
    d2h = ho.numel() * 4
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        c = caches[i % copies]
        if L == 1:
            c.step_host_packed(0, packed[i % bank], with_ids, ho[0], stream=stream)
        else:
            c.step_layers_host_packed(0, L, packed[i % bank], with_ids, ho, stream=stream)
    e1.record(stream)
    e1.synchronize()
    e2e_elapsed = e0.elapsed_time(e1) / 1e3
    e2e_value = e2e_steps * L * world / e2e_elapsed if e2e_steps else None
    for c in caches:
        c.check(stream)

    # algorithmic bytes of one decode launch (every layer at the timed
    # launches' lengths): resident K/V, q in, o out; a fused launch also reads
    # the new token's K, V and writes them into the window (1 KiB per layer,
    # sequence and kv head; the evicted row's move into the middle is not
    # counted)
    qo_bytes = L * B * w.num_q_heads * 128 * (2 + 4)
    if fused:
        alg_bytes = resident_step + qo_bytes + L * B * w.num_kv_heads * 1024
        kernel_s = elapsed / K                 # one launch per step
        kernel_timing = "the timed step graph: one fused append + decode launch per step, events around it"
        kernel_name = "decode_kernel (fused append)"
    else:
        alg_bytes = res_kernel + qo_bytes
        kernel_s = kdur
        kernel_timing = "graph of back-to-back decode launches over the rotating copies, events around it"
        kernel_name = "decode_kernel"
    peak, peak_kind = _peaks()
    achieved = alg_bytes / kernel_s / 1e9
    wkey = w.name if w.num_layers == S.WORKLOAD_BY_NAME[w.name].num_layers else f"{w.name}/{w.num_layers}L"
    # paged caches have entries of their own (their producer differs per tile)
    layout_key = "/paged" if paged else ""
    tkey = f"{_decode_source_hash()}:{wkey}{layout_key}:{args.kv}:{'fused' if fused else 'decode'}"
    traffic = NCU_TRAFFIC.get(tkey)
    traffic_scaled = traffic is None and tkey in NCU_TRAFFIC_RATIO
    if traffic_scaled:
        traffic = int(round(NCU_TRAFFIC_RATIO[tkey] * alg_bytes))

    line = {
        "metric": METRIC,
        "value": job_throughput(K, L, world, elapsed),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": elapsed / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if kvf == lkb.KV_BF16 else f"bf16 + {args.kv} (middle blocks)",
        "data": "synthetic (seeded K/V/q; LeanK masks from the library's mask builder on seeded importances)",
        "config": {
            **workload_config(w, args), "context_growth_max": growth,
            "steps_per_s": K * world / elapsed,
            "resident_bytes_per_call": int(resident_step // L),
            "effective_GBps": resident_step * K * world / elapsed / 1e9,
            "warmup_steps_run": warm_done,
            "step_mode": args.step,
            "launches_per_step": "one fused append + decode (all layers)" if fused
            else "append (all layers) + decode (all layers)",
            "cache_copies": copies, "l2_policy": "inputs larger than L2 (rotating cache copies)",
            "cuda_graph": True, "pdl": True, "parallelism": f"replicas x{world}",
            "clock_window": f"{load_reps} untimed decode-only graph replays ({load_reps * n_kg} launches), "
                            "then the timed steps",
            "decode_ctas": args.decode_ctas or "library default",
        },
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic,
            "traffic_source": None if traffic is None else
            ("the 4-layer ncu capture's DRAM bytes per algorithmic byte x this launch's algorithmic bytes"
             if traffic_scaled else "ncu capture"),
            "peak_source": peak_kind, "kernel": kernel_name,
            "kernel_ms": kernel_s * 1e3, "alg_bytes_per_launch": alg_bytes,
            "timed_launches": K if fused else reps * n_kg, "kernel_timing": kernel_timing,
            "decode_only_kernel_ms": kdur * 1e3,
            "decode_only_kernel_ms_isolated": kdur_isolated * 1e3,
        },
        "e2e": None if e2e_value is None else {
            "value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": e2e_steps},
        "gpu_launches": K if fused else 2 * K,
    }
    cs = clocks.summary()
    if cs is not None:
        line["clocks"] = cs
    return line


# ---------------------------------------------------------------------------
# the oracle (CPU)
# ---------------------------------------------------------------------------

class _OracleUnits:
    """The inputs of one workload's oracle units: one sequence of layer 0
    (its dense history, q, special flags) and its kv heads.  A unit is the
    decode of one (sequence, kv head); a call (the metric's unit) is
    batch x kv heads units."""

    def __init__(self, w_name, kv):
        from decode_attention_pruned_gb300 import synth as S
        from oracle import attention as OA
        from oracle import masks as OM
        from oracle import quant as OQ
        if kv == "bf16":
            self.head_fn = OA.decode_head
        else:
            self.head_fn = lambda *a: OQ.decode_head_quantized(*a, fmt=kv)
        w = S.WORKLOAD_BY_NAME[w_name]
        self.w = w
        self.N = w.context
        self.pol = S.make_policies(w)
        if w.prune_pct is None or w.budget == "choice64":
            masks = S.masks_with_counts(w, S.drawn_counts(w))
        else:
            alpha, elig = S.stage2_inputs(w, self.pol)
            masks = OM.top_s_prune(alpha, w.prune_pct, w.align, w.budget, elig)
        self.kept = [np.nonzero(masks[0, h])[0] for h in range(w.num_kv_heads)]
        spec = S.make_special_table(w)
        k, v = S.make_kv(w.scaled(batch=1), 0, self.N)           # one sequence of layer 0
        q = S.make_q(w.scaled(batch=1), 0, self.N - 1)
        self.K = k[0].float().numpy()
        self.V = v[0].float().numpy()
        self.Q = q[0].float().numpy()
        self.flags = spec[S.make_token_ids(w.scaled(batch=1), self.N)[0]].astype(bool) if len(spec) else None
        self.units_per_call = w.batch * w.num_kv_heads

    def run(self, u):
        w, G = self.w, self.w.group
        h = u % w.num_kv_heads
        self.head_fn(self.Q[h * G:(h + 1) * G], self.K[:, h], self.V[:, h], int(self.pol[0, h]), self.kept[h],
                     self.N, w.sink, w.local, w.local_only_window, self.flags)


def oracle_sample(w_name, budget_s, max_units=None, kv="bf16"):
    """Time the fp64 oracle on one core on (sequence, kv head) units of the
    workload's decode call until `budget_s` or `max_units`; returns (calls/s,
    units, s).  kv="int8" / "fp8": the oracle over the quantised middle (quantisation
    included)."""
    ou = _OracleUnits(w_name, kv)
    units, t0 = 0, time.perf_counter()
    while True:
        ou.run(units)
        units += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_units is not None and units >= max_units):
            break
    return units / el / ou.units_per_call, units, el


def _oracle_worker(w_name, kv, budget_s, max_units, start, ready, out):
    ou = _OracleUnits(w_name, kv)
    ou.run(0)                                      # first-touch warm-up
    ready.put(1)
    start.wait()
    units, t0 = 0, time.perf_counter()
    while True:
        ou.run(units)
        units += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_units is not None and units >= max_units):
            break
    out.put((units, el))


def oracle_sample_parallel(w_name, budget_s, workers, max_units=None, kv="bf16"):
    """The fp64 oracle on `workers` processes (one core each: one BLAS thread
    per process), all timed over the same window after their inputs are
    built; returns (calls/s of all workers, units, seconds).  Processes are
    spawned, never forked, so a CUDA context in the parent is not copied."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    start, ready, out = ctx.Event(), ctx.Queue(), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w_name, kv, budget_s, max_units, start, ready, out))
             for _ in range(workers)]
    for p in procs:
        p.start()
    for _ in procs:
        ready.get(timeout=600)
    start.set()
    res = [out.get(timeout=600 + 4 * budget_s) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    from decode_attention_pruned_gb300 import synth as S
    w = S.WORKLOAD_BY_NAME[w_name]
    units = sum(u for u, _ in res)
    el = max(e for _, e in res)
    rate = sum(u / e for u, e in res) / (w.batch * w.num_kv_heads)
    return rate, units, el


def host_cpu():
    """(CPU model, logical cores available to this process)."""
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    import platform
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    return model or platform.processor() or platform.machine(), cores


def cpu_baseline(w_name, budget_s, kv):
    """The oracle on every host core (the reported value) and on one core."""
    model, cores = host_cpu()
    v1, u1, e1 = oracle_sample(w_name, budget_s / 2, kv=kv)
    vn, un, en = oracle_sample_parallel(w_name, budget_s / 2, cores, kv=kv)
    return {
        "value": vn, "unit": UNIT, "cores": cores, "kind": "oracle",
        "sample": f"fp64 numpy oracle, (sequence, kv head) units of layer 0: {un} units on {cores} worker "
                  f"processes (one core each) in {en:.1f} s; calls/s = units/s / (batch x kv heads)",
        "cpu_model": model,
        "single_core": {"value": v1, "unit": UNIT, "cores": 1,
                        "sample": f"{u1} units on one core in {e1:.1f} s"},
    }


def workload_config(w, args):
    """The keys of `config` that define the workload (shared by both arms)."""
    return {
        "workload": w.name, "layers": w.num_layers, "batch": w.batch, "q_heads": w.num_q_heads,
        "kv_heads": w.num_kv_heads, "head_dim": 128, "context": w.context, "sink": w.sink, "local": w.local,
        "prune_pct": w.prune_pct, "mask_budget": w.budget,
        "cache_layout": "paged (128-row pages per width class)" if args.layout == "paged" else "contiguous",
        "middle_format": f"{args.kv} (complete 128-row blocks; per-channel K / per-token V scales)"
        if args.kv != "bf16" else "bf16",
    }


def run_reference(args):
    from decode_attention_pruned_gb300 import synth as S
    W, K = args.warmup, args.steps
    model, cores = host_cpu()
    workers = cores if args.reference_cores == 0 else args.reference_cores
    # a step is one (sequence, kv head) unit per worker process; the steps
    # stop at K or at the time budget, whichever comes first
    value, units, el = oracle_sample_parallel(args.workload, args.reference_budget, workers,
                                              max_units=max(1, K), kv=args.kv)
    steps = max(1, units // workers)
    sample = (f"fp64 numpy oracle on {workers} worker processes (one core each), one (sequence, kv head) unit of "
              f"layer 0 per worker and step: {units} units in {el:.1f} s (at most {K} steps, capped at "
              f"{args.reference_budget:.0f} s; the workers' inputs built and warmed before); calls/s = units/s / "
              f"(batch x kv heads)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": steps,
        "warmup": W, "ms_per_step": el / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(S.WORKLOAD_BY_NAME[args.workload], args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle", "sample": sample,
                         "cpu_model": model},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


# defaults per workload: (timed steps, warm-up steps, end-to-end steps); the
# timed region stays within a few seconds and the appends grow the context
# by about 1 % (the rotating copies of the 20 GB serving step are few)
DEFAULT_STEPS = {
    "tiny": (60000, 2000, 4000),
    "llama31_8b_layer": (60000, 2000, 4000),
    "serving_b64": (150, 10, 30),
    "qwen25_7b_long": (20000, 500, 2000),
    "fastgen_mix": (1000, 20, 200),
}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: per workload)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default: per workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="serving_b64", choices=sorted(DEFAULT_STEPS))
    ap.add_argument("--layout", default="contiguous", choices=["contiguous", "paged"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "int8", "fp8"])
    ap.add_argument("--decode-ctas", type=int, default=0, help="CTAs of a decode launch (0: the library's choice)")
    ap.add_argument("--step", default="auto", choices=["auto", "fused", "split"],
                    help="lk_step_layers mode: the library's choice, one fused launch, or append + decode")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run the workload's first LAYERS layers (0: all)")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--kernel-steps", type=int, default=2000)
    ap.add_argument("--cpu-budget", type=float, default=16.0,
                    help="seconds of oracle timing for cpu_baseline (half on one core, half on all)")
    ap.add_argument("--reference-budget", type=float, default=60.0)
    ap.add_argument("--reference-cores", type=int, default=0, help="oracle worker processes (0: every core)")
    ap.add_argument("--load-seconds", type=float, default=0.4,
                    help="untimed decode-only replays that load the GPU before the timed steps (0: none)")
    args = ap.parse_args(argv)
    d_steps, d_warm, d_e2e = DEFAULT_STEPS[args.workload]
    args.steps = d_steps if args.steps is None else args.steps
    args.warmup = d_warm if args.warmup is None else args.warmup
    args.e2e_steps = d_e2e if args.e2e_steps is None else args.e2e_steps
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    rank, local_rank, world = _rank_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_gpu(args, rank, local_rank, world)
    if rank == 0:
        if world == 1:
            line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_budget, args.kv) if args.cpu_budget > 0 \
                else None
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
