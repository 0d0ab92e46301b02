"""Host-side checks of bench.py: the multi-rank reduction over gloo (CPU,
world size 2) and the reference arm's JSON line (the oracle on the CPU)."""
import contextlib
import io
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.0 + rank, dist, torch.device("cpu"))
        out[rank] = (t, bench.job_throughput(100, 1, world, t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0][0] == out[1][0] == 2.0
    assert out[0][1] == pytest.approx(100 * 2 / 2.0)


def test_reference_arm_prints_contract_line(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "4", "--warmup", "3", "--workload", "tiny",
                         "--reference-budget", "2", "--reference-cores", "2"])
    assert rc == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "calls/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 2
    assert line["cpu_baseline"]["cpu_model"]
    assert line["steps"] == 4
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_default_workload_is_the_largest_single_gpu_one():
    from decode_attention_pruned_gb300 import synth as S
    sizes = {w.name: w.num_layers * w.batch * w.num_kv_heads * w.context for w in S.WORKLOADS}
    assert sizes["serving_b64"] == max(sizes.values())
    ap_default = bench.DEFAULT_STEPS["serving_b64"]
    assert ap_default[1] >= 3
    model, cores = bench.host_cpu()
    assert model and cores >= 1


def test_reference_arm_nonzero_rank_is_silent(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "tiny"])
    assert rc == 0 and buf.getvalue() == ""


def test_oracle_rate_counts_layer_calls():
    """A call is one layer's decode attention (every sequence and kv head),
    as in the GPU arm's value (steps x layers / s): a 32-layer workload's
    oracle rate is not divided by its layers."""
    from decode_attention_pruned_gb300 import synth as S
    w = S.WORKLOAD_BY_NAME["serving_b64"]
    value, units, el = bench.oracle_sample("serving_b64", 0.0, max_units=1)
    assert units == 1
    assert value == pytest.approx(units / el / (w.batch * w.num_kv_heads))
    assert bench.job_throughput(10, w.num_layers, 1, 2.0) == pytest.approx(10 * w.num_layers / 2.0)


def test_traffic_table_is_current_and_self_consistent():
    """The DRAM traffic the bench reports comes from captures of the kernel
    sources as they stand (every key carries their hash), and each 32-layer
    ratio is the matching 4-layer capture's traffic over a whole number of
    algorithmic bytes, just above one."""
    from decode_attention_pruned_gb300 import synth as S
    h = bench._decode_source_hash()
    keys = list(bench.NCU_TRAFFIC) + list(bench.NCU_TRAFFIC_RATIO)
    assert keys and all(k.split(":")[0] == h for k in keys), "kernel sources changed since the captures"
    for k in keys:
        _, wl, kv, mode = k.split(":")
        assert wl.split("/")[0] in S.WORKLOAD_BY_NAME
        assert kv in ("bf16", "int8", "fp8") and mode in ("fused", "decode")
    for k, ratio in bench.NCU_TRAFFIC_RATIO.items():
        _, wl, kv, mode = k.split(":")
        name, *rest = wl.split("/")
        assert S.WORKLOAD_BY_NAME[name].num_layers > 4
        cut = ":".join([h, "/".join([name, "4L", *rest]), kv, mode])
        assert cut in bench.NCU_TRAFFIC, cut
        alg4 = bench.NCU_TRAFFIC[cut] / ratio
        assert abs(alg4 - round(alg4)) < 1e-3
        assert 1.0 <= ratio < 1.05
