"""Host logic of bench.py without a GPU: the multi-replica aggregation (max of
the per-rank step times, sum of the per-rank work) over a gloo process group
with two ranks, the algorithmic work counts, and the recorded-traffic lookup."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from transformer_gqa_attention_qkv_gb300.inputs import DECODE_CONFIGS, PREFILL_CONFIGS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), BENCH_BACKEND="gloo")
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    t_max = bench.reduce_max(1.0 + r, w)           # rank 1 is the slow one
    work = bench.reduce_sum(10.0 * (r + 1), w)     # 10 + 20
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, t_max, work))


def test_replica_aggregation_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 2.0, 30.0), (1, 2, 2.0, 30.0)]


def test_single_process_needs_no_group():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.reduce_sum(3.5, 1) == 3.5


def test_algorithmic_counts():
    c = PREFILL_CONFIGS["qwen3_32b"]
    f = bench.prefill_flops(c)
    assert f["qkv"] == 2 * 16384 * 10240 * 5120
    assert f["oproj"] == 2 * 16384 * 5120 * 8192
    assert f["attn"] == 4 * 64 * 128 * (16384 * 16385 // 2)
    assert abs(f["total"] / 1e9 - 7490.7) < 0.5
    d = bench.decode_bytes(DECODE_CONFIGS["qwen3_8b_decode"])
    assert d["kv_read"] == 2 * 64 * 8 * 8193 * 128 * 2


def test_recorded_traffic_is_null_after_a_source_change(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    sha = bench.source_hash("k.cu")
    (tmp_path / "profiles" / "k_w.traffic.txt").write_text(f"dram_bytes_per_launch: 123\nsource_sha: {sha}\n")
    assert bench.recorded_traffic("k_w", ["k.cu"]) == 123
    src.write_text("kernel v2")
    assert bench.recorded_traffic("k_w", ["k.cu"]) is None


@pytest.mark.parametrize("rows", [["0", "1"]])
def test_clock_summary_parses_samples(rows):
    s = bench.ClockSampler(0)
    s.out = ("1965, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active\n"
             "2070, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Not Active\n")
    out = s.summary()
    assert out["sm_max_mhz"] == 2070 and out["samples"] == 2
    assert out["reasons"] == ["sw_power_cap"]
