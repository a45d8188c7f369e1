#!/usr/bin/env python3
"""Benchmark of the GQA attention layer forward on GB300.

Default workload: the Qwen3-32B-shaped prefill layer (B=1, S=16384, hidden
5120, 64 query heads, 8 KV heads, head_dim 128, QK-norm, RoPE theta 1e6,
causal), bf16 inputs resident in HBM.  One step = one full layer forward
(QKV projection + QK-norm + RoPE, causal GQA attention, o_proj + residual)
through gqa_attn_forward_ex.  Metric: algorithmic TFLOP/s (2*M*N*K per
projection, 4*d per visible (query head, query, key) pair) and its fraction of
the measured dense bf16 peak.  The same line carries the decode step
(Qwen3-8B shape, 64 sequences x 8192 cached tokens) in GB/s of algorithmic
bytes against the measured HBM bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the plain fp64 CPU oracle on the host cores (there is
no other implementation of this layer to compare against), on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn-layer fwd TFLOP/s & % bf16 peak (prefill); decode GB/s & % HBM peak"
CSRC = "transformer_gqa_attention_qkv_gb300/csrc/"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def prefill_flops(cfg):
    d = cfg.head_dim
    M = cfg.B * cfg.S
    qkv = 2 * M * (cfg.Hq + 2 * cfg.Hkv) * d * cfg.hidden
    pairs = cfg.S * (cfg.S + 1) // 2 if cfg.causal else cfg.S * cfg.S
    attn = 4 * cfg.B * cfg.Hq * d * pairs
    oproj = 2 * M * cfg.hidden * cfg.Hq * d
    return {"qkv": qkv, "attn": attn, "oproj": oproj, "total": qkv + attn + oproj}


def decode_bytes(cfg, kv_elem=2):
    """Algorithmic bytes of one decode step: each cached K/V entry read once
    (plus the new one), weights read once, x/out, q and the appended K/V.
    kv_elem: bytes per cache element (2 bf16, 1 E4M3)."""
    d, B = cfg.head_dim, cfg.B
    kv_read = 2 * B * cfg.Hkv * (cfg.cache_len + 1) * d * kv_elem
    weights = ((cfg.Hq + 2 * cfg.Hkv) * d * cfg.hidden + cfg.hidden * cfg.Hq * d) * 2
    act = 2 * B * cfg.hidden * 2 + 2 * B * cfg.Hkv * d * kv_elem
    return {"kv_read": kv_read, "weights": weights, "act": act, "total": kv_read + weights + act}


def source_hash(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(name, src_files):
    """dram bytes per launch recorded under profiles/ for a kernel, or None if
    the kernel's sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"{name}.traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha") != source_hash(*src_files):
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl) if v.lower() == "active"})
        loaded = [r[0] for r in rows if r[0] > 0.5 * r[1]] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- CPU oracle

def cpu_oracle_sample(cfg, tokens, seed):
    """Time the fp64 oracle on the first `tokens` positions of one sequence of
    the workload (all heads, all three stages).  Returns (flop/s, seconds,
    threads, description)."""
    import oracle
    from transformer_gqa_attention_qkv_gb300.inputs import make_layer_inputs
    sub = cfg.with_(B=1, S=tokens)
    t = make_layer_inputs(sub, seed=seed)
    threads = oracle.default_threads()
    oracle.build()
    t0 = time.perf_counter()
    oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], sub.rope_theta, sub.eps,
                   sub.B, sub.S, sub.hidden, sub.Hq, sub.Hkv, sub.head_dim, causal=sub.causal, threads=threads)
    dt = time.perf_counter() - t0
    fl = prefill_flops(sub)["total"]
    desc = f"fp64 oracle, whole layer, first {tokens} tokens of one {cfg.name} sequence ({fl / 1e9:.1f} GFLOP)"
    return fl / dt, dt, threads, desc


# --------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value, world, device=None):
    """max over ranks of a float (the slowest rank defines the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, world, device=None):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------- our arm

def _r(x, n=4):
    return None if x is None else round(x, n)


def run_ours(args, world, rank, local):
    import torch

    from transformer_gqa_attention_qkv_gb300 import binding as gq
    from transformer_gqa_attention_qkv_gb300.inputs import (DECODE_CONFIGS, PREFILL_CONFIGS, SEEDS,
                                                            make_decode_inputs, make_layer_inputs)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # a stream of our own (not the legacy default stream, which synchronises
    # implicitly with every blocking stream in the process)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    cfg = PREFILL_CONFIGS[args.workload]
    fl = prefill_flops(cfg)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    launches = 0

    def check_dev():
        if gq.gqa_check_device_error() != 0:
            raise RuntimeError("device error word set: " + gq.gqa_last_error())

    def time_it(fn, count=True):
        """Mean CUDA-event time (ms) of fn over args.steps launches after
        args.warmup, L2 flushed before each.  fn may return the launches of the
        entry points it called before its last one (the last one's count is
        read after it)."""
        nonlocal launches
        ts = []
        for i in range(args.warmup + args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush.zero_()
            e0.record(stream)
            earlier = fn() or 0
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                ts.append(e0.elapsed_time(e1))
                if count:
                    launches += earlier + gq.gqa_last_launch_count()
        return statistics.mean(ts)

    def layer_setup(c, seed_extra=0):
        t = make_layer_inputs(c, seed=SEEDS[c.name] + seed_extra + 7919 * rank, device=str(dev))
        out = torch.empty_like(t["x"])
        ws = gq.new_workspace(gq.gqa_attn_workspace_size(c.B, c.S, c.hidden, c.Hq, c.Hkv, c.head_dim), dev)

        def fwd():
            gq.gqa_attn_forward_ex(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], c.rope_theta, c.eps,
                                   c.B, c.S, c.hidden, c.Hq, c.Hkv, c.head_dim, c.causal, out, ws, stream)
        return t, out, ws, fwd

    def stage_times(c, t, out, ws):
        """The layer's three kernels launched one by one on the same stream
        (Q, K, V and attn in the layer's own workspace layout), CUDA events
        between them: mean ms per stage.  Each iteration follows 50 ms of
        idle time, so every kernel is timed alone at the clocks a single
        launch gets (back-to-back iterations settle under the power cap within
        ~50 ms, and the per-kernel roofline divides by the burst peak)."""
        d = c.head_dim
        n_q, n_kv = c.B * c.S * c.Hq * d * 2, c.B * c.S * c.Hkv * d * 2
        al = lambda x: (x + 255) // 256 * 256  # noqa: E731
        q = ws[:n_q].view(torch.float16)
        k = ws[al(n_q):al(n_q) + n_kv].view(torch.float16)
        v = ws[al(n_q) + al(n_kv):al(n_q) + al(n_kv) + n_kv].view(torch.float16)
        o0 = al(n_q) + 2 * al(n_kv)
        attn = ws[o0:o0 + n_q].view(torch.bfloat16)
        acc = {"qkv": [], "attn": [], "oproj": []}
        for i in range(args.warmup + args.steps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            time.sleep(0.05)
            flush.zero_()
            e[0].record(stream)
            gq.gqa_qkv_proj(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], c.rope_theta, c.eps, c.B, c.S,
                            c.hidden, c.Hq, c.Hkv, d, q, k, v, stream)
            e[1].record(stream)
            gq.gqa_attention(q, k, v, c.B, c.S, c.Hq, c.Hkv, d, c.causal, attn, stream)
            e[2].record(stream)
            gq.gqa_oproj_residual(attn, t["Wo"], t["x"], c.B * c.S, c.hidden, c.Hq * d, out, stream)
            e[3].record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                for j, s in enumerate(("qkv", "attn", "oproj")):
                    acc[s].append(e[j].elapsed_time(e[j + 1]))
        check_dev()
        return {s: statistics.mean(x) for s, x in acc.items()}

    # ---- headline: the prefill layer forward (inputs generated on the device, seeded; larger than L2)
    t, out, ws, fwd = layer_setup(cfg)
    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    check_dev()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # clocks are sampled from here to the end of the last timed loop (decode)
    clk = ClockSampler(local).__enter__()
    time.sleep(0.25)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()  # evict L2 between steps (outside the events)
        ev[i][0].record(stream)
        fwd()
        launches += gq.gqa_last_launch_count()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(step_ms)
    ms_job = reduce_max(ms, world, dev)
    value = reduce_sum(fl["total"], world, dev) / (ms_job * 1e-3) / 1e12
    check_dev()

    # ---- per-kernel durations of the headline workload (roofline of the dominant kernel)
    kern = stage_times(cfg, t, out, ws)
    dom = max(kern, key=lambda s: kern[s])
    dom_src = {"attn": [CSRC + "attention.cu", CSRC + "ptx.cuh"],
               "qkv": [CSRC + "gemm.cu", CSRC + "ptx.cuh"],
               "oproj": [CSRC + "gemm.cu", CSRC + "ptx.cuh"]}[dom]
    achieved = fl[dom] / (kern[dom] * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                "peak_source": f"{peak_src} bf16 dense burst (binary16 shares the rate); each launch timed "
                                  "alone after 50 ms idle",
                "traffic": recorded_traffic(f"{dom}_{cfg.name}", dom_src)}
    configs = {cfg.name: {"tflops": round(value, 1), "frac": round(value / world / peak_tf, 4), "ms": _r(ms_job),
                          "stage_ms": [_r(kern[s]) for s in ("qkv", "attn", "oproj")],
                          "stage_tflops": [round(fl[s] / (kern[s] * 1e-3) / 1e12, 1)
                                           for s in ("qkv", "attn", "oproj")]}}

    # ---- e2e: through the C-ABI entry point that takes host buffers (pinned x in,
    # out back); its copies run inside the timed region, overlapped with compute
    x_host = t["x"].cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    hws = gq.new_workspace(gq.gqa_attn_forward_host_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv,
                                                                   cfg.head_dim), dev)

    def fwd_e2e():
        gq.gqa_attn_forward_host(x_host, t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta,
                                 cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, cfg.causal,
                                 out_host, hws, stream)

    for _ in range(max(1, args.warmup)):
        fwd_e2e()
    torch.cuda.synchronize()
    barrier(world)
    ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ee[i][0].record(stream)
        fwd_e2e()
        ee[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(statistics.mean(a.elapsed_time(b) for a, b in ee), world, dev)
    e2e = {"value": round(reduce_sum(fl["total"], world, dev) / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": x_host.numel() * 2,
           "d2h_bytes_per_step": out_host.numel() * 2}
    check_dev()
    del t, out, ws, x_host, out_host, hws
    torch.cuda.empty_cache()

    # ---- the other prefill workloads: whole layer, then its kernels one by one
    for name in ("qwen3_0p6b", "vaswani_mha", "qwen3_4b"):
        if name == cfg.name:
            continue
        c = PREFILL_CONFIGS[name]
        cf = prefill_flops(c)
        ct, cout, cws, cfwd = layer_setup(c)
        cms = reduce_max(time_it(cfwd), world, dev)
        ck = stage_times(c, ct, cout, cws)
        configs[name] = {"tflops": round(reduce_sum(cf["total"], world, dev) / (cms * 1e-3) / 1e12, 1),
                         "frac": round(cf["total"] / (cms * 1e-3) / 1e12 / peak_tf, 4), "ms": _r(cms),
                         "stage_ms": [_r(ck[s]) for s in ("qkv", "attn", "oproj")],
                         "stage_tflops": [round(cf[s] / (ck[s] * 1e-3) / 1e12, 1) for s in ("qkv", "attn", "oproj")]}
        del ct, cout, cws
    torch.cuda.empty_cache()

    # ---- decode step
    dc = DECODE_CONFIGS["qwen3_8b_decode"]
    db = decode_bytes(dc)
    dt_ = make_decode_inputs(dc, seed=SEEDS[dc.name] + 7919 * rank, device=str(dev))
    dout = torch.empty_like(dt_["x"])
    dws = gq.new_workspace(gq.gqa_attn_decode_workspace_size(dc.B, dc.hidden, dc.Hq, dc.Hkv, dc.head_dim,
                                                             dc.lmax), dev)

    def dec():
        gq.gqa_attn_decode(dt_["x"], dt_["Wqkv"], dt_["Wo"], dt_["q_norm_w"], dt_["k_norm_w"], dc.rope_theta,
                           dc.eps, dc.B, dc.hidden, dc.Hq, dc.Hkv, dc.head_dim, dt_["k_cache"], dt_["v_cache"],
                           dt_["cache_len"], dc.lmax, dout, dws, stream)

    barrier(world)
    dms = reduce_max(time_it(dec), world, dev)
    clk.__exit__(None, None, None)
    # decode attention kernel alone (split + combine), for its roofline: a query
    # of unit-RMS rows (as QK-norm leaves them), so scores and the running max
    # move as in the real step
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEEDS[dc.name] + 3)
    qd = torch.randn((dc.B, dc.Hq, dc.head_dim), generator=gen, device=dev).to(torch.float16)
    ad = torch.empty((dc.B, dc.Hq * dc.head_dim), dtype=torch.bfloat16, device=dev)
    kl = (dt_["cache_len"] + 1).to(torch.int32)
    aws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(dc.B, dc.Hq, dc.Hkv, dc.head_dim, dc.lmax),
                           dev)
    ams = time_it(lambda: gq.gqa_decode_attention(qd, dt_["k_cache"], dt_["v_cache"], kl, dc.B, dc.Hq, dc.Hkv,
                                                  dc.head_dim, dc.lmax, ad, aws, stream), count=False)
    attn_bytes = db["kv_read"] + dc.B * dc.Hq * dc.head_dim * 2 * 2
    dec_ach = attn_bytes / (ams * 1e-3) / 1e9
    decode = {"workload": dc.name, "value": round(reduce_sum(db["total"], world, dev) / (dms * 1e-3) / 1e9, 1),
              "unit": "GB/s", "ms": _r(dms), "frac": round(db["total"] / (dms * 1e-3) / 1e9 / hbm, 4),
              "bytes": db["total"],
              "kernel": {"name": "decode_attention", "achieved": round(dec_ach, 1), "frac": round(dec_ach / hbm, 4),
                         "ms": _r(ams),
                         "traffic": recorded_traffic("decode_attention_" + dc.name,
                                                     [CSRC + "decode.cu", CSRC + "ptx.cuh"])}}
    check_dev()

    # ---- the same decode step over E4M3 caches (scale 2^-5: the N(0,1)
    # cache entries land well inside E4M3's range)
    f8s = 2.0 ** -5
    kc8 = (dt_["k_cache"].float() / f8s).to(torch.float8_e4m3fn).view(torch.uint8)
    vc8 = (dt_["v_cache"].float() / f8s).to(torch.float8_e4m3fn).view(torch.uint8)
    del dt_["k_cache"], dt_["v_cache"]
    db8 = decode_bytes(dc, kv_elem=1)

    def dec8():
        gq.gqa_attn_decode_fp8(dt_["x"], dt_["Wqkv"], dt_["Wo"], dt_["q_norm_w"], dt_["k_norm_w"], dc.rope_theta,
                               dc.eps, dc.B, dc.hidden, dc.Hq, dc.Hkv, dc.head_dim, kc8, vc8, f8s, f8s,
                               dt_["cache_len"], dc.lmax, dout, dws, stream)

    d8ms = reduce_max(time_it(dec8), world, dev)
    a8ms = time_it(lambda: gq.gqa_decode_attention_fp8(qd, kc8, vc8, f8s, f8s, kl, dc.B, dc.Hq, dc.Hkv,
                                                        dc.head_dim, dc.lmax, ad, aws, stream), count=False)
    a8_ach = (db8["kv_read"] + dc.B * dc.Hq * dc.head_dim * 2 * 2) / (a8ms * 1e-3) / 1e9
    decode_fp8 = {"value": round(reduce_sum(db8["total"], world, dev) / (d8ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                  "ms": _r(d8ms), "frac": round(db8["total"] / (d8ms * 1e-3) / 1e9 / hbm, 4),
                  "speedup_vs_bf16": round(dms / d8ms, 3),
                  "kernel": {"name": "decode_attention_fp8", "achieved": round(a8_ach, 1),
                             "frac": round(a8_ach / hbm, 4), "ms": _r(a8ms),
                             "traffic": recorded_traffic("decode_attention_fp8_" + dc.name,
                                                         [CSRC + "decode.cu", CSRC + "ptx.cuh"])}}
    check_dev()
    del dt_, dout, dws, kc8, vc8, aws
    torch.cuda.empty_cache()

    details = {}
    # ---- chunked prefill: the last 2048 tokens of a 16384-token Qwen3-32B context
    if not args.no_chunk:
        cc = PREFILL_CONFIGS["qwen3_32b"].with_(S=2048)
        p0, Lmax = 14336, 16384
        ct = make_layer_inputs(cc, seed=SEEDS["qwen3_32b"] + 17 + 7919 * rank, device=str(dev))
        gen.manual_seed(SEEDS["qwen3_32b"] + 18)
        kc = torch.randn((1, cc.Hkv, Lmax, cc.head_dim), generator=gen, device=dev).to(torch.bfloat16)
        vc = torch.randn((1, cc.Hkv, Lmax, cc.head_dim), generator=gen, device=dev).to(torch.bfloat16)
        cl = torch.full((1,), p0, dtype=torch.int32, device=dev)
        cout = torch.empty_like(ct["x"])
        cws = gq.new_workspace(gq.gqa_attn_prefill_cached_workspace_size(1, cc.S, cc.Hq, cc.Hkv, cc.head_dim, Lmax), dev)
        cf = (2 * cc.S * (cc.Hq + 2 * cc.Hkv) * cc.head_dim * cc.hidden
              + 4 * cc.Hq * cc.head_dim * (cc.S * p0 + cc.S * (cc.S + 1) // 2)
              + 2 * cc.S * cc.hidden * cc.Hq * cc.head_dim)

        def chunk_step():
            gq.gqa_attn_prefill_cached(ct["x"], ct["Wqkv"], ct["Wo"], ct["q_norm_w"], ct["k_norm_w"], cc.rope_theta,
                                       cc.eps, 1, cc.S, cc.hidden, cc.Hq, cc.Hkv, cc.head_dim, True, kc, vc, cl,
                                       Lmax, cout, cws, stream)

        cms = reduce_max(time_it(chunk_step), world, dev)
        details["chunked_prefill"] = {"workload": "qwen3_32b, 2048 new tokens after 14336 cached",
                                      "tflops": round(reduce_sum(cf, world, dev) / (cms * 1e-3) / 1e12, 1),
                                      "frac": round(cf / (cms * 1e-3) / 1e12 / peak_tf, 4), "ms": _r(cms)}
        check_dev()
        del ct, kc, vc, cout, cws

    # ---- other head widths: 256 at the Gemma-3 example's width, 80 and 96 at
    # the Qwen3-4B widths (4 x 4096 tokens each): the layer, then its attention alone
    if not args.no_widths:
        for name in ("gemma3_d256", "qwen3_4b_d80", "knob_d96"):
            wc = PREFILL_CONFIGS[name]
            wf = prefill_flops(wc)
            wt, wout, wws, wstep = layer_setup(wc)
            wms = reduce_max(time_it(wstep), world, dev)
            wk = stage_times(wc, wt, wout, wws)
            details[name] = {"tflops": round(reduce_sum(wf["total"], world, dev) / (wms * 1e-3) / 1e12, 1),
                             "frac": round(wf["total"] / (wms * 1e-3) / 1e12 / peak_tf, 4), "ms": _r(wms),
                             "stage_ms": [_r(wk[s]) for s in ("qkv", "attn", "oproj")],
                             "attn_frac": round(wf["attn"] / (wk["attn"] * 1e-3) / 1e12 / peak_tf, 4)}
            del wt, wout, wws

    # ---- backward of the headline layer: gradients of x, Wqkv, Wo and the norm weights
    if not args.no_bwd:
        bt = make_layer_inputs(cfg, seed=SEEDS[cfg.name] + 29 + 7919 * rank, device=str(dev))
        gen.manual_seed(SEEDS[cfg.name] + 31)
        bdo = torch.randn((cfg.B * cfg.S, cfg.hidden), generator=gen, device=dev).to(torch.bfloat16)
        d_ = cfg.head_dim
        Nq = (cfg.Hq + 2 * cfg.Hkv) * d_
        bdx = torch.empty_like(bt["x"])
        bdW = torch.empty((Nq, cfg.hidden), dtype=torch.float32, device=dev)
        bdWo = torch.empty((cfg.hidden, cfg.Hq * d_), dtype=torch.float32, device=dev)
        bqn = torch.empty(d_, dtype=torch.float32, device=dev)
        bkn = torch.empty(d_, dtype=torch.float32, device=dev)
        bws = gq.new_workspace(gq.gqa_attn_backward_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, d_),
                               dev)
        bout = torch.empty_like(bt["x"])
        args_ = (bt["x"], bt["Wqkv"], bt["Wo"], bt["q_norm_w"], bt["k_norm_w"], cfg.rope_theta, cfg.eps, cfg.B,
                 cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, d_, cfg.causal)

        def bwd_step():
            gq.gqa_attn_backward(*args_, bdo, bdx, bdW, bdWo, bqn, bkn, bws, stream)

        def fwd_train():
            gq.gqa_attn_forward_train(*args_, bout, bws, stream)

        def bwd_saved():
            gq.gqa_attn_backward_saved(*args_, bdo, bdx, bdW, bdWo, bqn, bkn, bws, stream)

        def train_step():
            fwd_train()
            n = gq.gqa_last_launch_count()
            bwd_saved()
            return n

        bms = reduce_max(time_it(bwd_step), world, dev)
        fwd_train()
        sms_ = reduce_max(time_it(bwd_saved), world, dev)  # the saved inputs are read, not changed
        tms = reduce_max(time_it(train_step), world, dev)
        # algorithmic: each projection twice (input and weight gradients), attention 2.5x its forward
        bflops = 2 * (fl["qkv"] + fl["oproj"]) + 5 * fl["attn"] // 2
        details["backward"] = {
            "workload": cfg.name, "tflops": round(reduce_sum(bflops, world, dev) / (bms * 1e-3) / 1e12, 1),
            "frac": round(bflops / (bms * 1e-3) / 1e12 / peak_tf, 4), "ms": _r(bms),
            "from_saved_ms": _r(sms_), "from_saved_frac": round(bflops / (sms_ * 1e-3) / 1e12 / peak_tf, 4),
            "train_step_ms": _r(tms),
            "train_step_frac": round((bflops + fl["total"]) / (tms * 1e-3) / 1e12 / peak_tf, 4)}
        check_dev()
        del bt, bdo, bdx, bdW, bdWo, bws, bout

    # ---- CPU baseline (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        fls, secs, threads, desc = cpu_oracle_sample(cfg, args.cpu_tokens, SEEDS[cfg.name])
        cpu = {"value": round(fls / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": round(secs, 2)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_job, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in/out, binary16 Q/K/V/P, fp32 accumulate", "data": "synthetic",
        "frac_of_peak": round(value / world / peak_tf, 4),
        "config": {"workload": cfg.name, "B": cfg.B, "S": cfg.S, "hidden": cfg.hidden, "Hq": cfg.Hq,
                   "Hkv": cfg.Hkv, "head_dim": cfg.head_dim, "qk_norm": cfg.qk_norm, "rope_theta": cfg.rope_theta,
                   "causal": cfg.causal, "flops_per_step": fl["total"], "parallelism": f"replicas x{world}",
                   "l2": "flushed before every timed launch"},
        "roofline": roofline, "configs": configs, "decode": decode, "decode_fp8": decode_fp8,
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": launches, "clocks": clk.summary(),
    }
    if rank == 0:
        # the per-workload extras on stderr, the one benchmark line last on stdout
        print("bench details: " + json.dumps({"step_ms": [round(x, 3) for x in step_ms], "wall_s": round(wall, 3),
                                              **details}), file=sys.stderr, flush=True)
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    """The fp64 CPU oracle, as it stands, on the host cores; each step is a
    bounded sample (a prefix of one sequence) of the same workload."""
    if rank != 0:
        return
    from transformer_gqa_attention_qkv_gb300.inputs import PREFILL_CONFIGS, SEEDS
    cfg = PREFILL_CONFIGS[args.workload]
    for _ in range(args.warmup):
        cpu_oracle_sample(cfg, args.ref_tokens, SEEDS[cfg.name])
    rates, secs = [], []
    for _ in range(args.steps):
        r, s, threads, desc = cpu_oracle_sample(cfg, args.ref_tokens, SEEDS[cfg.name])
        rates.append(r)
        secs.append(s)
    value = statistics.mean(rates) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.mean(secs), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{cfg.name}, first {args.ref_tokens} tokens of one sequence", "B": 1,
                       "S": args.ref_tokens, "hidden": cfg.hidden, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
                       "head_dim": cfg.head_dim, "causal": cfg.causal, "parallelism": "host cores"},
            "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": desc, "value": round(value, 6),
                             "unit": "TFLOP/s"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_stage(args, local):
    """Launch one stage alone, warmup + steps times, and print its mean time.
    Used for profiler captures of a single kernel (not a benchmark line)."""
    import torch

    from transformer_gqa_attention_qkv_gb300 import binding as gq
    from transformer_gqa_attention_qkv_gb300.inputs import (DECODE_CONFIGS, PREFILL_CONFIGS, SEEDS,
                                                            make_decode_inputs, make_layer_inputs)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    if args.stage in ("decode_attn", "decode_attn_fp8"):
        dc = DECODE_CONFIGS["qwen3_8b_decode"]
        t = make_decode_inputs(dc, seed=SEEDS[dc.name], device=str(dev))
        q = torch.randn((dc.B, dc.Hq, dc.head_dim), device=dev).to(torch.float16)
        a = torch.empty((dc.B, dc.Hq * dc.head_dim), dtype=torch.bfloat16, device=dev)
        kl = (t["cache_len"] + 1).to(torch.int32)
        ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(dc.B, dc.Hq, dc.Hkv, dc.head_dim, dc.lmax), dev)
        f8s = 2.0 ** -5
        if args.stage == "decode_attn_fp8":
            t["k_cache"] = (t["k_cache"].float() / f8s).to(torch.float8_e4m3fn).view(torch.uint8)
            t["v_cache"] = (t["v_cache"].float() / f8s).to(torch.float8_e4m3fn).view(torch.uint8)

        def go():
            if args.stage == "decode_attn_fp8":
                gq.gqa_decode_attention_fp8(q, t["k_cache"], t["v_cache"], f8s, f8s, kl, dc.B, dc.Hq, dc.Hkv,
                                            dc.head_dim, dc.lmax, a, ws, stream)
            else:
                gq.gqa_decode_attention(q, t["k_cache"], t["v_cache"], kl, dc.B, dc.Hq, dc.Hkv, dc.head_dim,
                                        dc.lmax, a, ws, stream)
        name = dc.name
    else:
        cfg = PREFILL_CONFIGS[args.workload]
        t = make_layer_inputs(cfg, seed=SEEDS[cfg.name], device=str(dev))
        d = cfg.head_dim
        q = torch.empty((cfg.B, cfg.Hq, cfg.S, d), dtype=torch.float16, device=dev)
        k = torch.empty((cfg.B, cfg.Hkv, cfg.S, d), dtype=torch.float16, device=dev)
        v = torch.empty_like(k)
        attn = torch.empty((cfg.B * cfg.S, cfg.Hq * d), dtype=torch.bfloat16, device=dev)
        out = torch.empty_like(t["x"])
        gq.gqa_qkv_proj(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps, cfg.B, cfg.S,
                        cfg.hidden, cfg.Hq, cfg.Hkv, d, q, k, v, stream)
        gq.gqa_attention(q, k, v, cfg.B, cfg.S, cfg.Hq, cfg.Hkv, d, cfg.causal, attn, stream)
        if args.stage == "layer_bwd":
            dout_ = torch.randn((cfg.B * cfg.S, cfg.hidden), device=dev).to(torch.bfloat16)
            ldx = torch.empty_like(t["x"])
            ldW = torch.empty(((cfg.Hq + 2 * cfg.Hkv) * d, cfg.hidden), dtype=torch.float32, device=dev)
            ldWo = torch.empty((cfg.hidden, cfg.Hq * d), dtype=torch.float32, device=dev)
            lqn = torch.empty(d, dtype=torch.float32, device=dev) if cfg.qk_norm else None
            lkn = torch.empty(d, dtype=torch.float32, device=dev) if cfg.qk_norm else None
            lws = gq.new_workspace(gq.gqa_attn_backward_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, d),
                                   dev)
        if args.stage == "attn_bwd":
            g_ = torch.randn_like(q, dtype=torch.float32).to(torch.float16)
            dq_ = torch.empty(q.shape, dtype=torch.float32, device=dev)
            dk_ = torch.empty(k.shape, dtype=torch.float32, device=dev)
            dv_ = torch.empty_like(dk_)
            bws_ = gq.new_workspace(gq.gqa_attention_backward_workspace_size(cfg.B, cfg.S, cfg.Hq, d), dev)

        def go():
            if args.stage == "layer_bwd":
                gq.gqa_attn_backward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                     cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, d, cfg.causal, dout_, ldx, ldW, ldWo,
                                     lqn, lkn, lws, stream)
            elif args.stage == "attn_bwd":
                gq.gqa_attention_backward(q, k, v, g_, cfg.B, cfg.S, cfg.Hq, cfg.Hkv, d, cfg.causal, dq_, dk_, dv_,
                                          bws_, stream)
            elif args.stage == "qkv":
                gq.gqa_qkv_proj(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps, cfg.B,
                                cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, d, q, k, v, stream)
            elif args.stage == "attn":
                gq.gqa_attention(q, k, v, cfg.B, cfg.S, cfg.Hq, cfg.Hkv, d, cfg.causal, attn, stream)
            else:
                gq.gqa_oproj_residual(attn, t["Wo"], t["x"], cfg.B * cfg.S, cfg.hidden, cfg.Hq * d, out, stream)
        name = cfg.name
    torch.cuda.synchronize()
    ms = []
    for i in range(args.warmup + args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        go()
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            ms.append(e0.elapsed_time(e1))
    if gq.gqa_check_device_error() != 0:
        raise RuntimeError(gq.gqa_last_error())
    print(json.dumps({"stage": args.stage, "workload": name, "ms": round(statistics.mean(ms), 4) if ms else None}))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_32b")
    ap.add_argument("--cpu-tokens", type=int, default=2048, help="tokens of the CPU-baseline sample")
    ap.add_argument("--ref-tokens", type=int, default=256, help="tokens per reference-arm step")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-chunk", action="store_true", help="skip the chunked-prefill measurement")
    ap.add_argument("--no-widths", "--no-d256", dest="no_widths", action="store_true",
                    help="skip the head_dim 256 / 80 / 96 measurements")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward measurement")
    ap.add_argument("--stage", choices=["qkv", "attn", "oproj", "decode_attn", "decode_attn_fp8", "attn_bwd",
                                            "layer_bwd"], default=None,
                    help="launch one stage alone (for profiler captures); prints its time, no benchmark line")
    args = ap.parse_args(argv)
    world, rank, local = dist_setup(args.gpus)
    if args.stage:
        run_stage(args, local)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
