"""Parity of the CUDA path with the fp64 oracle, prefill (GPU).

Each stage is checked alone on the GPU's own inputs to that stage (so one
stage's rounding does not hide another's error), then the whole layer end to
end.  Shapes span several tiles and ragged tails in every dimension (tokens,
output features, the contraction, keys), the degenerate cases (one token, one
KV head, G = 1 and G = 16), the five workload geometries at reduced length with
the full oracle, and the full-size workloads on sampled rows.

Tolerance: max|err| <= 1e-2 max|ref| and relative L1 <= 2e-3 (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import (PREFILL_CONFIGS, SEEDS, LayerConfig,
                                                        make_layer_inputs, sample_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dev(t):
    return None if t is None else t.to(DEV)


def bf16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.bfloat16)


def f16_randn(shape, gen, std=1.0):
    """Q/K/V of the attention stage are binary16 (see include/gqa_attn.h)."""
    return (torch.randn(*shape, generator=gen) * std).to(torch.float16)


# ----------------------------------------------------------------- stage 1

QKV_CASES = [
    # B, S, hidden, Hq, Hkv, d, qk_norm
    (1, 128, 1024, 16, 8, 128, True),   # Qwen3-0.6B geometry
    (2, 300, 256, 4, 2, 128, True),     # ragged token count, 4 output tiles
    (3, 77, 200, 2, 1, 64, False),      # contraction tail (200 = 3*64 + 8), d=64, no QK-norm
    (1, 1, 512, 8, 8, 64, True),        # a single token
    (2, 130, 384, 3, 1, 128, True),     # output width 640: a half tile at the end
]


@pytest.mark.parametrize("B,S,hidden,Hq,Hkv,d,qk", QKV_CASES)
def test_qkv_projection_stage(B, S, hidden, Hq, Hkv, d, qk):
    cfg = LayerConfig("t", B, S, hidden, Hq, Hkv, d, qk, 1e4 if d == 64 else 1e6)
    t = make_layer_inputs(cfg, seed=100 + S, w_std=0.05)
    q = torch.empty((B, Hq, S, d), dtype=torch.float16, device=DEV)
    k = torch.empty((B, Hkv, S, d), dtype=torch.float16, device=DEV)
    v = torch.empty_like(k)
    gq.gqa_qkv_proj(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
                    cfg.eps, B, S, hidden, Hq, Hkv, d, q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    rq, rk, rv = oracle.qkv_stage(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                  B, S, hidden, Hq, Hkv, d)
    assert_parity("Q", to64(q), rq)
    assert_parity("K", to64(k), rk)
    assert_parity("V", to64(v), rv)


# ----------------------------------------------------------------- stage 2

ATTN_CASES = [
    # B, S, Hq, Hkv, d, causal
    (1, 128, 16, 8, 128, True),    # Qwen3-0.6B heads, G=2
    (2, 300, 8, 1, 128, True),     # MQA-like G=8, ragged, crosses key tiles
    (1, 129, 4, 4, 64, True),      # G=1, one key past a tile
    (2, 7, 4, 2, 128, True),
    (1, 1, 2, 1, 64, True),        # a single token
    (1, 1000, 32, 8, 128, True),   # Qwen3-4B/8B heads, G=4
    (2, 300, 8, 2, 64, False),     # no mask
    (1, 257, 16, 1, 128, True),    # G=16
    (3, 520, 8, 8, 64, True),      # Vaswani heads
]


@pytest.mark.parametrize("B,S,Hq,Hkv,d,causal", ATTN_CASES)
def test_attention_stage(B, S, Hq, Hkv, d, causal):
    g = torch.Generator().manual_seed(200 + S)
    Q = f16_randn((B, Hq, S, d), g, 1.5)
    K = f16_randn((B, Hkv, S, d), g, 1.5)
    V = f16_randn((B, Hkv, S, d), g)
    out = torch.empty((B, S, Hq * d), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention(dev(Q), dev(K), dev(V), B, S, Hq, Hkv, d, causal, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.attention_stage(Q, K, V, B, S, Hq, Hkv, d, causal=causal)
    assert_parity("attn", to64(out).reshape(B * S, Hq * d), ref)


def test_attention_group_map_markers_gpu():
    """Distinguishable heads: every KV head's values are one constant marker,
    so each query head must return exactly its group's marker (g = j // G)."""
    B, S, Hq, Hkv, d = 2, 200, 16, 4, 128
    g = torch.Generator().manual_seed(5)
    markers = torch.arange(1, B * Hkv * d + 1, dtype=torch.float32).reshape(B, Hkv, 1, d) / (B * Hkv * d)
    V = markers.expand(B, Hkv, S, d).contiguous().to(torch.float16)
    Q = f16_randn((B, Hq, S, d), g)
    K = f16_randn((B, Hkv, S, d), g)
    out = torch.empty((B, S, Hq * d), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention(dev(Q), dev(K), dev(V), B, S, Hq, Hkv, d, True, out)
    torch.cuda.synchronize()
    o = to64(out).reshape(B, S, Hq, d)
    mk = to64(markers.to(torch.float16))
    for j in range(Hq):
        np.testing.assert_allclose(o[:, :, j], np.broadcast_to(mk[:, j // (Hq // Hkv)], (B, S, d)),
                                   rtol=1e-2, atol=0)


def test_attention_no_future_leak_gpu():
    """A huge value planted in V at position 700 leaves every earlier row
    bit-identical and changes every later row."""
    B, S, Hq, Hkv, d = 1, 1000, 8, 2, 128
    g = torch.Generator().manual_seed(6)
    Q = f16_randn((B, Hq, S, d), g)
    K = f16_randn((B, Hkv, S, d), g)
    V = f16_randn((B, Hkv, S, d), g)
    outs = []
    for spike in (False, True):
        V2 = V.clone()
        if spike:
            V2[:, :, 700] = 1000.0
        out = torch.empty((B, S, Hq * d), dtype=torch.bfloat16, device=DEV)
        gq.gqa_attention(dev(Q), dev(K), dev(V2), B, S, Hq, Hkv, d, True, out)
        outs.append(out.float().cpu())
    torch.cuda.synchronize()
    assert torch.equal(outs[0][:, :700], outs[1][:, :700])
    assert (outs[0][:, 700:] - outs[1][:, 700:]).abs().amax(dim=-1).min() > 1e-2


# ----------------------------------------------------------------- stage 3

OPROJ_CASES = [
    # M, hidden, q_width
    (128, 1024, 2048),   # Qwen3-0.6B o_proj 2048 -> 1024
    (300, 256, 512),
    (1, 512, 512),
    (77, 200, 128),      # output width 200: partial tile
    (64, 4096, 4096),    # decode-sized (one M block)
    (1000, 2560, 4096),  # Qwen3-4B o_proj 4096 -> 2560
]


@pytest.mark.parametrize("M,hidden,qw", OPROJ_CASES)
def test_oproj_residual_stage(M, hidden, qw):
    g = torch.Generator().manual_seed(300 + M)
    attn = bf16_randn((M, qw), g, 0.5)
    Wo = bf16_randn((hidden, qw), g, 0.05)
    x = bf16_randn((M, hidden), g)
    out = torch.empty((M, hidden), dtype=torch.bfloat16, device=DEV)
    gq.gqa_oproj_residual(dev(attn), dev(Wo), dev(x), M, hidden, qw, out)
    torch.cuda.synchronize()
    ref = oracle.oproj_stage(attn, Wo, x, M, hidden, qw)
    assert_parity("out", to64(out), ref)
    # the projection term alone, so the residual cannot hide an error in it; the
    # bound is looser because out is rounded to bf16 at the scale of |x + term|
    assert_parity("out - x", to64(out) - to64(x), ref - to64(x), tol_max=2e-2, tol_rel=1e-2)


# ----------------------------------------------------------------- the layer

def run_forward(cfg, t):
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim))
    gq.gqa_attn_forward_ex(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                           cfg.rope_theta, cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                           cfg.causal, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    return out, ws


def ws_views(cfg, ws):
    """Q, K, V, attn inside the workspace (layout of gqa_attn_workspace_size)."""
    def al(x):
        return (x + 255) // 256 * 256
    tok = cfg.B * cfg.S
    d = cfg.head_dim
    sizes = [tok * cfg.Hq * d * 2, tok * cfg.Hkv * d * 2, tok * cfg.Hkv * d * 2, tok * cfg.Hq * d * 2]
    offs = np.cumsum([0] + [al(s) for s in sizes])
    dts = [torch.float16, torch.float16, torch.float16, torch.bfloat16]
    views = [ws[offs[i]:offs[i] + sizes[i]].view(dts[i]) for i in range(4)]
    return (views[0].view(cfg.B, cfg.Hq, cfg.S, d), views[1].view(cfg.B, cfg.Hkv, cfg.S, d),
            views[2].view(cfg.B, cfg.Hkv, cfg.S, d), views[3].view(cfg.B * cfg.S, cfg.Hq * d))


REDUCED = [
    # name, overrides of the workload geometry (reduced length), Wqkv std
    ("qwen3_0p6b", {}, 0.02),
    ("vaswani_mha", {"B": 2, "S": 512}, 0.02),
    # larger Q/K weights: a peaked softmax (Wo stays at 0.02, so the output's
    # bf16 rounding floor stays below the tolerance)
    ("vaswani_mha", {"B": 2, "S": 300}, 0.1),
    ("qwen3_4b", {"B": 1, "S": 1024}, 0.02),
    ("qwen3_32b", {"B": 1, "S": 640}, 0.02),
]


@pytest.mark.parametrize("name,over,w_std", REDUCED)
def test_forward_reduced_workloads(name, over, w_std):
    cfg = PREFILL_CONFIGS[name].with_(**over)
    t = make_layer_inputs(cfg, seed=SEEDS[name], w_std=w_std, wo_std=0.02)
    out, ws = run_forward(cfg, t)
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, causal=cfg.causal,
                         want_stages=True)
    assert_parity("out", to64(out).reshape(ref["out"].shape), ref["out"])
    q, k, v, attn = ws_views(cfg, ws)
    assert_parity("K", to64(k), ref["k"])
    assert_parity("V", to64(v), ref["v"])
    assert_parity("attn", to64(attn), ref["attn"])


@pytest.mark.parametrize("name", ["qwen3_0p6b", "vaswani_mha", "qwen3_4b", "qwen3_32b"])
def test_forward_full_workloads_sampled(name):
    """The workload at full size, in the launch configuration the benchmark
    times; the oracle computes keys/values for every token and the output for a
    seeded sample of rows (first, last, both sides of tile edges, random)."""
    cfg = PREFILL_CONFIGS[name]
    t = make_layer_inputs(cfg, seed=SEEDS[name])
    out, ws = run_forward(cfg, t)
    sel = sample_rows(cfg.B, cfg.S, 96, seed=SEEDS[name]).numpy()
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, causal=cfg.causal,
                         sel=sel, want_stages=True)
    o = out.view(cfg.B * cfg.S, cfg.hidden)[torch.from_numpy(sel).to(DEV)]
    assert_parity("out", to64(o), ref["out"])
    q, k, v, attn = ws_views(cfg, ws)
    assert_parity("attn", to64(attn[torch.from_numpy(sel).to(DEV)]), ref["attn"])
    # K and V of every token (the oracle has them all)
    assert_parity("K", to64(k), ref["k"])
    assert_parity("V", to64(v), ref["v"])


def test_range_guard_reports_clamped_values():
    """Q/K/V are stored as binary16: a value beyond +-65504 (here V from huge
    value weights) is clamped and reported as GQA_ERR_RANGE; normal inputs are
    not flagged."""
    cfg = LayerConfig("t", 1, 64, 256, 2, 1, 64, True, 1e4)
    t = make_layer_inputs(cfg, seed=3)
    W = t["Wqkv"].clone()
    W[3 * 64:] = 3000.0  # V rows: |v| ~ 3000 * |sum(x)| >> 65504
    q = torch.empty((1, 2, 64, 64), dtype=torch.float16, device=DEV)
    k = torch.empty((1, 1, 64, 64), dtype=torch.float16, device=DEV)
    v = torch.empty_like(k)
    gq.gqa_qkv_proj(dev(t["x"]), dev(W), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta, cfg.eps,
                    1, 64, 256, 2, 1, 64, q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_ERR_RANGE
    assert torch.isfinite(v.float()).all() and v.float().abs().max() == 65504.0
    gq.gqa_qkv_proj(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
                    cfg.eps, 1, 64, 256, 2, 1, 64, q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_OK


def test_forward_default_stream_entry_point():
    """gqa_attn_forward (library-owned workspace, legacy stream) gives the same
    bits as gqa_attn_forward_ex."""
    cfg = PREFILL_CONFIGS["qwen3_0p6b"].with_(B=2, S=200)
    t = make_layer_inputs(cfg, seed=9)
    out_ex, _ = run_forward(cfg, t)
    out = torch.empty_like(out_ex)
    gq.gqa_attn_forward(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                        cfg.rope_theta, cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, True,
                        out)
    torch.cuda.synchronize()
    assert torch.equal(out, out_ex)
    assert gq.gqa_last_launch_count() == 3
