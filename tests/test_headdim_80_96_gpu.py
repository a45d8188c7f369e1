"""Parity of head_dim 80 and 96 with the fp64 oracle (GPU).

[Knob] "Where the invariance breaks" names both widths: 80 is the quotient
hidden / heads of Qwen3-4B's widths (2560 / 32), and 96 is the width a fused
kernel usually has no tile for.  Here the QKV GEMM uses tiles of whole heads
(3 x 80 = 240 and 2 x 96 = 192 columns) and the attention stages the heads as
128-wide rows whose extra columns are zero.  Checked: the attention stage over
group sizes 1, 4 and 8, ragged lengths, a single token and the unmasked case;
marker values for the head map with peaked scores; the cached-prefill
attention; the QKV stage with full and partial rotary (d, d/2, d/4, 0); the
whole layer and the layer written into a KV cache; the full 4 x 4096-token
workloads on sampled rows.

Tolerance: max|err| <= 1e-2 max|ref| and relative L1 <= 2e-3 (tests/parity.py);
the cached path computes with bf16 Q and P, as at the other widths.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import PREFILL_CONFIGS, LayerConfig, make_layer_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
WIDTHS = [80, 96]


def dev(t):
    return None if t is None else t.to(DEV)


def f16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.float16)


def bf16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.bfloat16)


@pytest.mark.parametrize("D", WIDTHS)
@pytest.mark.parametrize("B,S,Hq,Hkv,causal", [
    (1, 300, 8, 2, True),     # G = 4, ragged: several key tiles and query blocks
    (2, 129, 8, 8, True),     # G = 1, one key past a tile
    (1, 700, 16, 2, True),    # G = 8
    (2, 200, 4, 2, False),    # no mask
    (1, 1, 4, 1, True),       # a single token
])
def test_attention_stage(D, B, S, Hq, Hkv, causal):
    g = torch.Generator().manual_seed(4000 + S + D)
    Q = f16_randn((B, Hq, S, D), g, 1.5)
    K = f16_randn((B, Hkv, S, D), g, 1.5)
    V = f16_randn((B, Hkv, S, D), g)
    out = torch.empty((B, S, Hq * D), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention(dev(Q), dev(K), dev(V), B, S, Hq, Hkv, D, causal, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.attention_stage(Q, K, V, B, S, Hq, Hkv, D, causal=causal)
    assert_parity(f"attn d{D}", to64(out).reshape(B * S, Hq * D), ref)


@pytest.mark.parametrize("D", WIDTHS)
def test_attention_group_markers_and_peaked_scores(D):
    """Each KV head's values are one constant marker row, so every query head
    returns its group's marker (all D columns, none of them zero-padding);
    with large scores the output is still the oracle's."""
    B, S, Hq, Hkv = 2, 400, 8, 2
    g = torch.Generator().manual_seed(4100 + D)
    markers = torch.arange(1, B * Hkv * D + 1, dtype=torch.float32).reshape(B, Hkv, 1, D) / (B * Hkv * D)
    V = markers.expand(B, Hkv, S, D).contiguous().to(torch.float16)
    Q = f16_randn((B, Hq, S, D), g, 4.0)
    K = f16_randn((B, Hkv, S, D), g, 4.0)
    out = torch.empty((B, S, Hq * D), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention(dev(Q), dev(K), dev(V), B, S, Hq, Hkv, D, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    o = to64(out).reshape(B, S, Hq, D)
    mk = to64(markers.to(torch.float16))
    for j in range(Hq):
        np.testing.assert_allclose(o[:, :, j], np.broadcast_to(mk[:, j // (Hq // Hkv)], (B, S, D)),
                                   rtol=1e-2, atol=0)
    V2 = f16_randn((B, Hkv, S, D), g)
    gq.gqa_attention(dev(Q), dev(K), dev(V2), B, S, Hq, Hkv, D, True, out)
    torch.cuda.synchronize()
    ref = oracle.attention_stage(Q, K, V2, B, S, Hq, Hkv, D)
    assert_parity(f"attn d{D} peaked", to64(out).reshape(B * S, -1), ref)


@pytest.mark.parametrize("D", WIDTHS)
def test_attention_cached(D):
    B, S, Hq, Hkv, Lmax = 2, 100, 8, 2, 400
    p0 = [0, 237]
    g = torch.Generator().manual_seed(4200 + D)
    q = (torch.randn((B, Hq, S, D), generator=g) * 1.5).to(torch.float16)
    kc = bf16_randn((B, Hkv, Lmax, D), g, 1.5)
    vc = bf16_randn((B, Hkv, Lmax, D), g)
    cl = torch.tensor(p0, dtype=torch.int32)
    out = torch.empty((B, S, Hq * D), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention_cached(dev(q), dev(kc), dev(vc), dev(cl), B, S, Hq, Hkv, D, Lmax, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = np.empty((B, S, Hq * D))
    for t in range(S):
        ref[:, t] = oracle.decode_attention_stage(q[:, :, t].contiguous(), kc, vc, [p + t + 1 for p in p0],
                                                  B, Hq, Hkv, D, Lmax)
    assert_parity(f"cached attn d{D}", to64(out).reshape(B, S, -1), ref)


@pytest.mark.parametrize("D,rd", [(80, 80), (80, 40), (80, 20), (80, 0), (96, 96), (96, 48), (96, 24), (96, 0)])
def test_qkv_stage(D, rd):
    # 5 KV heads: 5 + 2*5 = 15 heads = 5 tiles of 3 at d = 80, a ragged last tile at d = 96
    cfg = LayerConfig("t", B=2, S=300, hidden=384, Hq=5, Hkv=5, head_dim=D, qk_norm=True, rope_theta=1e6)
    B, S, h, Hq, Hkv = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv
    t = make_layer_inputs(cfg, seed=4300 + D + rd, w_std=0.05)
    q = torch.empty((B, Hq, S, D), dtype=torch.float16, device=DEV)
    k = torch.empty((B, Hkv, S, D), dtype=torch.float16, device=DEV)
    v = torch.empty_like(k)
    gq.gqa_qkv_proj_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
                       cfg.eps, rd, B, S, h, Hq, Hkv, D, q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    rq, rk, rv = oracle.qkv_stage(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                  B, S, h, Hq, Hkv, D, rotary_dim=rd)
    assert_parity(f"Q d{D} rd{rd}", to64(q), rq)
    assert_parity(f"K d{D} rd{rd}", to64(k), rk)
    assert_parity(f"V d{D} rd{rd}", to64(v), rv)


@pytest.mark.parametrize("D,Hq,Hkv,qk", [(80, 8, 2, True), (96, 6, 3, True), (80, 4, 4, False)])
def test_forward_layer(D, Hq, Hkv, qk):
    cfg = LayerConfig("t", B=2, S=333, hidden=320, Hq=Hq, Hkv=Hkv, head_dim=D, qk_norm=qk,
                      rope_theta=1e6 if qk else 1e4)
    t = make_layer_inputs(cfg, seed=4400 + D)
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D))
    gq.gqa_attn_forward_ex(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                           cfg.rope_theta, cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, True, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, want_stages=True)
    assert_parity(f"out d{D}", to64(out).reshape(-1, cfg.hidden), ref["out"])


@pytest.mark.parametrize("D", WIDTHS)
def test_prefill_cached_layer(D):
    cfg = LayerConfig("t", B=2, S=130, hidden=512, Hq=8, Hkv=2, head_dim=D, qk_norm=True, rope_theta=1e6)
    p0, Lmax = [300, 7], 440
    t = make_layer_inputs(cfg, seed=4500 + D)
    g = torch.Generator().manual_seed(4501)
    kc = torch.zeros((cfg.B, cfg.Hkv, Lmax, D), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for b, p in enumerate(p0):
        kc[b, :, :p] = bf16_randn((cfg.Hkv, p, D), g)
        vc[b, :, :p] = bf16_randn((cfg.Hkv, p, D), g)
    kd, vd = dev(kc), dev(vc)
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_prefill_cached_workspace_size(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, D, Lmax))
    gq.gqa_attn_prefill_cached(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                               cfg.rope_theta, cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, True,
                               kd, vd, dev(torch.tensor(p0, dtype=torch.int32)), Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.prefill_cached(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, kc, vc, p0, Lmax)
    assert_parity(f"out cached d{D}", to64(out).reshape(-1, cfg.hidden), ref["out"])
    k_after, v_after = kd.cpu(), vd.cpu()
    for b, p in enumerate(p0):
        assert_parity(f"k slots d{D} b={b}", to64(k_after[b, :, p:p + cfg.S]), ref["k"][b])
        assert_parity(f"v slots d{D} b={b}", to64(v_after[b, :, p:p + cfg.S]), ref["v"][b])
        assert torch.equal(k_after[b, :, :p], kc[b, :, :p]) and torch.equal(k_after[b, :, p + cfg.S:],
                                                                            kc[b, :, p + cfg.S:])


@pytest.mark.parametrize("name", ["qwen3_4b_d80", "knob_d96"])
def test_forward_full_workload_sampled(name):
    """The full 4 x 4096-token workload on the launch configuration the
    benchmark times; the oracle evaluates sampled rows."""
    cfg = PREFILL_CONFIGS[name]
    D = cfg.head_dim
    t = make_layer_inputs(cfg, seed=4600 + D)
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attn_forward(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                        cfg.rope_theta, cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    rows = [0, 1, 31, 32, 63, 64, 127, 128, 2047, 2048, 4095, 4096, 4096 + 77, 3 * 4096 + 4095]
    rows += list(np.random.default_rng(6).integers(0, cfg.B * cfg.S, 40))
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, sel=rows)
    assert_parity(f"out {name} sampled", to64(out).reshape(-1, cfg.hidden)[rows], ref)
