"""Parity of the decode step (one new token per sequence over a KV cache) with
the fp64 oracle (GPU).

Stages alone (projection + QK-norm + RoPE at position cache_len[b] with the
cache append; split-KV attention over ragged per-sequence lengths), then the
whole step on a reduced and on the full Qwen3-8B-shaped workload.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import (DECODE_CONFIGS, SEEDS, DecodeConfig,
                                                        make_decode_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dev(t):
    return None if t is None else t.to(DEV)


def bf16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.bfloat16)


@pytest.mark.parametrize("B,L,hidden,Hq,Hkv,d,qk", [
    (4, 300, 1024, 16, 8, 128, True),
    (3, 17, 256, 4, 4, 64, False),
    (64, 8192, 4096, 32, 8, 128, True),
])
def test_decode_qkv_stage_and_append(B, L, hidden, Hq, Hkv, d, qk):
    cfg = DecodeConfig("t", B, L, hidden, Hq, Hkv, d, qk, 1e6, Lmax=L + 3)
    t = make_decode_inputs(cfg, seed=400 + B)
    # ragged positions: sequence b holds L - b*5 tokens (at least 0)
    cl = torch.tensor([max(0, L - 5 * b) for b in range(B)], dtype=torch.int32)
    kc, vc = dev(t["k_cache"]), dev(t["v_cache"])
    q = torch.empty((B, Hq, d), dtype=torch.float16, device=DEV)  # q of the new tokens is binary16
    gq.gqa_decode_qkv(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
                      cfg.eps, B, hidden, Hq, Hkv, d, kc, vc, dev(cl), cfg.lmax, q)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                        B, hidden, Hq, Hkv, d, t["k_cache"], t["v_cache"], cl, cfg.lmax)
    assert_parity("q", to64(q), ref["q"])
    idx = cl.long()
    kn = kc[torch.arange(B, device=DEV), :, idx.to(DEV)]  # [B, Hkv, d]
    vn = vc[torch.arange(B, device=DEV), :, idx.to(DEV)]
    assert_parity("k appended", to64(kn), ref["k"])
    assert_parity("v appended", to64(vn), ref["v"])
    # every other slot is untouched
    mask = torch.ones((B, cfg.lmax), dtype=torch.bool)
    mask[torch.arange(B), idx] = False
    assert torch.equal(kc.cpu().permute(0, 2, 1, 3)[mask], t["k_cache"].permute(0, 2, 1, 3)[mask])
    assert torch.equal(vc.cpu().permute(0, 2, 1, 3)[mask], t["v_cache"].permute(0, 2, 1, 3)[mask])


@pytest.mark.parametrize("B,Hq,Hkv,d,Lmax,lens", [
    (4, 16, 4, 128, 1000, [1, 5, 300, 1000]),
    (3, 8, 8, 64, 700, [700, 64, 129]),
    (2, 16, 2, 128, 5000, [5000, 2049]),
    (5, 4, 2, 64, 33, [33, 32, 31, 2, 1]),
])
def test_decode_attention_stage(B, Hq, Hkv, d, Lmax, lens):
    g = torch.Generator().manual_seed(500 + Lmax)
    q = (torch.randn((B, Hq, d), generator=g) * 1.5).to(torch.float16)
    kc = bf16_randn((B, Hkv, Lmax, d), g)
    vc = bf16_randn((B, Hkv, Lmax, d), g)
    kl = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax))
    gq.gqa_decode_attention(dev(q), dev(kc), dev(vc), dev(kl), B, Hq, Hkv, d, Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_attention_stage(q, kc, vc, kl, B, Hq, Hkv, d, Lmax)
    assert_parity("decode attn", to64(out), ref)


def run_decode(cfg, t, cache_len=None, want_attn=False):
    kc, vc = dev(t["k_cache"]), dev(t["v_cache"])
    cl = dev(t["cache_len"] if cache_len is None else cache_len)
    out = torch.empty((cfg.B, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_decode_workspace_size(cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                                                            cfg.lmax))
    gq.gqa_attn_decode(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                       cfg.rope_theta, cfg.eps, cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, cl,
                       cfg.lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    if not want_attn:
        return out
    # workspace layout: q [B,Hq,d] bf16, then attn [B,Hq*d] bf16, each 256-byte aligned
    n = cfg.B * cfg.Hq * cfg.head_dim * 2
    off = (n + 255) // 256 * 256
    attn = ws[off:off + n].view(torch.bfloat16).view(cfg.B, cfg.Hq * cfg.head_dim)
    return out, attn


def test_decode_step_reduced_ragged():
    cfg = DecodeConfig("t", 6, 500, 1024, 16, 4, 128, True, 1e6, Lmax=512)
    t = make_decode_inputs(cfg, seed=601)
    cl = torch.tensor([500, 1, 0, 257, 128, 511], dtype=torch.int32)
    out = run_decode(cfg, t, cl)
    ref = oracle.decode(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                        cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, t["k_cache"], t["v_cache"], cl,
                        cfg.lmax)
    assert_parity("decode out", to64(out), ref["out"])


def test_decode_step_full_workload():
    """64 sequences x 8192 cached tokens, Qwen3-8B attention geometry, the
    launch configuration the benchmark times; full oracle."""
    cfg = DECODE_CONFIGS["qwen3_8b_decode"]
    t = make_decode_inputs(cfg, seed=SEEDS["qwen3_8b_decode"])
    out, attn = run_decode(cfg, t, want_attn=True)
    ref = oracle.decode(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                        cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, t["k_cache"], t["v_cache"],
                        t["cache_len"], cfg.lmax)
    assert_parity("decode out", to64(out), ref["out"])
    # the attention output itself: the o_proj term (~1e-2) sits below the bf16
    # resolution of out (|x| ~ 1), so out alone cannot show an error in it
    assert_parity("decode attn", to64(attn), ref["attn"])


@pytest.mark.parametrize("B,hidden,Hq,Hkv,d", [
    (1, 2048, 16, 8, 128),    # M = 1
    (128, 1024, 8, 2, 64),    # M = 128 (one full M block); head_dim 64 tiles
    (5, 520, 4, 4, 64),       # hidden not a multiple of 64: a ragged o_proj tile
])
def test_decode_step_shapes(B, hidden, Hq, Hkv, d):
    """The decode step at the edges of its projection tiling: one sequence,
    a full 128-row M block, a ragged output width; output and attention match
    the oracle, and a second call on the same workspace repeats the first."""
    cfg = DecodeConfig("t", B, 40, hidden, Hq, Hkv, d, d == 128, 1e6, Lmax=48)
    t = make_decode_inputs(cfg, seed=650 + B)
    cl = torch.tensor([(7 * b) % 41 for b in range(B)], dtype=torch.int32)
    out, attn = run_decode(cfg, t, cl, want_attn=True)
    ref = oracle.decode(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                        cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, t["k_cache"], t["v_cache"], cl, cfg.lmax)
    assert_parity("decode attn", to64(attn), ref["attn"])
    assert_parity("decode out", to64(out), ref["out"])
    out2, _ = run_decode(cfg, t, cl, want_attn=True)
    assert torch.equal(out, out2)
