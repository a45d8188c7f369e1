"""Parity of prefill into a KV cache (chunked prefill) with the fp64 oracle (GPU).

Q and P are binary16 as in the plain prefill (the attention widens each bf16
cache tile to binary16 in shared memory), so the attention output and the
layer output are both held to the standard tolerance.  Cache slots past the
last written key may hold anything, NaN included, without reaching the
output; a cached value beyond the binary16 range is saturated and reported.

S new tokens per sequence sit at positions cache_len[b] .. cache_len[b]+S-1:
their K/V are appended to the bf16 cache and each attends to the cached prefix
plus the new tokens up to itself.  Checked: the attention stage alone (against
the oracle's decode attention evaluated row by row), the whole call on ragged
per-sequence offsets (output, attention, the cache slots written and the slots
left alone), two chunks against one prefill, and a Qwen3-32B-shaped chunk late
in a 16K-token context.
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


def dev(t):
    return None if t is None else t.to(DEV)


def bf16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.bfloat16)


@pytest.mark.parametrize("B,S,Hq,Hkv,d,Lmax,p0", [
    (3, 150, 16, 8, 128, 600, [0, 200, 450]),
    (2, 77, 8, 1, 128, 300, [5, 223]),
    (2, 64, 8, 8, 64, 200, [136, 1]),
])
def test_attention_cached_stage(B, S, Hq, Hkv, d, Lmax, p0):
    g = torch.Generator().manual_seed(700 + S)
    q = (torch.randn((B, Hq, S, d), generator=g) * 1.5).to(torch.float16)
    kc = bf16_randn((B, Hkv, Lmax, d), g, 1.5)
    vc = bf16_randn((B, Hkv, Lmax, d), g)
    cl = torch.tensor(p0, dtype=torch.int32)
    out = torch.empty((B, S, Hq * d), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention_cached(dev(q), dev(kc), dev(vc), dev(cl), B, S, Hq, Hkv, d, Lmax, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = np.empty((B, S, Hq * d))
    for t in range(S):  # query t of sequence b = decode of one token over keys [0, p0[b] + t]
        ref[:, t] = oracle.decode_attention_stage(q[:, :, t].contiguous(), kc, vc, [p + t + 1 for p in p0],
                                                  B, Hq, Hkv, d, Lmax)
    assert_parity("cached attn", to64(out).reshape(B, S, -1), ref)


def run_cached(cfg, t, kc, vc, p0, Lmax):
    B, S = cfg.B, cfg.S
    kd, vd = dev(kc), dev(vc)
    out = torch.empty((B, S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_prefill_cached_workspace_size(B, S, cfg.Hq, cfg.Hkv, cfg.head_dim, Lmax))
    gq.gqa_attn_prefill_cached(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                               cfg.rope_theta, cfg.eps, B, S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, cfg.causal,
                               kd, vd, dev(torch.tensor(p0, dtype=torch.int32)), Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    # workspace layout: Q [B,Hq,S,d] binary16, then attn [B*S, Hq*d] bf16, each 256-byte aligned
    n = B * S * cfg.Hq * cfg.head_dim * 2
    off = (n + 255) // 256 * 256
    attn = ws[off:off + n].view(torch.bfloat16).view(B * S, -1)
    return out, attn, kd, vd


@pytest.mark.parametrize("geom,S,p0,Lmax", [
    ({"hidden": 1024, "Hq": 16, "Hkv": 8, "head_dim": 128, "qk_norm": True, "rope_theta": 1e6}, 200, [0, 100, 257], 512),
    ({"hidden": 512, "Hq": 16, "Hkv": 2, "head_dim": 128, "qk_norm": True, "rope_theta": 1e6}, 130, [300, 7], 440),
    ({"hidden": 512, "Hq": 8, "Hkv": 8, "head_dim": 64, "qk_norm": False, "rope_theta": 1e4}, 96, [64, 129], 256),
])
def test_prefill_cached_layer(geom, S, p0, Lmax):
    cfg = LayerConfig("t", B=len(p0), S=S, **geom)
    t = make_layer_inputs(cfg, seed=800 + S)
    g = torch.Generator().manual_seed(801)
    kc = torch.zeros((cfg.B, cfg.Hkv, Lmax, cfg.head_dim), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for b, p in enumerate(p0):  # earlier tokens: normed/rotated keys ~ N(0,1), values ~ N(0,1)
        kc[b, :, :p] = bf16_randn((cfg.Hkv, p, cfg.head_dim), g)
        vc[b, :, :p] = bf16_randn((cfg.Hkv, p, cfg.head_dim), g)
    out, attn, kd, vd = run_cached(cfg, t, kc, vc, p0, Lmax)
    ref = oracle.prefill_cached(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                cfg.B, S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, p0, Lmax)
    assert_parity("out", to64(out).reshape(-1, cfg.hidden), ref["out"])
    assert_parity("attn", to64(attn), ref["attn"])
    k_after, v_after = kd.cpu(), vd.cpu()
    for b, p in enumerate(p0):
        assert_parity(f"k slots b={b}", to64(k_after[b, :, p:p + S]), ref["k"][b])
        assert_parity(f"v slots b={b}", to64(v_after[b, :, p:p + S]), ref["v"][b])
        assert torch.equal(k_after[b, :, :p], kc[b, :, :p]) and torch.equal(k_after[b, :, p + S:], kc[b, :, p + S:])
        assert torch.equal(v_after[b, :, :p], vc[b, :, :p]) and torch.equal(v_after[b, :, p + S:], vc[b, :, p + S:])


def test_two_chunks_match_one_prefill():
    """Chunked prefill into an empty cache, 300 + 212 tokens, reproduces the
    plain prefill of all 512 tokens."""
    cfg = PREFILL_CONFIGS["qwen3_0p6b"].with_(B=2, S=512)
    t = make_layer_inputs(cfg, seed=900)
    Lmax, S1 = 512, 300
    kc = torch.zeros((cfg.B, cfg.Hkv, Lmax, cfg.head_dim), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kd, vd = dev(kc), dev(vc)
    outs = []
    for lo, hi in ((0, S1), (S1, cfg.S)):
        sub = cfg.with_(S=hi - lo)
        x = dev(t["x"][:, lo:hi].contiguous())
        out = torch.empty((cfg.B, hi - lo, cfg.hidden), dtype=torch.bfloat16, device=DEV)
        ws = gq.new_workspace(gq.gqa_attn_prefill_cached_workspace_size(cfg.B, hi - lo, cfg.Hq, cfg.Hkv, cfg.head_dim, Lmax))
        gq.gqa_attn_prefill_cached(x, dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                                   cfg.rope_theta, cfg.eps, cfg.B, sub.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                                   True, kd, vd, dev(torch.full((cfg.B,), lo, dtype=torch.int32)), Lmax, out, ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    got = torch.cat(outs, dim=1)
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim)
    assert_parity("chunked out", to64(got).reshape(ref.shape), ref)


def test_prefill_cached_qwen3_32b_chunk_late_in_context():
    """Qwen3-32B shape: 256 new tokens after 14336 cached ones (Lmax 16384)."""
    cfg = PREFILL_CONFIGS["qwen3_32b"].with_(S=256)
    t = make_layer_inputs(cfg, seed=901)
    Lmax, p = 16384, 14336
    g = torch.Generator().manual_seed(902)
    kc = torch.zeros((1, cfg.Hkv, Lmax, cfg.head_dim), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kc[:, :, :p] = bf16_randn((1, cfg.Hkv, p, cfg.head_dim), g)
    vc[:, :, :p] = bf16_randn((1, cfg.Hkv, p, cfg.head_dim), g)
    out, attn, kd, vd = run_cached(cfg, t, kc, vc, [p], Lmax)
    ref = oracle.prefill_cached(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                1, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, [p], Lmax)
    assert_parity("out", to64(out).reshape(-1, cfg.hidden), ref["out"])
    assert_parity("attn", to64(attn), ref["attn"])
    assert_parity("k slots", to64(kd.cpu()[0, :, p:p + cfg.S]), ref["k"][0])


def test_prefill_cached_rejects_an_offset_past_the_cache():
    """cache_len[b] + S > Lmax: the sequence gets zero rows and the device
    error word reports it; the other sequence is computed."""
    cfg = LayerConfig("t", B=2, S=64, hidden=256, Hq=4, Hkv=2, head_dim=128, qk_norm=True, rope_theta=1e6)
    t = make_layer_inputs(cfg, seed=903)
    Lmax = 128
    kc = torch.zeros((2, 2, Lmax, 128), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kd, vd = dev(kc), dev(vc)
    out = torch.empty((2, 64, 256), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_prefill_cached_workspace_size(2, 64, 4, 2, 128, Lmax))
    gq.gqa_attn_prefill_cached(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                               1e6, 1e-6, 2, 64, 256, 4, 2, 128, True, kd, vd,
                               dev(torch.tensor([10, 100], dtype=torch.int32)), Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_ERR_ARG
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("d", [128, 256])
def test_unwritten_cache_slots_never_reach_the_output(d):
    """Slots past cache_len[b] + S hold NaN (never written): the output equals
    the one over zero-filled slots, bit for bit, and nothing is reported."""
    B, S, Hq, Hkv, Lmax = 2, 70, 8, 2, 320
    p0 = [100, 5]
    g = torch.Generator().manual_seed(960 + d)
    q = (torch.randn((B, Hq, S, d), generator=g) * 1.5).to(torch.float16)
    kc = bf16_randn((B, Hkv, Lmax, d), g, 1.5)
    vc = bf16_randn((B, Hkv, Lmax, d), g)
    cl = torch.tensor(p0, dtype=torch.int32)
    outs = []
    for fill in (0.0, float("nan")):
        k2, v2 = kc.clone(), vc.clone()
        for b, p in enumerate(p0):
            k2[b, :, p + S:] = fill
            v2[b, :, p + S:] = fill
        out = torch.empty((B, S, Hq * d), dtype=torch.bfloat16, device=DEV)
        gq.gqa_attention_cached(dev(q), dev(k2), dev(v2), dev(cl), B, S, Hq, Hkv, d, Lmax, True, out)
        torch.cuda.synchronize()
        assert gq.gqa_check_device_error() == 0
        outs.append(out.cpu())
    assert torch.isfinite(outs[1].float()).all()
    assert torch.equal(outs[0], outs[1])


def test_cached_value_beyond_binary16_is_saturated_and_reported():
    """A cached value of 2^17 (a bf16 value past binary16's 65504) is widened to
    65504 and flagged; the status is read and cleared."""
    B, S, Hq, Hkv, d, Lmax = 1, 16, 4, 1, 128, 64
    g = torch.Generator().manual_seed(970)
    q = torch.randn((B, Hq, S, d), generator=g).to(torch.float16)
    kc = bf16_randn((B, Hkv, Lmax, d), g)
    vc = bf16_randn((B, Hkv, Lmax, d), g)
    vc[0, 0, 3, 5] = 2.0 ** 17
    out = torch.empty((B, S, Hq * d), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention_cached(dev(q), dev(kc), dev(vc), dev(torch.tensor([20], dtype=torch.int32)), B, S, Hq, Hkv, d,
                            Lmax, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_ERR_RANGE
    assert gq.gqa_check_device_error() == gq.GQA_OK
    assert torch.isfinite(out.float()).all()
