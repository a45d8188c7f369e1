"""The backward at head widths 80 and 96 and with partial rotary (GPU),
against the fp64 oracle.

[Knob] "Where the invariance breaks" names the widths 80 (Qwen3-4B's hidden /
heads) and 96; [NeoX] "Scaling and RoPE" the rotary_pct that rotates only the
leading features.  The attention backward stages 80- and 96-wide rows as
128-wide tiles whose extra columns are zero; the inverse RoPE acts on the
first rotary_dim features (R16).  Checked: the attention backward stage at
both widths, the whole layer's gradients at both widths and at rotary widths
d/2, d/4 and 0, and the training pair with a rotary width (bit-identical to
the recomputing backward).

Tolerance: as for the other backward tests, max|err| <= 2e-2 max|ref| and
relative L1 <= 1e-2 (binary16 P, dS and dO, bf16 projection gradient).
"""
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import LayerConfig, make_layer_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = dict(tol_max=2e-2, tol_rel=1e-2)


def dev(t):
    return None if t is None else t.to(DEV)


def f16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.float16)


@pytest.mark.parametrize("B,S,Hq,Hkv,d,causal", [
    (2, 300, 8, 2, 80, True),
    (1, 257, 4, 4, 96, True),
    (1, 200, 8, 1, 80, False),
    (2, 129, 16, 2, 96, True),
])
def test_attention_backward_stage_width(B, S, Hq, Hkv, d, causal):
    g = torch.Generator().manual_seed(6000 + S + d)
    Q = f16_randn((B, Hq, S, d), g, 1.5)
    K = f16_randn((B, Hkv, S, d), g, 1.5)
    V = f16_randn((B, Hkv, S, d), g)
    dO = f16_randn((B, Hq, S, d), g)
    dq = torch.empty((B, Hq, S, d), dtype=torch.float32, device=DEV)
    dk = torch.empty((B, Hkv, S, d), dtype=torch.float32, device=DEV)
    dv = torch.empty_like(dk)
    ws = gq.new_workspace(gq.gqa_attention_backward_workspace_size(B, S, Hq, d))
    gq.gqa_attention_backward(dev(Q), dev(K), dev(V), dev(dO), B, S, Hq, Hkv, d, causal, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    dO_tok = dO.permute(0, 2, 1, 3).reshape(B, S, Hq * d).contiguous()
    rq, rk, rv = oracle.attention_backward(Q, K, V, dO_tok, B, S, Hq, Hkv, d, causal=causal)
    assert_parity(f"dv d{d}", dv.cpu().double().numpy(), rv, **TOL)
    assert_parity(f"dq d{d}", dq.cpu().double().numpy(), rq, **TOL)
    assert_parity(f"dk d{d}", dk.cpu().double().numpy(), rk, **TOL)


def _layer_grads(cfg, rd, saved=False):
    B, S, h, Hq, Hkv, d = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
    t = make_layer_inputs(cfg, seed=6100 + S + d + rd, w_std=0.05)
    dout = (torch.randn((B * S, h), generator=torch.Generator().manual_seed(6101)) * 0.5).to(torch.bfloat16)
    N = (Hq + 2 * Hkv) * d
    dx = torch.empty((B, S, h), dtype=torch.bfloat16, device=DEV)
    dW = torch.empty((N, h), dtype=torch.float32, device=DEV)
    dWo = torch.empty((h, Hq * d), dtype=torch.float32, device=DEV)
    dqn = torch.empty(d, dtype=torch.float32, device=DEV) if cfg.qk_norm else None
    dkn = torch.empty(d, dtype=torch.float32, device=DEV) if cfg.qk_norm else None
    ws = gq.new_workspace(gq.gqa_attn_backward_workspace_size(B, S, h, Hq, Hkv, d))
    args = (dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
            cfg.eps, rd, B, S, h, Hq, Hkv, d, cfg.causal)
    if saved:
        out = torch.empty((B, S, h), dtype=torch.bfloat16, device=DEV)
        gq.gqa_attn_forward_train_rd(*args, out, ws)
        gq.gqa_attn_backward_saved_rd(*args, dev(dout), dx, dW, dWo, dqn, dkn, ws)
    else:
        gq.gqa_attn_backward_rd(*args, dev(dout), dx, dW, dWo, dqn, dkn, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    return t, dout, (dx, dW, dWo, dqn, dkn)


@pytest.mark.parametrize("d,rd,qk", [
    (80, 80, True), (96, 96, False), (128, 64, True), (128, 32, True), (64, 0, True), (80, 20, True), (96, 48, True),
])
def test_layer_backward_width_and_rotary(d, rd, qk):
    cfg = LayerConfig("t", B=2, S=200, hidden=512, Hq=8, Hkv=2, head_dim=d, qk_norm=qk, rope_theta=1e6)
    t, dout, (dx, dW, dWo, dqn, dkn) = _layer_grads(cfg, rd)
    ref = oracle.backward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                          cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, d, dout, rotary_dim=rd)
    tag = f"d{d} rd{rd}"
    assert_parity(f"dWo {tag}", dWo.cpu().double().numpy(), ref["dWo"], **TOL)
    assert_parity(f"dWqkv {tag}", dW.cpu().double().numpy(), ref["dWqkv"], **TOL)
    assert_parity(f"dx {tag}", to64(dx).reshape(-1, cfg.hidden), ref["dx"], **TOL)
    if qk:
        assert_parity(f"dq_norm_w {tag}", dqn.cpu().double().numpy(), ref["dq_norm_w"], **TOL)
        assert_parity(f"dk_norm_w {tag}", dkn.cpu().double().numpy(), ref["dk_norm_w"], **TOL)


def test_training_pair_with_rotary_width_matches_recomputing_backward():
    cfg = LayerConfig("t", B=1, S=300, hidden=384, Hq=8, Hkv=2, head_dim=96, qk_norm=True, rope_theta=1e6)
    _, _, g_saved = _layer_grads(cfg, 48, saved=True)
    _, _, g_rec = _layer_grads(cfg, 48, saved=False)
    for name, a, b in zip(("dx", "dWqkv", "dWo"), g_saved[:3], g_rec[:3]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), name
    for a, b in zip(g_saved[3:], g_rec[3:]):
        torch.testing.assert_close(a, b, rtol=1e-5, atol=1e-6 * float(b.abs().max()))
