"""Parity of the backward pass with the fp64 oracle (GPU).

The attention backward alone (from binary16 q, k, v, dO) and the whole
layer's gradients (dx, dWqkv, dWo and the QK-norm weight gradients) against
oracle.attention_backward / oracle.backward on the same inputs.

Tolerance: the GPU computes P and dS in binary16 (the MMA operand type of the
binary16 Q, K, V, dO), the output gradient dO in binary16 and the fused
projection's gradient in bf16 (the MMA operand type of the bf16 weights and
x); each rounds a relative 2^-11 (binary16) or 2^-9 (bf16) per element before
a long contraction.  Measured relative L1: 2e-4 (dv) to 1.4e-3 (dq, dk) for
the attention stage, 1.6-1.9e-3 for dWqkv, dWo and dx.  The bound, max|err|
<= 2e-2 max|ref| and relative L1 <= 1e-2, keeps a margin of about five over
those; the forward's 2e-3 applies to forward outputs only.
"""
import numpy as np
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
    (2, 300, 8, 2, 128, True),    # G = 4, ragged, several key blocks and query tiles
    (1, 257, 16, 1, 128, True),   # G = 16 (8 positions per query tile)
    (2, 129, 4, 4, 64, True),     # G = 1, d = 64, one key past a block
    (1, 200, 8, 2, 64, False),    # no mask
    (1, 1, 4, 1, 128, True),      # a single token
    (1, 640, 32, 8, 128, True),   # Qwen3-4B/8B heads
    (1, 260, 32, 1, 128, True),   # G = 32 (4 positions per query tile)
    (1, 256, 8, 2, 128, False),   # no mask, no ragged edge: every tile unmasked
    (2, 1024, 8, 1, 64, True),    # many tiles per CTA (both operand rings wrap often)
    # group sizes that are not powers of two: R = floor(128/G) rounded down to a
    # multiple of 4 positions per head, so a tile packs G*R < 128 query rows
    (1, 300, 24, 8, 128, True),   # G = 3: 40 positions x 3 heads = 120 rows
    (2, 257, 10, 2, 64, True),    # G = 5: 24 x 5 = 120
    (1, 333, 40, 8, 128, True),   # G = 5 (Hq = 40, Hkv = 8)
    (1, 200, 12, 2, 128, False),  # G = 6: 20 x 6 = 120, no mask
    (1, 129, 7, 1, 64, True),     # G = 7: 16 x 7 = 112
    (1, 150, 24, 1, 128, True),   # G = 24: 4 x 24 = 96
])
def test_attention_backward_stage(B, S, Hq, Hkv, d, causal):
    g = torch.Generator().manual_seed(3000 + S)
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
    assert_parity("dv", dv.cpu().double().numpy(), rv, **TOL)
    if S == 1:
        # one key: the exact dq and dk are 0 (dS = P (dP - D) with P = 1 and
        # D = dP).  The GPU's D uses the bf16-stored output O, so dP - D is
        # bf16 rounding of O: |dS| <= 2^-8 sum_c |dO_c O_c|, and
        # |dq| <= |dS| max|k| / sqrt(d) (likewise dk with q).
        ds_max = 2.0 ** -8 * float((dO.double().abs() * V.double().abs().repeat_interleave(Hq // Hkv, 1))
                                   .sum(-1).max())
        assert float(dq.abs().max()) <= ds_max * float(K.double().abs().max()) / d ** 0.5
        assert float(dk.abs().max()) <= ds_max * float(Q.double().abs().max()) / d ** 0.5 * (Hq // Hkv)
        return
    assert_parity("dq", dq.cpu().double().numpy(), rq, **TOL)
    assert_parity("dk", dk.cpu().double().numpy(), rk, **TOL)


@pytest.mark.parametrize("geom,causal", [
    ({"B": 2, "S": 300, "hidden": 512, "Hq": 8, "Hkv": 2, "head_dim": 128, "qk_norm": True, "rope_theta": 1e6},
     True),
    ({"B": 2, "S": 150, "hidden": 256, "Hq": 4, "Hkv": 4, "head_dim": 64, "qk_norm": False, "rope_theta": 1e4},
     True),
    ({"B": 1, "S": 200, "hidden": 384, "Hq": 8, "Hkv": 1, "head_dim": 128, "qk_norm": True, "rope_theta": 1e6},
     False),
    ({"B": 1, "S": 260, "hidden": 640, "Hq": 10, "Hkv": 2, "head_dim": 64, "qk_norm": True, "rope_theta": 1e6},
     True),  # G = 5
])
def test_layer_backward(geom, causal):
    cfg = LayerConfig("t", **geom)
    B, S, h, Hq, Hkv, d = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
    t = make_layer_inputs(cfg, seed=3100 + S, w_std=0.05)
    dout = (torch.randn((B * S, h), generator=torch.Generator().manual_seed(3101)) * 0.5).to(torch.bfloat16)
    N = (Hq + 2 * Hkv) * d
    dx = torch.empty((B, S, h), dtype=torch.bfloat16, device=DEV)
    dW = torch.empty((N, h), dtype=torch.float32, device=DEV)
    dWo = torch.empty((h, Hq * d), dtype=torch.float32, device=DEV)
    dqn = torch.empty(d, dtype=torch.float32, device=DEV) if cfg.qk_norm else None
    dkn = torch.empty(d, dtype=torch.float32, device=DEV) if cfg.qk_norm else None
    ws = gq.new_workspace(gq.gqa_attn_backward_workspace_size(B, S, h, Hq, Hkv, d))
    gq.gqa_attn_backward(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                         cfg.rope_theta, cfg.eps, B, S, h, Hq, Hkv, d, causal, dev(dout), dx, dW, dWo, dqn, dkn, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.backward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                          B, S, h, Hq, Hkv, d, dout, causal=causal)
    assert_parity("dWo", dWo.cpu().double().numpy(), ref["dWo"], **TOL)
    assert_parity("dWqkv", dW.cpu().double().numpy(), ref["dWqkv"], **TOL)
    assert_parity("dx", to64(dx).reshape(-1, h), ref["dx"], **TOL)
    # the path through the projection alone (dx minus the residual's dout):
    # dx is stored in bf16 at the scale of |dout + term|, so its rounding
    # (<= 2^-9 |dx| per element) adds to the bound in proportion to |dx| / |term|
    term_ref = ref["dx"] - to64(dout)
    term_gpu = to64(dx).reshape(-1, h) - to64(dout)
    slack = 2.0 ** -9 * float(np.abs(ref["dx"]).sum() / np.abs(term_ref).sum())
    slack_max = 2.0 ** -9 * float(np.abs(ref["dx"]).max() / np.abs(term_ref).max())
    assert_parity("dx - dout", term_gpu, term_ref, tol_max=TOL["tol_max"] + slack_max,
                  tol_rel=TOL["tol_rel"] + slack)
    if cfg.qk_norm:
        assert_parity("dq_norm_w", dqn.cpu().double().numpy(), ref["dq_norm_w"], **TOL)
        assert_parity("dk_norm_w", dkn.cpu().double().numpy(), ref["dk_norm_w"], **TOL)


def test_backward_rejects_unsupported_shapes():
    q = torch.zeros((1, 64, 8, 128), dtype=torch.float16, device=DEV)   # G = 64 > 32
    k = torch.zeros((1, 1, 8, 128), dtype=torch.float16, device=DEV)
    f = torch.zeros((1, 64, 8, 128), dtype=torch.float32, device=DEV)
    g = torch.zeros((1, 1, 8, 128), dtype=torch.float32, device=DEV)
    ws = gq.new_workspace(1 << 20)
    with pytest.raises(gq.GqaError, match=f"status {gq.GQA_ERR_UNSUPPORTED}"):
        gq.gqa_attention_backward(q, k, k, q, 1, 8, 64, 1, 128, True, f, g, g, ws)
    q = torch.zeros((1, 4, 8, 256), dtype=torch.float16, device=DEV)    # head_dim 256
    k = torch.zeros((1, 1, 8, 256), dtype=torch.float16, device=DEV)
    f = torch.zeros((1, 4, 8, 256), dtype=torch.float32, device=DEV)
    g = torch.zeros((1, 1, 8, 256), dtype=torch.float32, device=DEV)
    with pytest.raises(gq.GqaError, match=f"status {gq.GQA_ERR_UNSUPPORTED}"):
        gq.gqa_attention_backward(q, k, k, q, 1, 8, 4, 1, 256, True, f, g, g, ws)
