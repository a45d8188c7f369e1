"""Parity of head_dim 256 with the fp64 oracle (GPU).

The [NeoX] page's Gemma-3 example ("Background": hidden 640, four query
heads, an explicit head_dim of 256) needs 256-wide heads.  The QKV GEMM
handles them with one head per 256-column tile; the attention has a kernel of
its own (by default on 2-CTA clusters with 128-key S tiles; the one-CTA form,
one query tile with two S buffers of 64 keys, is re-run under
gqa_set_cta_pairs(0) in tests/test_one_cta_forms_gpu.py).  Checked: the
attention stage over group sizes 1, 4, 8 and 16, ragged lengths and the
unmasked case, with marker values for the head map; the cached-prefill
attention; the QKV stage with full and partial rotary; the whole layer at
the Gemma-3 width (decode at head_dim 256: tests/test_decode_widths_gpu.py).

Tolerance: max|err| <= 1e-2 max|ref| and relative L1 <= 2e-3 (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import PREFILL_CONFIGS, make_layer_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 256


def dev(t):
    return None if t is None else t.to(DEV)


def f16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.float16)


@pytest.mark.parametrize("B,S,Hq,Hkv,causal", [
    (1, 300, 4, 1, True),     # the Gemma-3 group (G = 4), ragged, crosses 64-key tiles
    (2, 129, 8, 8, True),     # G = 1, one key past two tiles
    (1, 1000, 16, 2, True),   # G = 8
    (1, 257, 16, 1, True),    # G = 16: 8 positions per tile
    (2, 200, 4, 2, False),    # no mask
    (1, 1, 4, 1, True),       # a single token
    (1, 64, 4, 1, True),      # exactly one key tile
])
def test_attention_stage_d256(B, S, Hq, Hkv, causal):
    g = torch.Generator().manual_seed(2000 + S)
    Q = f16_randn((B, Hq, S, D), g, 1.5)
    K = f16_randn((B, Hkv, S, D), g, 1.5)
    V = f16_randn((B, Hkv, S, D), g)
    out = torch.empty((B, S, Hq * D), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention(dev(Q), dev(K), dev(V), B, S, Hq, Hkv, D, causal, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.attention_stage(Q, K, V, B, S, Hq, Hkv, D, causal=causal)
    assert_parity("attn d256", to64(out).reshape(B * S, Hq * D), ref)


def test_attention_d256_group_markers_and_peaked_scores():
    """Each KV head's values are one constant marker, so every query head
    must return its group's marker; with large scores (a peaked softmax that
    moves the running max across tiles) the output is still the oracle's."""
    B, S, Hq, Hkv = 2, 400, 8, 2
    g = torch.Generator().manual_seed(7)
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
    assert_parity("attn d256 peaked", to64(out).reshape(B * S, -1), ref)


def test_attention_cached_d256():
    B, S, Hq, Hkv, Lmax = 2, 100, 4, 1, 400
    p0 = [0, 237]
    g = torch.Generator().manual_seed(2100)
    q = (torch.randn((B, Hq, S, D), generator=g) * 1.5).to(torch.float16)
    kc = (torch.randn((B, Hkv, Lmax, D), generator=g) * 1.5).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, Lmax, D), generator=g).to(torch.bfloat16)
    cl = torch.tensor(p0, dtype=torch.int32)
    out = torch.empty((B, S, Hq * D), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention_cached(dev(q), dev(kc), dev(vc), dev(cl), B, S, Hq, Hkv, D, Lmax, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = np.empty((B, S, Hq * D))
    for t in range(S):
        ref[:, t] = oracle.decode_attention_stage(q[:, :, t].contiguous(), kc, vc, [p + t + 1 for p in p0],
                                                  B, Hq, Hkv, D, Lmax)
    assert_parity("cached attn d256", to64(out).reshape(B, S, -1), ref)


@pytest.mark.parametrize("rd", [256, 64, 0])
def test_qkv_stage_d256(rd):
    cfg = PREFILL_CONFIGS["gemma3_d256"].with_(B=2, S=300)
    B, S, h, Hq, Hkv = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv
    t = make_layer_inputs(cfg, seed=2200 + rd, w_std=0.05)
    q = torch.empty((B, Hq, S, D), dtype=torch.float16, device=DEV)
    k = torch.empty((B, Hkv, S, D), dtype=torch.float16, device=DEV)
    v = torch.empty_like(k)
    gq.gqa_qkv_proj_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
                       cfg.eps, rd, B, S, h, Hq, Hkv, D, q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    rq, rk, rv = oracle.qkv_stage(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                  B, S, h, Hq, Hkv, D, rotary_dim=rd)
    assert_parity("Q d256", to64(q), rq)
    assert_parity("K d256", to64(k), rk)
    assert_parity("V d256", to64(v), rv)


def test_forward_d256_gemma3_width():
    cfg = PREFILL_CONFIGS["gemma3_d256"].with_(B=2, S=700)
    t = make_layer_inputs(cfg, seed=2300)
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D))
    gq.gqa_attn_forward_ex(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                           cfg.rope_theta, cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, True, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, want_stages=True)
    assert_parity("out d256", to64(out).reshape(-1, cfg.hidden), ref["out"])
    tok = cfg.B * cfg.S
    n_q, n_kv = tok * cfg.Hq * D * 2, tok * cfg.Hkv * D * 2
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    off = al(n_q) + 2 * al(n_kv)
    attn = ws[off:off + n_q].view(torch.bfloat16).view(tok, -1)
    assert_parity("attn d256", to64(attn), ref["attn"])


def test_forward_d256_full_workload_sampled():
    """The full Gemma-3-width workload (4 x 4096 tokens) on the launch
    configuration the benchmark times; the oracle evaluates sampled rows."""
    cfg = PREFILL_CONFIGS["gemma3_d256"]
    t = make_layer_inputs(cfg, seed=2400)
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attn_forward(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                        cfg.rope_theta, cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    rows = [0, 1, 63, 64, 65, 127, 128, 2047, 2048, 4095, 4096, 4096 + 77, 3 * 4096 + 4095]
    rows += list(np.random.default_rng(5).integers(0, cfg.B * cfg.S, 48))
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, D, sel=rows)
    assert_parity("out d256 sampled", to64(out).reshape(-1, cfg.hidden)[rows], ref)
