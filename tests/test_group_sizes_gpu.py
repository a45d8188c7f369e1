"""Grouped-query attention at group sizes that are not a power of two, and
large groups in decode (GPU), against the fp64 oracle.

Each KV head serves G = Hq / Hkv query heads ([T07] §4 step 6; "Attention
head partitions": a KV head's dependencies are all the query heads of its
group).  The pages put no restriction on G beyond Hq being a multiple of Hkv,
so the kernels take any G up to 128:

* prefill packs floor(128 / G) positions of each of the G heads into a
  128-row query tile (the remaining rows are idle), so G = 3, 5, 6, 7, 12 and
  24 are checked stage by stage and as whole layers (Hq = 40 over Hkv = 8 is
  G = 5), with distinguishable per-head values that catch a wrong head-to-group
  map;
* decode over bf16 caches holds up to 16 heads per work item (the MMA's 16
  rows), over E4M3 caches up to 8 (its 8 columns); larger groups are split
  into equal sub-groups, so G = 3, 5, 12, 16, 24 and 32 are checked, with the
  whole decode step at Hq = 64 over Hkv = 4 (G = 16).

Tolerance: max|err| <= 1e-2 max|ref| and relative L1 <= 2e-3 (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import DecodeConfig, LayerConfig, make_decode_inputs, make_layer_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dev(t):
    return None if t is None else t.to(DEV)


def f16_randn(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.float16)


@pytest.mark.parametrize("B,S,Hq,Hkv,d,causal", [
    (2, 300, 24, 8, 128, True),    # G = 3: 42 positions per head in a tile
    (1, 257, 40, 8, 128, True),    # G = 5 (Hq = 40 over 8 KV heads)
    (2, 200, 12, 2, 64, True),     # G = 6
    (1, 333, 7, 1, 128, False),    # G = 7, no mask
    (1, 150, 12, 1, 80, True),     # G = 12, head_dim 80
    (2, 100, 48, 2, 96, True),     # G = 24, head_dim 96
    (1, 130, 6, 2, 256, True),     # G = 3, head_dim 256
    (1, 70, 5, 1, 256, True),      # G = 5, head_dim 256
])
def test_attention_stage_any_group(B, S, Hq, Hkv, d, causal):
    g = torch.Generator().manual_seed(3000 + Hq + S)
    Q = f16_randn((B, Hq, S, d), g, 1.5)
    K = f16_randn((B, Hkv, S, d), g, 1.5)
    V = f16_randn((B, Hkv, S, d), g)
    out = torch.empty((B, S, Hq * d), dtype=torch.bfloat16, device=DEV)
    gq.gqa_attention(dev(Q), dev(K), dev(V), B, S, Hq, Hkv, d, causal, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.attention_stage(Q, K, V, B, S, Hq, Hkv, d, causal=causal)
    assert_parity(f"attn G={Hq // Hkv}", to64(out).reshape(B * S, Hq * d), ref)


@pytest.mark.parametrize("Hq,Hkv", [(15, 3), (40, 8)])
def test_group_map_markers_any_group(Hq, Hkv):
    """Every KV head's values are one constant marker, so each query head must
    return exactly its group's marker (g = j // G)."""
    B, S, d = 2, 150, 128
    g = torch.Generator().manual_seed(3100 + Hq)
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


@pytest.mark.parametrize("B,S,hidden,Hq,Hkv,d", [
    (2, 200, 1024, 40, 8, 128),   # G = 5
    (1, 300, 768, 18, 3, 64),     # G = 6
])
def test_layer_forward_any_group(B, S, hidden, Hq, Hkv, d):
    cfg = LayerConfig("t", B, S, hidden, Hq, Hkv, d, True, 1e6)
    t = make_layer_inputs(cfg, seed=3200 + Hq, w_std=0.05)
    out = torch.empty((B, S, hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_workspace_size(B, S, hidden, Hq, Hkv, d))
    gq.gqa_attn_forward_ex(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                           cfg.rope_theta, cfg.eps, B, S, hidden, Hq, Hkv, d, True, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         B, S, hidden, Hq, Hkv, d, want_stages=True)
    # the attention output from the workspace (after Q, K and V), then the layer
    n_q, n_kv = B * S * Hq * d * 2, B * S * Hkv * d * 2
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    o0 = al(n_q) + 2 * al(n_kv)
    attn = ws[o0:o0 + n_q].view(torch.bfloat16)
    assert_parity("attn", to64(attn).reshape(B * S, Hq * d), ref["attn"])
    assert_parity("out", to64(out).reshape(B * S, hidden), ref["out"])


@pytest.mark.parametrize("B,Hq,Hkv,d,Lmax,lens", [
    (3, 9, 3, 128, 700, [700, 65, 1]),          # G = 3
    (2, 10, 2, 64, 300, [300, 129]),            # G = 5
    (2, 24, 2, 128, 1000, [1000, 333]),         # G = 12: rows 8..11 of the MMA
    (3, 64, 4, 128, 2000, [2000, 1, 1500]),     # G = 16: all 16 rows
    (2, 48, 2, 64, 500, [500, 77]),             # G = 24: two sub-groups of 12
    (2, 64, 2, 128, 800, [800, 640]),           # G = 32: two sub-groups of 16
])
def test_decode_attention_any_group(B, Hq, Hkv, d, Lmax, lens):
    g = torch.Generator().manual_seed(3300 + Hq + Lmax)
    q = f16_randn((B, Hq, d), g, 1.5)
    kc = (torch.randn((B, Hkv, Lmax, d), generator=g)).to(torch.bfloat16)
    vc = (torch.randn((B, Hkv, Lmax, d), generator=g)).to(torch.bfloat16)
    kl = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax))
    gq.gqa_decode_attention(dev(q), dev(kc), dev(vc), dev(kl), B, Hq, Hkv, d, Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_attention_stage(q, kc, vc, kl, B, Hq, Hkv, d, Lmax)
    assert_parity(f"decode attn G={Hq // Hkv}", to64(out), ref)


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (3, 9, 3, 700, [700, 65, 1]),        # G = 3
    (2, 32, 2, 1000, [1000, 333]),       # G = 16: two sub-groups of 8
    (2, 64, 2, 500, [500, 130]),         # G = 32: four sub-groups of 8
    (2, 24, 1, 300, [300, 299]),         # G = 24: three sub-groups of 8
])
def test_decode_attention_fp8_any_group(B, Hq, Hkv, Lmax, lens):
    d, ks, vs = 128, 2.0 ** -5, 0.03
    g = torch.Generator().manual_seed(3400 + Hq + Lmax)
    q = f16_randn((B, Hq, d), g, 1.5)
    kc = (torch.randn((B, Hkv, Lmax, d), generator=g).double() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (torch.randn((B, Hkv, Lmax, d), generator=g).double() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
    for b, n in enumerate(lens):  # never-written slots: NaN codes
        if n < Lmax:
            kc[b, :, n:] = 0x7F
            vc[b, :, n:] = 0x7F
    kl = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax))
    gq.gqa_decode_attention_fp8(dev(q), dev(kc), dev(vc), ks, vs, dev(kl), B, Hq, Hkv, d, Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_attention_stage_fp8(q, kc, vc, ks, vs, kl, B, Hq, Hkv, d, Lmax)
    assert_parity(f"fp8 decode attn G={Hq // Hkv}", to64(out), ref)


def test_decode_step_group_of_16():
    """The whole decode step with 64 query heads over 4 KV heads."""
    cfg = DecodeConfig("t", 8, 1000, 2048, 64, 4, 128, True, 1e6, Lmax=1024)
    t = make_decode_inputs(cfg, seed=3500)
    cl = torch.tensor([1000, 0, 1, 511, 512, 777, 1023, 64], dtype=torch.int32)
    kc, vc = dev(t["k_cache"]), dev(t["v_cache"])
    out = torch.empty((cfg.B, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_decode_workspace_size(cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                                                            cfg.lmax))
    gq.gqa_attn_decode(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                       cfg.rope_theta, cfg.eps, cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, dev(cl),
                       cfg.lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                        cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, t["k_cache"], t["v_cache"], cl, cfg.lmax)
    n = cfg.B * cfg.Hq * cfg.head_dim * 2
    attn = ws[(n + 255) // 256 * 256:(n + 255) // 256 * 256 + n].view(torch.bfloat16)
    assert_parity("decode attn", to64(attn).reshape(cfg.B, -1), ref["attn"])
    assert_parity("decode out", to64(out), ref["out"])


def test_group_beyond_128_is_rejected():
    q = torch.zeros((1, 130, 4, 64), dtype=torch.float16, device=DEV)
    k = torch.zeros((1, 1, 4, 64), dtype=torch.float16, device=DEV)
    out = torch.empty((1, 4, 130 * 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gq.GqaError, match=f"status {gq.GQA_ERR_UNSUPPORTED}"):
        gq.gqa_attention(q, k, k, 1, 4, 130, 1, 64, True, out)
