"""Decode at head widths 80, 96 and 256 (GPU), against the fp64 oracle.

[Knob] "Where the invariance breaks" names 80 (Qwen3-4B's hidden / heads) and
96 as widths kernels must tile; [NeoX] "Background" gives the Gemma-3 example
with head_dim 256.  The split-KV decode stages 80- and 96-wide rows as two
64-wide boxes whose columns past d the tensor copy fills with zeros, and
contracts over the d real columns; 256-wide rows are four boxes.  Groups of
up to 8 heads use the transposed products (keys in the MMA rows), 9 to 16 the
heads-in-rows form (widths up to 128), larger groups split into sub-groups.
Checked: the attention stage over ragged lengths and group sizes, and the
whole decode step (projection with QK-norm and RoPE at the cache position,
append, attention, o_proj) at the Qwen3-4B widths with head_dim 80 and at the
Gemma-3 width with head_dim 256.

Tolerance: max|err| <= 1e-2 max|ref| and relative L1 <= 2e-3 (tests/parity.py).
"""
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import DecodeConfig, make_decode_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dev(t):
    return None if t is None else t.to(DEV)


@pytest.mark.parametrize("d,B,Hq,Hkv,Lmax,lens", [
    (80, 4, 32, 8, 700, [700, 1, 64, 333]),      # G = 4
    (80, 2, 24, 2, 300, [300, 129]),             # G = 12: heads in the MMA rows
    (96, 3, 8, 8, 500, [500, 65, 2]),            # G = 1
    (96, 2, 32, 2, 400, [400, 200]),             # G = 16
    (256, 3, 4, 1, 600, [600, 1, 257]),          # G = 4 (the Gemma-3 head geometry)
    (256, 2, 16, 1, 300, [300, 99]),             # G = 16: two sub-groups of 8
    (256, 2, 6, 2, 130, [130, 64]),              # G = 3
])
def test_decode_attention_width(d, B, Hq, Hkv, Lmax, lens):
    g = torch.Generator().manual_seed(5000 + d + Hq)
    q = (torch.randn((B, Hq, d), generator=g) * 1.5).to(torch.float16)
    kc = torch.randn((B, Hkv, Lmax, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, Lmax, d), generator=g).to(torch.bfloat16)
    kl = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax))
    gq.gqa_decode_attention(dev(q), dev(kc), dev(vc), dev(kl), B, Hq, Hkv, d, Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_attention_stage(q, kc, vc, kl, B, Hq, Hkv, d, Lmax)
    assert_parity(f"decode attn d{d} G={Hq // Hkv}", to64(out), ref)


@pytest.mark.parametrize("name,cfg", [
    ("qwen3_4b_d80", DecodeConfig("t", 16, 2000, 2560, 32, 8, 80, True, 1e6, Lmax=2048)),
    ("knob_d96", DecodeConfig("t", 8, 1000, 3072, 32, 8, 96, True, 1e6, Lmax=1024)),
    ("gemma3_d256", DecodeConfig("t", 8, 3000, 640, 4, 1, 256, True, 1e6, Lmax=3072)),
])
def test_decode_step_width(name, cfg):
    t = make_decode_inputs(cfg, seed=5100 + cfg.head_dim)
    cl = torch.tensor([(cfg.cache_len * (b + 1)) // cfg.B - b for b in range(cfg.B)], dtype=torch.int32)
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
    # workspace layout: q [B,Hq,d] binary16, then attn [B,Hq*d] bf16, each 256-byte aligned
    n = cfg.B * cfg.Hq * cfg.head_dim * 2
    off = (n + 255) // 256 * 256
    attn = ws[off:off + n].view(torch.bfloat16).view(cfg.B, -1)
    assert_parity(f"{name} decode attn", to64(attn), ref["attn"])
    assert_parity(f"{name} decode out", to64(out), ref["out"])
    # the appended key and value: the bf16 cache slots the step wrote
    idx = cl.long()
    kn = kc[torch.arange(cfg.B, device=DEV), :, idx.to(DEV)]
    vn = vc[torch.arange(cfg.B, device=DEV), :, idx.to(DEV)]
    assert_parity(f"{name} k appended", to64(kn), ref["k"])
    assert_parity(f"{name} v appended", to64(vn), ref["v"])
