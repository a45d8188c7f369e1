"""Parity of partial rotary (rotary_dim < head_dim) with the fp64 oracle (GPU).

RoPE rotates only the first rotary_dim features of each Q and K head (GPT-NeoX
issue page, "Scaling and RoPE": RoPE follows the effective head_dim subject
to rotary_pct).  The kernels implement rotary_dim = head_dim, head_dim/2,
head_dim/4 and 0; head_dim/4 of a 64-wide head (16) and of a 128-wide head
(32) pair features inside one 32-column slice, head_dim/2 of a 128-wide head
pairs two slices.  Checked: the QKV stage alone, the whole prefill layer, the
decode step and the cached prefill, against the oracle with the same width;
rotary_dim = head_dim is bit-identical to the plain entry point; bad widths
are rejected before any launch.

Tolerance: max|err| <= 1e-2 max|ref| and relative L1 <= 2e-3 (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import (DecodeConfig, LayerConfig, make_decode_inputs,
                                                        make_layer_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dev(t):
    return None if t is None else t.to(DEV)


GEOMS = {
    "d128": LayerConfig("d128", B=2, S=300, hidden=1024, Hq=16, Hkv=8, head_dim=128, qk_norm=True, rope_theta=1e6),
    "d64": LayerConfig("d64", B=2, S=257, hidden=512, Hq=8, Hkv=2, head_dim=64, qk_norm=False, rope_theta=1e4),
}


@pytest.mark.parametrize("geom", ["d128", "d64"])
@pytest.mark.parametrize("frac", [2, 4, 0])
def test_qkv_stage_partial_rotary(geom, frac):
    cfg = GEOMS[geom]
    B, S, h, Hq, Hkv, d = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
    rd = d // frac if frac else 0
    t = make_layer_inputs(cfg, seed=1100 + rd, w_std=0.05)
    q = torch.empty((B, Hq, S, d), dtype=torch.float16, device=DEV)
    k = torch.empty((B, Hkv, S, d), dtype=torch.float16, device=DEV)
    v = torch.empty_like(k)
    gq.gqa_qkv_proj_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta, cfg.eps,
                       rd, B, S, h, Hq, Hkv, d, q, k, v)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    rq, rk, rv = oracle.qkv_stage(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                  B, S, h, Hq, Hkv, d, rotary_dim=rd)
    assert_parity(f"Q rd={rd}", to64(q), rq)
    assert_parity(f"K rd={rd}", to64(k), rk)
    assert_parity(f"V rd={rd}", to64(v), rv)
    # the features past the rotary width are not rotated: they match the
    # rotary_dim = 0 result exactly (same arithmetic up to the rotation)
    if rd:
        q0 = torch.empty_like(q)
        k0, v0 = torch.empty_like(k), torch.empty_like(v)
        gq.gqa_qkv_proj_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
                           cfg.eps, 0, B, S, h, Hq, Hkv, d, q0, k0, v0)
        torch.cuda.synchronize()
        assert torch.equal(q[..., rd:], q0[..., rd:]) and torch.equal(k[..., rd:], k0[..., rd:])
        assert torch.equal(v, v0)
        # position 0 is not rotated at all
        assert torch.equal(q[:, :, 0], q0[:, :, 0])


@pytest.mark.parametrize("geom", ["d128", "d64"])
def test_forward_partial_rotary(geom):
    cfg = GEOMS[geom]
    rd = cfg.head_dim // 4
    t = make_layer_inputs(cfg, seed=1200)
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim))
    gq.gqa_attn_forward_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                           cfg.rope_theta, cfg.eps, rd, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, True,
                           out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                         cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, want_stages=True, rotary_dim=rd)
    assert_parity("out", to64(out).reshape(-1, cfg.hidden), ref["out"])
    tok = cfg.B * cfg.S
    n_q = tok * cfg.Hq * cfg.head_dim * 2
    n_kv = tok * cfg.Hkv * cfg.head_dim * 2
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    off = al(n_q) + 2 * al(n_kv)
    attn = ws[off:off + n_q].view(torch.bfloat16).view(tok, -1)
    assert_parity("attn", to64(attn), ref["attn"])


def test_full_width_is_the_plain_entry_point():
    cfg = GEOMS["d128"]
    t = make_layer_inputs(cfg, seed=1300)
    args = (dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
            cfg.eps)
    dims = (cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, True)
    ws = gq.new_workspace(gq.gqa_attn_workspace_size(cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim))
    a = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    gq.gqa_attn_forward_ex(*args, *dims, a, ws)
    gq.gqa_attn_forward_rd(*args, cfg.head_dim, *dims, b, ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_decode_partial_rotary():
    cfg = DecodeConfig("t", B=6, cache_len=700, hidden=1024, Hq=16, Hkv=4, head_dim=128, qk_norm=True,
                       rope_theta=1e6, Lmax=720)
    rd = 32
    t = make_decode_inputs(cfg, seed=1400)
    cl = torch.tensor([700, 1, 0, 333, 64, 719], dtype=torch.int32)
    kc, vc = dev(t["k_cache"]), dev(t["v_cache"])
    out = torch.empty((cfg.B, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_decode_workspace_size(cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                                                            cfg.lmax))
    gq.gqa_attn_decode_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                          cfg.rope_theta, cfg.eps, rd, cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc,
                          dev(cl), cfg.lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                        cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, t["k_cache"], t["v_cache"], cl, cfg.lmax,
                        rotary_dim=rd)
    idx = cl.long().to(DEV)
    ar = torch.arange(cfg.B, device=DEV)
    assert_parity("k appended", to64(kc[ar, :, idx]), ref["k"])
    assert_parity("v appended", to64(vc[ar, :, idx]), ref["v"])
    # the decode's own attention output, in the workspace after q
    n_q = cfg.B * cfg.Hq * cfg.head_dim * 2
    off = (n_q + 255) // 256 * 256
    attn = ws[off:off + n_q].view(torch.bfloat16).view(cfg.B, -1)
    assert_parity("attn", to64(attn), ref["attn"])
    assert_parity("out", to64(out), ref["out"])


def test_prefill_cached_partial_rotary():
    cfg = GEOMS["d128"].with_(B=2, S=150)
    rd, Lmax, p0 = 64, 512, [0, 301]
    t = make_layer_inputs(cfg, seed=1500)
    g = torch.Generator().manual_seed(1501)
    kc = torch.zeros((cfg.B, cfg.Hkv, Lmax, cfg.head_dim), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for b, p in enumerate(p0):
        kc[b, :, :p] = torch.randn((cfg.Hkv, p, cfg.head_dim), generator=g).to(torch.bfloat16)
        vc[b, :, :p] = torch.randn((cfg.Hkv, p, cfg.head_dim), generator=g).to(torch.bfloat16)
    kd, vd = dev(kc), dev(vc)
    out = torch.empty((cfg.B, cfg.S, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_prefill_cached_workspace_size(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.head_dim, Lmax))
    gq.gqa_attn_prefill_cached_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]),
                                  dev(t["k_norm_w"]), cfg.rope_theta, cfg.eps, rd, cfg.B, cfg.S, cfg.hidden, cfg.Hq,
                                  cfg.Hkv, cfg.head_dim, True, kd, vd, dev(torch.tensor(p0, dtype=torch.int32)),
                                  Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.prefill_cached(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, p0, Lmax,
                                rotary_dim=rd)
    assert_parity("out", to64(out).reshape(-1, cfg.hidden), ref["out"])
    k_after = kd.cpu()
    for b, p in enumerate(p0):
        assert_parity(f"k slots b={b}", to64(k_after[b, :, p:p + cfg.S]), ref["k"][b])


def test_rejects_bad_rotary_widths():
    cfg = GEOMS["d128"].with_(B=1, S=8)
    t = make_layer_inputs(cfg, seed=1)
    q = torch.empty((1, cfg.Hq, 8, 128), dtype=torch.float16, device=DEV)
    k = torch.empty((1, cfg.Hkv, 8, 128), dtype=torch.float16, device=DEV)
    v = torch.empty_like(k)
    for rd, code in ((-2, gq.GQA_ERR_ARG), (31, gq.GQA_ERR_ARG), (130, gq.GQA_ERR_ARG),
                     (96, gq.GQA_ERR_UNSUPPORTED), (24, gq.GQA_ERR_UNSUPPORTED)):
        with pytest.raises(gq.GqaError) as e:
            gq.gqa_qkv_proj_rd(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), 1e6, 1e-6, rd,
                               1, 8, cfg.hidden, cfg.Hq, cfg.Hkv, 128, q, k, v)
        assert f"status {code}" in str(e.value)
