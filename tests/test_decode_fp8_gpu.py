"""Parity of the decode step over FP8 (E4M3) KV caches with the fp64 oracle (GPU).

A cache element is an E4M3 code worth code * k_scale (keys) or code * v_scale
(values) ("Head Dimension" article, §5.2: FP8 for the K, V cache).  The
oracle attends over exactly the dequantised codes, so the attention and the
layer output are held to the standard tolerance; the codes the step appends
are the nearest codes of the new key / value over their scale, which the GPU
computes from fp32 values and the oracle from fp64 values, so they are held
to agreement on all but near-tie elements and to E4M3's half-step bound.

Checked: the attention stage over ragged lengths and every group size (slots
past each sequence hold NaN codes, which must not leak), the projection and
append stage, the whole step on a reduced and on the full Qwen3-8B-shaped
workload, saturation reporting, and argument checks.  Head widths 64, 80 and
96 (rows staged as 128 codes, the tensor copy filling codes past d with zeros)
and 256 (rows of two 128-code boxes): the attention stage and the whole step
at the widths' workloads ([Knob] "Where the invariance breaks"; [NeoX]
"Background", Gemma-3's head_dim 256).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import DECODE_CONFIGS, DecodeConfig, make_decode_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAN_CODE = 0x7F


def dev(t):
    return None if t is None else t.to(DEV)


def quantize(x: torch.Tensor, scale: float) -> torch.Tensor:
    """Nearest E4M3 codes of x / scale (in-range inputs), as uint8."""
    return (x.double() / scale).to(torch.float8_e4m3fn).view(torch.uint8)


def fp8_caches(cfg, t, k_scale, v_scale, lens=None):
    """The bf16 test caches of make_decode_inputs as E4M3 codes; slots at or
    past lens[b] (if given) hold NaN codes."""
    kc, vc = quantize(t["k_cache"], k_scale), quantize(t["v_cache"], v_scale)
    if lens is not None:
        for b, n in enumerate(lens):
            kc[b, :, n:] = NAN_CODE
            vc[b, :, n:] = NAN_CODE
    return kc.contiguous(), vc.contiguous()


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (4, 16, 4, 1000, [1, 5, 300, 1000]),
    (3, 8, 8, 700, [700, 64, 129]),
    (2, 16, 2, 5000, [5000, 2049]),
    (5, 8, 1, 65, [65, 64, 63, 2, 1]),
])
def test_decode_attention_fp8_stage(B, Hq, Hkv, Lmax, lens):
    d, ks, vs = 128, 2.0 ** -5, 0.03
    g = torch.Generator().manual_seed(1600 + Lmax)
    q = (torch.randn((B, Hq, d), generator=g) * 1.5).to(torch.float16)
    kc = quantize(torch.randn((B, Hkv, Lmax, d), generator=g), ks)
    vc = quantize(torch.randn((B, Hkv, Lmax, d), generator=g), vs)
    for b, n in enumerate(lens):  # never-written slots: NaN codes
        if n < Lmax:
            kc[b, :, n:] = NAN_CODE
            vc[b, :, n:] = NAN_CODE
    kl = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax))
    gq.gqa_decode_attention_fp8(dev(q), dev(kc), dev(vc), ks, vs, dev(kl), B, Hq, Hkv, d, Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_attention_stage_fp8(q, kc, vc, ks, vs, kl, B, Hq, Hkv, d, Lmax)
    assert_parity("fp8 decode attn", to64(out), ref)


@pytest.mark.parametrize("d,B,Hq,Hkv,Lmax,lens", [
    (64, 4, 16, 4, 700, [700, 1, 64, 333]),
    (80, 3, 32, 8, 500, [500, 65, 2]),
    (96, 2, 8, 8, 300, [300, 129]),
    (256, 3, 4, 1, 600, [600, 1, 257]),  # the Gemma-3 head geometry
    (256, 2, 16, 2, 200, [200, 99]),     # G = 8
])
def test_decode_attention_fp8_widths(d, B, Hq, Hkv, Lmax, lens):
    ks, vs = 2.0 ** -5, 0.03
    g = torch.Generator().manual_seed(1650 + d + Hq)
    q = (torch.randn((B, Hq, d), generator=g) * 1.5).to(torch.float16)
    kc = quantize(torch.randn((B, Hkv, Lmax, d), generator=g), ks)
    vc = quantize(torch.randn((B, Hkv, Lmax, d), generator=g), vs)
    for b, n in enumerate(lens):  # never-written slots: NaN codes
        if n < Lmax:
            kc[b, :, n:] = NAN_CODE
            vc[b, :, n:] = NAN_CODE
    kl = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax))
    gq.gqa_decode_attention_fp8(dev(q), dev(kc), dev(vc), ks, vs, dev(kl), B, Hq, Hkv, d, Lmax, out, ws)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_attention_stage_fp8(q, kc, vc, ks, vs, kl, B, Hq, Hkv, d, Lmax)
    assert_parity(f"fp8 decode attn d{d}", to64(out), ref)


def _check_appended(name, codes_gpu, ref_vals, ref_codes, scale):
    """Appended codes: equal to the oracle's except at near-ties, and within
    half an E4M3 step (2^-4 relative, 2^-10 absolute in code units)."""
    got = oracle.e4m3_decode(codes_gpu) * scale
    bound = np.maximum(np.abs(ref_vals) * 2.0 ** -4, 2.0 ** -10 * scale) * (1 + 1e-5) + 1e-7 * np.abs(ref_vals)
    err = np.abs(got - ref_vals)
    assert np.all(err <= bound), (name, float((err - bound).max()))
    same = float((codes_gpu == ref_codes).mean())
    print(f"{name}: {same:.5f} of codes equal to the oracle's")
    assert same >= 0.995, (name, same)


@pytest.mark.parametrize("B,L,hidden,Hq,Hkv,qk", [
    (4, 300, 1024, 16, 8, True),
    (3, 17, 512, 8, 8, False),
    (64, 8192, 4096, 32, 8, True),
])
def test_decode_qkv_fp8_append(B, L, hidden, Hq, Hkv, qk):
    d, ks, vs = 128, 2.0 ** -5, 2.0 ** -5
    cfg = DecodeConfig("t", B, L, hidden, Hq, Hkv, d, qk, 1e6, Lmax=L + 3)
    t = make_decode_inputs(cfg, seed=1700 + B)
    cl = torch.tensor([max(0, L - 5 * b) for b in range(B)], dtype=torch.int32)
    kc8, vc8 = fp8_caches(cfg, t, ks, vs)
    kd, vd = dev(kc8), dev(vc8)
    q = torch.empty((B, Hq, d), dtype=torch.float16, device=DEV)
    gq.gqa_decode_qkv_fp8(dev(t["x"]), dev(t["Wqkv"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), cfg.rope_theta,
                          cfg.eps, B, hidden, Hq, Hkv, d, kd, vd, ks, vs, dev(cl), cfg.lmax, q)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_fp8(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                            B, hidden, Hq, Hkv, d, kc8, vc8, ks, vs, cl, cfg.lmax)
    assert_parity("q", to64(q), ref["q"])
    idx = cl.long()
    ka, va = kd.cpu(), vd.cpu()
    ar = torch.arange(B)
    _check_appended("k codes", ka[ar, :, idx].numpy(), ref["k"], ref["k_code"], ks)
    _check_appended("v codes", va[ar, :, idx].numpy(), ref["v"], ref["v_code"], vs)
    mask = torch.ones((B, cfg.lmax), dtype=torch.bool)
    mask[ar, idx] = False
    assert torch.equal(ka.permute(0, 2, 1, 3)[mask], kc8.permute(0, 2, 1, 3)[mask])
    assert torch.equal(va.permute(0, 2, 1, 3)[mask], vc8.permute(0, 2, 1, 3)[mask])


def _run_step(cfg, t, kc8, vc8, ks, vs, cl):
    kd, vd = dev(kc8), dev(vc8)
    out = torch.empty((cfg.B, cfg.hidden), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(gq.gqa_attn_decode_workspace_size(cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                                                            cfg.lmax))
    gq.gqa_attn_decode_fp8(dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]),
                           cfg.rope_theta, cfg.eps, cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kd, vd, ks,
                           vs, dev(cl), cfg.lmax, out, ws)
    torch.cuda.synchronize()
    n_q = cfg.B * cfg.Hq * cfg.head_dim * 2
    off = (n_q + 255) // 256 * 256
    attn = ws[off:off + n_q].view(torch.bfloat16).view(cfg.B, -1)
    return out, attn


@pytest.mark.parametrize("name,over", [
    ("reduced", {"B": 6, "cache_len": 700, "Lmax": 720}),
    ("qwen3_8b_decode", {}),
])
def test_decode_fp8_step(name, over):
    cfg = DECODE_CONFIGS["qwen3_8b_decode"].with_(**over)
    ks, vs = 2.0 ** -5, 2.0 ** -5
    t = make_decode_inputs(cfg, seed=1800)
    cl = torch.full((cfg.B,), cfg.cache_len, dtype=torch.int32)
    if name == "reduced":
        cl = torch.tensor([700, 1, 0, 333, 64, 719], dtype=torch.int32)
    kc8, vc8 = fp8_caches(cfg, t, ks, vs, lens=None)
    out, attn = _run_step(cfg, t, kc8, vc8, ks, vs, cl)
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_fp8(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                            cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc8, vc8, ks, vs, cl, cfg.lmax)
    assert_parity("attn", to64(attn), ref["attn"])
    assert_parity("out", to64(out), ref["out"])


@pytest.mark.parametrize("name,cfg", [
    ("qwen3_0p6b_d64", DecodeConfig("t", 8, 700, 1024, 16, 8, 64, True, 1e6, Lmax=720)),
    ("qwen3_4b_d80", DecodeConfig("t", 16, 2000, 2560, 32, 8, 80, True, 1e6, Lmax=2048)),
    ("knob_d96", DecodeConfig("t", 8, 1000, 3072, 32, 8, 96, True, 1e6, Lmax=1024)),
    ("gemma3_d256", DecodeConfig("t", 8, 3000, 640, 4, 1, 256, True, 1e6, Lmax=3072)),
])
def test_decode_fp8_step_widths(name, cfg):
    ks, vs = 2.0 ** -5, 2.0 ** -5
    t = make_decode_inputs(cfg, seed=1850 + cfg.head_dim)
    cl = torch.tensor([(cfg.cache_len * (b + 1)) // cfg.B - b for b in range(cfg.B)], dtype=torch.int32)
    kc8, vc8 = fp8_caches(cfg, t, ks, vs, lens=None)
    out, attn = _run_step(cfg, t, kc8, vc8, ks, vs, cl)
    assert gq.gqa_check_device_error() == 0
    ref = oracle.decode_fp8(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                            cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc8, vc8, ks, vs, cl, cfg.lmax)
    assert_parity(f"{name} fp8 attn", to64(attn), ref["attn"])
    assert_parity(f"{name} fp8 out", to64(out), ref["out"])


def test_fp8_saturation_is_reported():
    cfg = DECODE_CONFIGS["qwen3_8b_decode"].with_(B=2, cache_len=40, Lmax=64)
    t = make_decode_inputs(cfg, seed=1900)
    kc8, vc8 = fp8_caches(cfg, t, 1.0, 1.0)
    cl = torch.tensor([40, 3], dtype=torch.int32)
    _, _ = _run_step(cfg, t, kc8, vc8, 1e-4, 1.0, cl)  # keys / 1e-4 far beyond 448
    assert gq.gqa_check_device_error() == gq.GQA_ERR_RANGE
    assert gq.gqa_check_device_error() == gq.GQA_OK  # the flag was cleared


def test_fp8_argument_checks():
    q = torch.zeros((1, 8, 160), dtype=torch.float16, device=DEV)
    c = torch.zeros((1, 1, 16, 160), dtype=torch.uint8, device=DEV)
    kl = torch.ones(1, dtype=torch.int32, device=DEV)
    out = torch.empty((1, 8 * 160), dtype=torch.bfloat16, device=DEV)
    ws = gq.new_workspace(1 << 20)
    with pytest.raises(gq.GqaError, match=f"status {gq.GQA_ERR_UNSUPPORTED}"):
        gq.gqa_decode_attention_fp8(q, c, c, 1.0, 1.0, kl, 1, 8, 1, 160, 16, out, ws)
    q = torch.zeros((1, 8, 128), dtype=torch.float16, device=DEV)
    c = torch.zeros((1, 1, 16, 128), dtype=torch.uint8, device=DEV)
    out = torch.empty((1, 8 * 128), dtype=torch.bfloat16, device=DEV)
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (1.0, float("nan"))):
        with pytest.raises(gq.GqaError, match=f"status {gq.GQA_ERR_ARG}"):
            gq.gqa_decode_attention_fp8(q, c, c, ks, vs, kl, 1, 8, 1, 128, 16, out, ws)
