"""The layer forward from host buffers (gqa_attn_forward_host), GPU.

Its token chunks are multiples of the 128-row GEMM tile, so every output
element is computed by the same products in the same order as by the one-shot
gqa_attn_forward_ex: the two must agree bit for bit.  Cases: one chunk, four
chunks, and a ragged two-chunk split whose boundary falls inside a sequence
(rows 0..2559 | 2560..4999 with S = 1000), which checks the chunk's row offset
in the QKV epilogue (positions and head-major slots of the later chunk).  The
small case is also held to the fp64 oracle at the usual tolerance.
"""
import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import LayerConfig, make_layer_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dev(t):
    return None if t is None else t.to(DEV)


CASES = [
    # B, S, hidden, Hq, Hkv, d, qk_norm, chunks
    (1, 128, 1024, 16, 8, 128, True, 1),
    (2, 4096, 512, 8, 2, 128, True, 4),
    (5, 1000, 256, 4, 4, 64, False, 2),
]


@pytest.mark.parametrize("B,S,hidden,Hq,Hkv,d,qk,chunks", CASES)
def test_host_forward_matches_device_forward(B, S, hidden, Hq, Hkv, d, qk, chunks):
    cfg = LayerConfig("h", B, S, hidden, Hq, Hkv, d, qk, 1e6 if qk else 1e4)
    t = make_layer_inputs(cfg, seed=4242 + S, w_std=0.05)
    x_host = t["x"].contiguous().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    W, Wo, qn, kn = dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"])
    ws = gq.new_workspace(gq.gqa_attn_forward_host_workspace_size(B, S, hidden, Hq, Hkv, d), torch.device(DEV))
    out_host.fill_(float("nan"))
    for _ in range(2):  # the second call reuses the pipeline's stream and events
        gq.gqa_attn_forward_host(x_host, W, Wo, qn, kn, cfg.rope_theta, cfg.eps, B, S, hidden, Hq, Hkv, d, True,
                                 out_host, ws)
        torch.cuda.current_stream().synchronize()
        assert gq.gqa_last_launch_count() == 2 * chunks + 1
    assert gq.gqa_check_device_error() == 0
    x = dev(t["x"])
    out = torch.empty_like(x)
    ws2 = gq.new_workspace(gq.gqa_attn_workspace_size(B, S, hidden, Hq, Hkv, d), torch.device(DEV))
    gq.gqa_attn_forward_ex(x, W, Wo, qn, kn, cfg.rope_theta, cfg.eps, B, S, hidden, Hq, Hkv, d, True, out, ws2)
    torch.cuda.synchronize()
    assert torch.equal(out_host.view(torch.int16), out.cpu().view(torch.int16))
    if B * S <= 128:
        ref = oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                             B, S, hidden, Hq, Hkv, d, causal=True)
        assert_parity("out (host forward)", to64(out_host).reshape(ref.shape), ref)


def test_host_forward_rejects_device_buffers():
    cfg = LayerConfig("h", 1, 128, 256, 2, 1, 128, True, 1e6)
    t = make_layer_inputs(cfg, seed=7)
    x = dev(t["x"])
    ws = gq.new_workspace(gq.gqa_attn_forward_host_workspace_size(1, 128, 256, 2, 1, 128), torch.device(DEV))
    with pytest.raises(ValueError):
        gq.gqa_attn_forward_host(x, dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"]), 1e6, 1e-6,
                                 1, 128, 256, 2, 1, 128, True, torch.empty_like(t["x"]), ws)
    # the C-ABI itself checks too (the binding's own check bypassed)
    rc = gq.lib().gqa_attn_forward_host(gq._ptr(x), gq._bf16(dev(t["Wqkv"])), gq._bf16(dev(t["Wo"])),
                                        gq._bf16(dev(t["q_norm_w"])), gq._bf16(dev(t["k_norm_w"])), 1e6, 1e-6,
                                        1, 128, 256, 2, 1, 128, 1, gq._host_bf16(torch.empty_like(t["x"])),
                                        gq._ptr(ws), ws.numel(), gq._stream(None))
    assert rc == -1


def test_host_forward_from_pageable_memory():
    """Page-locked memory is only faster: pageable x and out give the same
    bits (the copies then run synchronously with the host)."""
    cfg = LayerConfig("h", 2, 2048, 256, 4, 2, 128, True, 1e6)
    t = make_layer_inputs(cfg, seed=4343)
    x_host = t["x"].contiguous()
    assert not x_host.is_pinned()
    out_host = torch.empty_like(x_host)
    W, Wo, qn, kn = dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"])
    ws = gq.new_workspace(gq.gqa_attn_forward_host_workspace_size(2, 2048, 256, 4, 2, 128), torch.device(DEV))
    gq.gqa_attn_forward_host(x_host, W, Wo, qn, kn, 1e6, cfg.eps, 2, 2048, 256, 4, 2, 128, True, out_host, ws)
    torch.cuda.current_stream().synchronize()
    x = dev(t["x"])
    out = torch.empty_like(x)
    gq.gqa_attn_forward_ex(x, W, Wo, qn, kn, 1e6, cfg.eps, 2, 2048, 256, 4, 2, 128, True, out,
                           gq.new_workspace(gq.gqa_attn_workspace_size(2, 2048, 256, 4, 2, 128), torch.device(DEV)))
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    assert torch.equal(out_host.view(torch.int16), out.cpu().view(torch.int16))
