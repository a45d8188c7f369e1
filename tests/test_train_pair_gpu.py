"""The training pair (GPU): gqa_attn_forward_train keeps the backward's inputs in
the backward workspace and gqa_attn_backward_saved uses them instead of
recomputing the QKV projection and the forward attention.

Both run the same kernels on the same inputs as gqa_attn_forward_ex and
gqa_attn_backward, so out, dx, dWqkv and dWo must agree with those bit for bit;
the norm-weight gradients are sums of per-row terms added in a nondeterministic
order, so they are held to a relative 1e-5.  One case is also held to the
fp64 oracle at the backward's tolerance.
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


def grads(cfg):
    d, h = cfg.head_dim, cfg.hidden
    N = (cfg.Hq + 2 * cfg.Hkv) * d
    return (torch.empty((cfg.B, cfg.S, h), dtype=torch.bfloat16, device=DEV),
            torch.empty((N, h), dtype=torch.float32, device=DEV),
            torch.empty((h, cfg.Hq * d), dtype=torch.float32, device=DEV),
            torch.empty(d, dtype=torch.float32, device=DEV) if cfg.qk_norm else None,
            torch.empty(d, dtype=torch.float32, device=DEV) if cfg.qk_norm else None)


@pytest.mark.parametrize("geom,causal,oracle_check", [
    ({"B": 2, "S": 300, "hidden": 512, "Hq": 8, "Hkv": 2, "head_dim": 128, "qk_norm": True, "rope_theta": 1e6},
     True, True),
    ({"B": 1, "S": 200, "hidden": 256, "Hq": 4, "Hkv": 4, "head_dim": 64, "qk_norm": False, "rope_theta": 1e4},
     False, False),
])
def test_forward_train_then_backward_saved(geom, causal, oracle_check):
    cfg = LayerConfig("t", **geom)
    B, S, h, Hq, Hkv, d = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
    t = make_layer_inputs(cfg, seed=5100 + S, w_std=0.05)
    x, W, Wo, qn, kn = dev(t["x"]), dev(t["Wqkv"]), dev(t["Wo"]), dev(t["q_norm_w"]), dev(t["k_norm_w"])
    dout = dev((torch.randn((B * S, h), generator=torch.Generator().manual_seed(5101)) * 0.5).to(torch.bfloat16))
    nbytes = gq.gqa_attn_backward_workspace_size(B, S, h, Hq, Hkv, d)
    # the training pair
    ws = gq.new_workspace(nbytes)
    out = torch.empty_like(x)
    gq.gqa_attn_forward_train(x, W, Wo, qn, kn, cfg.rope_theta, cfg.eps, B, S, h, Hq, Hkv, d, causal, out, ws)
    g1 = grads(cfg)
    gq.gqa_attn_backward_saved(x, W, Wo, qn, kn, cfg.rope_theta, cfg.eps, B, S, h, Hq, Hkv, d, causal, dout, *g1, ws)
    # the one-shot forward and the recomputing backward
    out_ref = torch.empty_like(x)
    fws = gq.new_workspace(gq.gqa_attn_workspace_size(B, S, h, Hq, Hkv, d))
    gq.gqa_attn_forward_ex(x, W, Wo, qn, kn, cfg.rope_theta, cfg.eps, B, S, h, Hq, Hkv, d, causal, out_ref, fws)
    g2 = grads(cfg)
    gq.gqa_attn_backward(x, W, Wo, qn, kn, cfg.rope_theta, cfg.eps, B, S, h, Hq, Hkv, d, causal, dout, *g2,
                         gq.new_workspace(nbytes))
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))
    for name, a, b in zip(("dx", "dWqkv", "dWo"), g1[:3], g2[:3]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), name
    if cfg.qk_norm:
        for a, b in zip(g1[3:], g2[3:]):
            torch.testing.assert_close(a, b, rtol=1e-5, atol=1e-6 * float(b.abs().max()))
    if oracle_check:
        ref = oracle.backward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                              B, S, h, Hq, Hkv, d, dout.cpu(), causal=causal)
        tol = dict(tol_max=2e-2, tol_rel=1e-2)
        assert_parity("dWo (saved)", g1[2].cpu().double().numpy(), ref["dWo"], **tol)
        assert_parity("dWqkv (saved)", g1[1].cpu().double().numpy(), ref["dWqkv"], **tol)
