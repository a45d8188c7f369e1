"""Failure detection without a GPU fault: a kernel waits on an mbarrier that
nothing will ever complete; its bounded wait gives up, reports
GQA_ERR_TIMEOUT through the device error word, and the device keeps working."""
import pytest
import torch

from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import PREFILL_CONFIGS, make_layer_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_device_survives():
    assert gq.gqa_check_device_error() == gq.GQA_OK
    rc = gq.gqa_selftest_bounded_wait(200)
    assert rc == gq.GQA_ERR_TIMEOUT, gq.gqa_last_error()
    assert "bounded device wait" in gq.gqa_last_error()
    assert gq.gqa_check_device_error() == gq.GQA_OK  # the word was cleared
    # the device still runs the layer
    cfg = PREFILL_CONFIGS["qwen3_0p6b"]
    t = make_layer_inputs(cfg, seed=1)
    g = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    out = torch.empty_like(g["x"])
    gq.gqa_attn_forward(g["x"], g["Wqkv"], g["Wo"], g["q_norm_w"], g["k_norm_w"], cfg.rope_theta, cfg.eps,
                        cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, True, out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_OK
    assert torch.isfinite(out.float()).all()


def test_selftest_rejects_bad_limit():
    assert gq.gqa_selftest_bounded_wait(0) == gq.GQA_ERR_ARG
    assert gq.gqa_selftest_bounded_wait(100000) == gq.GQA_ERR_ARG


def test_stream_error_check_reports_and_clears():
    """gqa_check_stream_error waits for one stream only: a projection whose Q/K/V
    values pass binary16's range (saturated, flagged) on a private stream is
    reported there, and the word is cleared by the check."""
    assert gq.gqa_check_device_error() == gq.GQA_OK
    s = torch.cuda.Stream()
    B, S, h, Hq, Hkv, d = 1, 128, 64, 1, 1, 64
    x = torch.full((B, S, h), 2000.0, device="cuda").to(torch.bfloat16)  # q = 2000 * 64 > 65504
    W = torch.ones(((Hq + 2 * Hkv) * d, h), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((B, Hq, S, d), dtype=torch.float16, device="cuda")
    k = torch.empty((B, Hkv, S, d), dtype=torch.float16, device="cuda")
    v = torch.empty_like(k)
    s.wait_stream(torch.cuda.current_stream())
    gq.gqa_qkv_proj(x, W, None, None, 1e4, 1e-6, B, S, h, Hq, Hkv, d, q, k, v, s)
    assert gq.gqa_check_stream_error(s) == gq.GQA_ERR_RANGE
    assert "binary16 range" in gq.gqa_last_error()
    assert gq.gqa_check_stream_error(s) == gq.GQA_OK
    # saturated, not infinite
    assert float(v.float().abs().max()) == 65504.0
    # in range: nothing to report
    x.fill_(0.5)
    s.wait_stream(torch.cuda.current_stream())
    gq.gqa_qkv_proj(x, W, None, None, 1e4, 1e-6, B, S, h, Hq, Hkv, d, q, k, v, s)
    assert gq.gqa_check_stream_error(s) == gq.GQA_OK
    assert gq.gqa_check_device_error() == gq.GQA_OK
