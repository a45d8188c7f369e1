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
