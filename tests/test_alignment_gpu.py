"""Outputs that are 16-byte aligned but not 32-byte aligned (GPU).

The interface promises 16-byte alignment only; the GEMM epilogues store
32 bytes at a time where an output row allows it and two 16-byte stores where
it does not.  Both must give the same bits: the QKV stage and o_proj are run
once into 32-byte-aligned outputs and once into outputs offset by 16 bytes.
"""
import pytest
import torch

from transformer_gqa_attention_qkv_gb300 import binding as gq
from transformer_gqa_attention_qkv_gb300.inputs import LayerConfig, make_layer_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def offset_empty(shape, dtype, offset_elems):
    """A contiguous tensor whose data starts offset_elems past a 256-byte-aligned allocation."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.empty(n + offset_elems, dtype=dtype, device=DEV)
    assert buf.data_ptr() % 256 == 0
    return buf[offset_elems:].view(shape)


@pytest.mark.parametrize("d", [128, 256])
def test_qkv_stage_outputs_off_32_byte_alignment(d):
    cfg = LayerConfig("a", 2, 256, 512, 4, 2, d, True, 1e6)
    t = make_layer_inputs(cfg, seed=6100 + d)
    args = [t[k].to(DEV) if t[k] is not None else None for k in ("x", "Wqkv", "q_norm_w", "k_norm_w")]
    outs = []
    for off in (0, 8):  # 8 binary16 elements = 16 bytes
        q = offset_empty((2, 4, 256, d), torch.float16, off)
        k = offset_empty((2, 2, 256, d), torch.float16, off)
        v = offset_empty((2, 2, 256, d), torch.float16, off)
        assert (q.data_ptr() % 32 == 16) == (off == 8)
        gq.gqa_qkv_proj(*args, cfg.rope_theta, cfg.eps, 2, 256, 512, 4, 2, d, q, k, v)
        outs.append((q, k, v))
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_oproj_output_off_32_byte_alignment():
    g = torch.Generator().manual_seed(6200)
    M, hidden, qw = 300, 640, 512
    attn = (torch.randn((M, qw), generator=g) * 0.5).to(torch.bfloat16).to(DEV)
    Wo = (torch.randn((hidden, qw), generator=g) * 0.05).to(torch.bfloat16).to(DEV)
    x = torch.randn((M, hidden), generator=g).to(torch.bfloat16).to(DEV)
    outs = []
    for off in (0, 8):  # 8 bf16 elements = 16 bytes
        out = offset_empty((M, hidden), torch.bfloat16, off)
        gq.gqa_oproj_residual(attn, Wo, x, M, hidden, qw, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
