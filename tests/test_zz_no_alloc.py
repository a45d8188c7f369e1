"""The decode attention entry point for callers that cannot allocate device
memory (gqa_decode_attention_noalloc), called through the C ABI.

Such callers (custom-op hosts that pass only inputs and outputs, serving loops
whose memory belongs to another allocator) get no workspace argument: the
split partials live in a fixed array inside the library.  The test checks the
result against the workspace-taking gqa_decode_attention on two calls in a
row with different inputs, so a stale partial left in the shared array by the
first call would show up in the second.  It is collected last and stands
alone: it builds its own inputs and needs no state from other tests.
"""
import ctypes

import pytest
import torch

from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq

pytestmark = pytest.mark.gpu


def _reference(q, kc, vc, kl, B, Hq, Hkv, d, Lmax):
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device="cuda")
    ws = gq.new_workspace(gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax))
    gq.gqa_decode_attention(q, kc, vc, kl, B, Hq, Hkv, d, Lmax, out, ws)
    return out


def _noalloc_via_cabi(q, kc, vc, kl, B, Hq, Hkv, d, Lmax):
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device="cuda")
    P = ctypes.c_void_p
    rc = gq.lib().gqa_decode_attention_noalloc(P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()),
                                               P(kl.data_ptr()), B, Hq, Hkv, d, Lmax, P(out.data_ptr()),
                                               P(torch.cuda.current_stream().cuda_stream))
    assert rc == gq.GQA_OK, gq.gqa_last_error()
    return out


@pytest.mark.parametrize("B,Hq,Hkv,d,Lmax", [(64, 32, 8, 128, 8193), (3, 8, 8, 64, 700)])
def test_noalloc_matches_workspace_entry_point_twice(B, Hq, Hkv, d, Lmax):
    g = torch.Generator(device="cuda").manual_seed(900 + B)
    for call in range(2):
        q = (torch.randn((B, Hq, d), generator=g, device="cuda") * 1.5).to(torch.float16)
        kc = torch.randn((B, Hkv, Lmax, d), generator=g, device="cuda").to(torch.bfloat16)
        vc = torch.randn((B, Hkv, Lmax, d), generator=g, device="cuda").to(torch.bfloat16)
        # ragged lengths that differ between the two calls
        kl = torch.randint(1, Lmax + 1, (B,), generator=g, device="cuda", dtype=torch.int32)
        kl[0] = Lmax if call == 0 else 1
        ref = _reference(q, kc, vc, kl, B, Hq, Hkv, d, Lmax)
        got = _noalloc_via_cabi(q, kc, vc, kl, B, Hq, Hkv, d, Lmax)
        torch.cuda.synchronize()
        assert_parity(f"noalloc call {call + 1}", to64(got), to64(ref))


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    P = ctypes.c_void_p
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    # B*Hq*(d+2) = 4096*64*130 floats > the 4 Mi-float array
    rc = gq.lib().gqa_decode_attention_noalloc(P(dummy.data_ptr()), P(dummy.data_ptr()), P(dummy.data_ptr()),
                                               P(lens.data_ptr()), 4096, 64, 8, 128, 16, P(dummy.data_ptr()), None)
    assert rc == gq.GQA_ERR_UNSUPPORTED
    assert "exceed" in gq.gqa_last_error()
