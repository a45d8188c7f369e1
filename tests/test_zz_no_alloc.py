"""The decode attention entry point for callers that cannot allocate device
memory (gqa_decode_attention_noalloc), called through the C ABI.

Such callers (custom-op hosts that pass only inputs and outputs, serving loops
whose memory belongs to another allocator) get no workspace argument: the
split partials live in a fixed array inside the library.  The tests check the
result against the fp64 oracle on two calls in a row with different inputs,
so a stale partial left in the shared array by the first call would show up
in the second; a workload whose split partials would not fit in the array
(fewer splits than gqa_decode_attention uses) is held to the same tolerance;
and the array's error word is read by gqa_check_device_error() and cleared
by each call.  The file is collected last and stands alone: it builds its own
inputs and needs no state from other tests.
"""
import ctypes

import pytest
import torch

import oracle
from parity import assert_parity, to64
from transformer_gqa_attention_qkv_gb300 import binding as gq

pytestmark = pytest.mark.gpu


def _noalloc_via_cabi(q, kc, vc, kl, B, Hq, Hkv, d, Lmax):
    out = torch.empty((B, Hq * d), dtype=torch.bfloat16, device="cuda")
    P = ctypes.c_void_p
    rc = gq.lib().gqa_decode_attention_noalloc(P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()),
                                               P(kl.data_ptr()), B, Hq, Hkv, d, Lmax, P(out.data_ptr()),
                                               P(torch.cuda.current_stream().cuda_stream))
    assert rc == gq.GQA_OK, gq.gqa_last_error()
    assert gq.gqa_last_launch_count() == 2
    return out


def _inputs(g, B, Hq, Hkv, d, Lmax):
    q = (torch.randn((B, Hq, d), generator=g) * 1.5).to(torch.float16)
    kc = torch.randn((B, Hkv, Lmax, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, Lmax, d), generator=g).to(torch.bfloat16)
    return q, kc, vc


@pytest.mark.parametrize("B,Hq,Hkv,d,Lmax", [(64, 32, 8, 128, 8193), (3, 8, 8, 64, 700)])
def test_noalloc_matches_the_oracle_twice(B, Hq, Hkv, d, Lmax):
    g = torch.Generator().manual_seed(900 + B)
    for call in range(2):
        q, kc, vc = _inputs(g, B, Hq, Hkv, d, Lmax)
        # ragged lengths that differ between the two calls
        kl = torch.randint(1, Lmax + 1, (B,), generator=g, dtype=torch.int32)
        kl[0] = Lmax if call == 0 else 1
        got = _noalloc_via_cabi(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(), B, Hq, Hkv, d, Lmax)
        torch.cuda.synchronize()
        assert gq.gqa_check_device_error() == gq.GQA_OK
        ref = oracle.decode_attention_stage(q, kc, vc, kl, B, Hq, Hkv, d, Lmax)
        assert_parity(f"noalloc call {call + 1}", to64(got), ref)


def test_noalloc_with_fewer_splits_than_the_workspace_path():
    """253 sequences x 64 query heads x head_dim 128: one split's partials take
    2.1 Mi of the array's 4 Mi floats, while gqa_decode_attention would use a
    workspace larger than the array (more splits); the reduced-split result
    still meets the oracle tolerance."""
    B, Hq, Hkv, d, Lmax = 253, 64, 8, 128, 1792
    assert gq.gqa_decode_attention_workspace_size(B, Hq, Hkv, d, Lmax) > 16 * 2 ** 20
    g = torch.Generator().manual_seed(911)
    q, kc, vc = _inputs(g, B, Hq, Hkv, d, Lmax)
    kl = torch.randint(1, Lmax + 1, (B,), generator=g, dtype=torch.int32)
    got = _noalloc_via_cabi(q.cuda(), kc.cuda(), vc.cuda(), kl.cuda(), B, Hq, Hkv, d, Lmax)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_OK
    ref = oracle.decode_attention_stage(q, kc, vc, kl, B, Hq, Hkv, d, Lmax)
    assert_parity("noalloc, reduced splits", to64(got), ref)


def test_noalloc_error_word_is_reported_and_cleared_by_the_next_call():
    """A kv_len of 0 is caught by the kernel's own index check (that sequence
    gets a zero row, nothing is read out of range) and recorded in the
    array's error word.  gqa_check_device_error() reports it after that call;
    a following valid call clears the word before it runs."""
    B, Hq, Hkv, d, Lmax = 2, 8, 4, 128, 64
    g = torch.Generator().manual_seed(913)
    q, kc, vc = (t.cuda() for t in _inputs(g, B, Hq, Hkv, d, Lmax))
    bad = torch.tensor([0, 40], dtype=torch.int32, device="cuda")
    good = torch.tensor([64, 40], dtype=torch.int32, device="cuda")
    out = _noalloc_via_cabi(q, kc, vc, bad, B, Hq, Hkv, d, Lmax)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_ERR_ARG
    assert gq.gqa_check_device_error() == gq.GQA_OK  # read and cleared
    assert torch.count_nonzero(out[0]) == 0
    _noalloc_via_cabi(q, kc, vc, bad, B, Hq, Hkv, d, Lmax)  # flags the word again, unchecked
    _noalloc_via_cabi(q, kc, vc, good, B, Hq, Hkv, d, Lmax)
    torch.cuda.synchronize()
    assert gq.gqa_check_device_error() == gq.GQA_OK


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    P = ctypes.c_void_p
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    # B*Hq*(d+2) = 4096*64*130 floats > the 4 Mi-float array
    rc = gq.lib().gqa_decode_attention_noalloc(P(dummy.data_ptr()), P(dummy.data_ptr()), P(dummy.data_ptr()),
                                               P(lens.data_ptr()), 4096, 64, 8, 128, 16, P(dummy.data_ptr()), None)
    assert rc == gq.GQA_ERR_UNSUPPORTED
    assert "exceed" in gq.gqa_last_error()
    assert gq.gqa_last_launch_count() == 0


def test_noalloc_rejects_what_the_workspace_path_rejects():
    """The same argument checks as gqa_decode_attention, with the same statuses."""
    P = ctypes.c_void_p
    dummy = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    ws = gq.new_workspace(1 << 20)
    for (B, Hq, Hkv, d, Lmax) in ((1, 8, 3, 128, 16), (1, 8, 8, 160, 16), (0, 8, 8, 128, 16),
                                  (1, 8, 8, 128, 0), (1 << 20, 8, 8, 128, 1 << 20)):
        rc = gq.lib().gqa_decode_attention_noalloc(P(dummy.data_ptr()), P(dummy.data_ptr()), P(dummy.data_ptr()),
                                                   P(lens.data_ptr()), B, Hq, Hkv, d, Lmax, P(dummy.data_ptr()),
                                                   None)
        rc_ws = gq.lib().gqa_decode_attention(P(dummy.data_ptr()), P(dummy.data_ptr()), P(dummy.data_ptr()),
                                              P(lens.data_ptr()), B, Hq, Hkv, d, Lmax, P(dummy.data_ptr()),
                                              P(ws.data_ptr()), ws.numel(), None)
        assert rc == rc_ws != gq.GQA_OK, (B, Hq, Hkv, d, Lmax, rc, rc_ws)
