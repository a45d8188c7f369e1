"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every function include/gqa_attn.h declares; the cost accounting
matches the counts printed on the pages; argument validation rejects bad calls
with the documented status before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT, golden_rows


@pytest.fixture(scope="module")
def L():
    from transformer_gqa_attention_qkv_gb300.build import build_library
    build_library()
    from transformer_gqa_attention_qkv_gb300 import binding
    return binding


def header_functions():
    src = open(os.path.join(ROOT, "include", "gqa_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_\w+)\s*\(", src)))


def test_exports_match_header(L):
    names = header_functions()
    assert len(names) == 42
    assert sorted(L.EXPORTS) == names
    lib = L.lib()
    for n in names:
        assert hasattr(lib, n), n


def test_cta_pairs_switch_returns_previous_setting(L):
    """gqa_set_cta_pairs is host state only (no device work): it returns the
    previous setting, and the default is on."""
    assert L.gqa_set_cta_pairs(False) is True
    assert L.gqa_set_cta_pairs(False) is False
    assert L.gqa_set_cta_pairs(True) is False
    assert L.gqa_set_cta_pairs(True) is True


def test_cost_matches_capacity_knob_counts(L):
    """[Knob] "Why the cost does not move": weights 4*d_model^2 for any h,
    score+value MACs per token 2*n*d_model (non-causal: every query sees all n
    keys), pinned-128 weight counts."""
    for kind, dm, h, hd, n, val in golden_rows("capacity_knob_counts.txt"):
        dm, h, hd, val = int(dm), int(h), int(hd), int(val)
        S = int(n) if n != "-" else 1
        c = L.gqa_attn_cost(1, S, dm, h, h, hd, causal=False)
        if kind in ("params", "proj_macs"):
            assert c["weights"] == val and c["proj_macs_per_token"] == val
        else:
            assert c["attn_macs"] // S == val
    # causal counts only the S(S+1)/2 visible pairs
    c = L.gqa_attn_cost(2, 10, 64, 4, 2, 16, causal=True)
    assert c["attn_macs"] == 2 * 16 * 4 * 55 * 2
    assert c["flops"] == 2 * (2 * 10 * c["weights"] + c["attn_macs"])


def test_cost_geometry_qwen3_0p6b(L):
    """[NeoX] "Qwen3-0.6B example": QKV 1024 -> 4096 and o_proj 2048 -> 1024."""
    c = L.gqa_attn_cost(1, 1, 1024, 16, 8, 128)
    assert c["weights"] == 1024 * 4096 + 2048 * 1024


FAKE = 1 << 20  # an aligned, never-dereferenced address: validation fails first


def fwd(L, **kw):
    a = dict(x=FAKE, W=FAKE * 2, Wo=FAKE * 3, qn=FAKE * 4, kn=FAKE * 5, theta=1e6, eps=1e-6, B=1, S=16,
             hidden=64, Hq=4, Hkv=2, d=128, causal=1, out=FAKE * 6, ws=FAKE * 8, wsb=1 << 30)
    a.update(kw)
    P = ctypes.c_void_p
    return L.lib().gqa_attn_forward_ex(P(a["x"]), P(a["W"]), P(a["Wo"]), P(a["qn"]), P(a["kn"]), a["theta"],
                                       a["eps"], a["B"], a["S"], a["hidden"], a["Hq"], a["Hkv"], a["d"],
                                       a["causal"], P(a["out"]), P(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    ({"S": 0}, -1), ({"B": -1}, -1), ({"Hq": 3}, -1), ({"d": 127}, -1), ({"qn": 0}, -1),
    ({"d": 160}, -2), ({"d": 512}, -2), ({"d": 320}, -2), ({"hidden": 100}, -2), ({"Hq": 258, "Hkv": 2}, -2),
    ({"x": 0}, -1), ({"out": FAKE + 2}, -1), ({"out": FAKE}, -1), ({"theta": 0.0}, -1),
    ({"wsb": 100}, -5), ({"ws": 0}, -5), ({"ws": FAKE * 8 + 16}, -1),
])
def test_forward_validation(L, kw, code):
    assert fwd(L, **kw) == code
    msg = L.gqa_last_error()
    assert msg
    if code == -2 and "d" in kw:
        assert "head_dim" in msg and str(kw["d"]) in msg  # names the dimension


def test_other_entry_points_validate(L):
    lib = L.lib()
    P = ctypes.c_void_p
    assert lib.gqa_attention(P(FAKE), P(FAKE), P(FAKE), 1, 8, 6, 4, 128, 1, P(FAKE), None) == -1
    assert lib.gqa_oproj_residual(P(FAKE), P(FAKE), P(FAKE), 4, 100, 64, P(FAKE * 2), None) == -2
    assert lib.gqa_oproj_residual(P(FAKE), P(FAKE), P(FAKE), 4, 64, 64, P(FAKE), None) == -1
    assert lib.gqa_decode_attention(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 2, 260, 2, 128, 100, P(FAKE), P(FAKE),
                                    1 << 30, None) == -2   # group of 130
    assert lib.gqa_decode_attention(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 2, 8, 2, 160, 100, P(FAKE), P(FAKE),
                                    1 << 30, None) == -2   # decode: no tile for head_dim 160
    assert lib.gqa_attn_decode(P(FAKE), P(FAKE), P(FAKE), None, None, 1e6, 1e-6, 2, 64, 8, 2, 128, P(FAKE),
                               P(FAKE), None, 100, P(FAKE * 3), P(FAKE * 4), 1 << 30, None) == -1  # cache_len NULL
    assert lib.gqa_attn_workspace_size(0, 1, 1, 1, 1, 1) == 0
    assert L.gqa_attn_workspace_size(1, 16, 64, 4, 2, 128) >= 16 * (4 + 2 + 2 + 4) * 128 * 2


def test_resolve_head_dim():
    """[NeoX] "Proposed configuration behavior": an explicit head_dim wins
    (no divisibility needed); without one head_dim = hidden / heads, which
    must divide ([Knob] "Where the invariance breaks": 2560 / 32 = 80)."""
    from transformer_gqa_attention_qkv_gb300.binding import resolve_head_dim
    assert resolve_head_dim(2560, 32) == 80
    assert resolve_head_dim(2560, 32, 128) == 128
    assert resolve_head_dim(1024, 16, 128) == 128      # Qwen3-0.6B: Q width 2048 != hidden
    assert resolve_head_dim(512, 8) == 64               # the Vaswani layer
    assert resolve_head_dim(1000, 16, 128) == 128      # explicit: hidden need not divide
    with pytest.raises(ValueError):
        resolve_head_dim(1000, 16)
    with pytest.raises(ValueError):
        resolve_head_dim(2560, 32, 0)


def test_host_forward_and_training_pair_validate(L):
    """The host-buffer forward and the training pair reject bad arguments
    before touching a device (no GPU needed)."""
    lib = L.lib()
    P = ctypes.c_void_p

    def host(x=FAKE, out=FAKE * 6, d=128, ws=FAKE * 8, wsb=1 << 34):
        return lib.gqa_attn_forward_host(P(x), P(FAKE * 2), P(FAKE * 3), P(FAKE * 4), P(FAKE * 5), 1e6, 1e-6,
                                         1, 16, 64, 4, 2, d, 1, P(out), P(ws), wsb, None)
    assert host(x=0) == -1
    assert host(d=160) == -2
    assert host(out=FAKE) == -1                      # out_host overlaps x_host
    assert host(wsb=100) == -5
    assert host(ws=FAKE * 8 + 16) == -1              # workspace not 256-byte aligned
    assert lib.gqa_attn_forward_host_workspace_size(0, 16, 64, 4, 2, 128) == 0
    assert (L.gqa_attn_forward_host_workspace_size(1, 16, 64, 4, 2, 128)
            >= L.gqa_attn_workspace_size(1, 16, 64, 4, 2, 128) + 2 * 16 * 64 * 2)

    def train(d=128, x=FAKE, wsb=1 << 34):
        return lib.gqa_attn_forward_train(P(x), P(FAKE * 2), P(FAKE * 3), P(FAKE * 4), P(FAKE * 5), 1e6, 1e-6,
                                          1, 16, 64, 4, 2, d, 1, P(FAKE * 6), P(FAKE * 8), wsb, None)
    assert train(x=0) == -1
    assert train(d=256) == -2                        # the backward has no head_dim 256
    assert train(wsb=100) == -5

    def saved(d=128, dout=FAKE * 7):
        return lib.gqa_attn_backward_saved(P(FAKE), P(FAKE * 2), P(FAKE * 3), P(FAKE * 4), P(FAKE * 5), 1e6, 1e-6,
                                           1, 16, 64, 4, 2, d, 1, P(dout), P(FAKE * 9), P(FAKE * 10),
                                           P(FAKE * 11), P(FAKE * 12), P(FAKE * 13), P(FAKE * 16), 100, None)
    assert saved(dout=0) == -1
    assert saved(d=160) == -2
    assert saved() == -5                             # 100 bytes of workspace


def test_error_checks_without_a_device(L):
    """The device error checks report a CUDA failure, not a crash, where no
    device can be reached."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert L.gqa_check_device_error() == L.GQA_ERR_CUDA
    assert L.gqa_last_error()
    assert L.lib().gqa_check_stream_error(ctypes.c_void_p(0)) == L.GQA_ERR_CUDA
    assert L.gqa_last_error()
