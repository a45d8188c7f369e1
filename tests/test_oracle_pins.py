"""Pins of the fp64 CPU oracle against what the pages and mathematics fix.

Each test ties one step of the oracle to something other than the oracle:
numbers printed on the pages (tests/golden/*.txt, each line cited), closed
forms worked out by hand, invariants of the mathematics, and special cases that
reduce to a library routine evaluated independently (torch in float64 on the
CPU).  The cases are chosen so that a plausible slip (a dropped term, a wrong
sign or index, a transposed operand, an off-by-one in the mask, a wrong head
map) fails at least one of them.

Sources cited by title and section:
  [NeoX]  "Support explicit attention head_dim independent of hidden_size / num_attention_heads"
  [T07]   "Tutorial 07: Multi-Head and Grouped-Query Attention (Full Layer)"
  [Knob]  "num_heads Is Not a Capacity Knob"
  [Part]  "Attention head partitions: keep each head's dependencies intact"
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from conftest import golden_rows
from transformer_gqa_attention_qkv_gb300.inputs import LayerConfig, make_layer_inputs

T = 4  # oracle threads in these tests


def bf16(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.float().double()


def _bf16_rne(x):
    """float64 -> nearest bf16 value, ties to even, written out with numpy
    (8 significant bits: spacing 2^(e-8) for |x| in [2^(e-1), 2^e); np.round
    rounds halves to even).  Finite values inside bf16's normal range only."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(1.0, e - 8)
    return np.round(x / q) * q


# ----------------------------------------------------------------- geometry / cost

def test_geometry_matches_pages():
    """[NeoX] "Qwen3-0.6B example", "Current GPT-NeoX limitation"; [T07] §2; [Knob] §"Where the invariance breaks"."""
    for name, hidden, heads, kvh, hd, *want in golden_rows("geometry.txt"):
        hidden, heads = int(hidden), int(heads)
        kvh = int(kvh) if kvh != "-" else heads
        d = oracle.effective_head_dim(hidden, heads, int(hd) or None)
        w = oracle.widths(hidden, heads, kvh, d)
        got = [w["query_hidden"], w["kv_hidden"], w["qkv_out"], w["o_in"], w["o_out"]]
        for g, e in zip(got, want):
            if e != "-":
                assert g == int(e), (name, got, want)


def test_derived_head_dim_quotients():
    """[NeoX] opening: hidden/heads is 64, 80, 80 while the configs set 128."""
    for name, hidden, heads, explicit, quotient in golden_rows("quotients.txt"):
        assert oracle.effective_head_dim(int(hidden), int(heads)) == int(quotient)
        assert oracle.effective_head_dim(int(hidden), int(heads), int(explicit)) == int(explicit)
    # divisibility only matters when deriving ([NeoX] "Proposed configuration behavior")
    assert oracle.effective_head_dim(1000, 3) == -1
    assert oracle.effective_head_dim(1000, 3, 128) == 128


def test_capacity_knob_counts():
    """[Knob]: 4*d_model^2 weights for every h, pinned-128 counts, 2*n*d_model MACs."""
    for kind, dm, h, hd, n, val in golden_rows("capacity_knob_counts.txt"):
        dm, h, hd, val = int(dm), int(h), int(hd), int(val)
        if kind == "params":
            assert oracle.attn_param_count(dm, h, h, hd) == val
        elif kind == "proj_macs":
            assert oracle.proj_macs_per_token(dm, h, h, hd) == val
        else:
            assert oracle.score_value_macs_per_token(int(n), h, hd) == val


# ----------------------------------------------------------------- projection

def test_linear_orientation_is_x_times_w_transpose():
    """W is stored [out, in] and y = x @ W^T ([NeoX] "Checkpoint conversion";
    [T07] §4 step 1).  Unit rows of x pick out columns of W^T, i.e. rows of W."""
    rng = np.random.default_rng(0)
    K, N = 5, 3
    W = bf16(rng.integers(-8, 8, size=(N, K)))
    x = bf16(np.eye(K))
    y = oracle.linear(x, W, threads=T)
    assert y.shape == (K, N)
    np.testing.assert_array_equal(y, f64(W).numpy().T)


# ----------------------------------------------------------------- QK-norm

def test_rmsnorm_closed_forms():
    """Reading R3: v*w/sqrt(mean(v^2)+eps) over head_dim ([T07] §3)."""
    ones = bf16([1, 1, 1, 1])
    out = oracle.rmsnorm_rows(np.array([[3.0, 4.0, 0.0, 0.0]]), ones, 0.0)
    np.testing.assert_allclose(out, [[1.2, 1.6, 0.0, 0.0]], rtol=0, atol=1e-15)
    w = bf16([2.0, 0.5, 1.0, 1.0])
    out = oracle.rmsnorm_rows(np.array([[3.0, 4.0, 0.0, 0.0]]), w, 0.0)
    np.testing.assert_allclose(out, [[2.4, 0.8, 0.0, 0.0]], rtol=0, atol=1e-15)
    # eps sits inside the square root: mean(1)=1, eps=3 -> 1/2
    out = oracle.rmsnorm_rows(np.array([[1.0, 1.0, 1.0, 1.0]]), ones, 3.0)
    np.testing.assert_allclose(out, [[0.5] * 4], rtol=0, atol=1e-15)


def test_rmsnorm_invariant_and_library():
    """With unit weights the normed row has rms sqrt(ms/(ms+eps)); and the
    step equals torch.nn.functional.rms_norm evaluated in float64."""
    rng = np.random.default_rng(1)
    rows = rng.standard_normal((7, 128)) * 3.0
    eps = 1e-2
    out = oracle.rmsnorm_rows(rows, bf16(np.ones(128)), eps)
    ms = (rows ** 2).mean(1)
    np.testing.assert_allclose(np.sqrt((out ** 2).mean(1)), np.sqrt(ms / (ms + eps)), rtol=1e-13)
    w = bf16(1.0 + 0.1 * rng.standard_normal(128))
    ref = F.rms_norm(torch.from_numpy(rows), (128,), weight=f64(w), eps=eps).numpy()
    np.testing.assert_allclose(oracle.rmsnorm_rows(rows, w, eps), ref, rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------- RoPE

def test_rope_closed_forms():
    """Reading R4: pair (i, i+d/2), angle pos*theta^(-2i/d) ([T07] §4 RoPE)."""
    # d=2: one pair, frequency 1: (1,0) at position p -> (cos p, sin p)
    for p in (0.0, 1.0, 2.5, 100.0):
        out = oracle.rope_rows(np.array([[1.0, 0.0]]), [p], 10000.0)
        np.testing.assert_allclose(out, [[math.cos(p), math.sin(p)]], atol=1e-14)
    # d=4, theta=100: frequencies (1, 0.1).  e_1 at position 10 turns by 1 rad in
    # the (1,3) plane; e_0 turns by 10 rad in the (0,2) plane.
    out = oracle.rope_rows(np.array([[0.0, 1.0, 0.0, 0.0], [1.0, 0.0, 0.0, 0.0]]), [10.0, 10.0], 100.0)
    np.testing.assert_allclose(out[0], [0.0, math.cos(1.0), 0.0, math.sin(1.0)], atol=1e-14)
    np.testing.assert_allclose(out[1], [math.cos(10.0), 0.0, math.sin(10.0), 0.0], atol=1e-14)


def test_rope_invariants():
    """Identity at position 0, norm preserving, and <R_m q, R_n k> depends only on m-n."""
    rng = np.random.default_rng(2)
    d = 128
    v = rng.standard_normal((3, d))
    np.testing.assert_allclose(oracle.rope_rows(v, [0.0] * 3, 1e6), v, atol=0)
    r = oracle.rope_rows(v, [5.0, 77.0, 16383.0], 1e6)
    np.testing.assert_allclose(np.linalg.norm(r, axis=1), np.linalg.norm(v, axis=1), rtol=1e-13)
    q, k = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    dots = []
    for shift in (0.0, 13.0, 4000.0):
        rq = oracle.rope_rows(q, [20.0 + shift], 1e4)
        rk = oracle.rope_rows(k, [7.0 + shift], 1e4)
        dots.append(float((rq @ rk.T).item()))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


def test_rope_equals_complex_rotation():
    """Rotate-half RoPE is multiplication of z_i = v_i + i*v_{i+d/2} by
    exp(i*pos*theta^(-2i/d)), evaluated with torch complex128."""
    rng = np.random.default_rng(3)
    d, theta = 64, 1e4
    v = rng.standard_normal((5, d))
    pos = np.array([0.0, 1.0, 9.0, 300.0, 8192.0])
    out = oracle.rope_rows(v, pos, theta)
    half = d // 2
    z = torch.complex(torch.from_numpy(v[:, :half]), torch.from_numpy(v[:, half:]))
    freq = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.from_numpy(pos)[:, None] * freq[None, :]
    zr = z * torch.polar(torch.ones_like(ang), ang)
    ref = torch.cat([zr.real, zr.imag], dim=1).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- attention

def _att(Q, K, V, causal=True, sel=None):
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    return oracle.attention_stage(Q, K, V, B, S, Hq, Hkv, d, causal=causal, sel=sel, threads=T)


def test_attention_two_keys_closed_form():
    """Scale head_dim^-0.5 ([NeoX] "Scaling and RoPE"; [T07] §4).  d=4, query
    (2,0,0,0), keys 0 and (1,0,0,0): scores 0 and 1, so row 1 weights are
    1/(1+e) and e/(1+e); row 0 sees only key 0 (causal, diagonal included)."""
    Q = bf16(np.zeros((1, 1, 2, 4))); Q[0, 0, 1, 0] = 2.0
    K = bf16(np.zeros((1, 1, 2, 4))); K[0, 0, 1, 0] = 1.0
    V = bf16(np.zeros((1, 1, 2, 4)))
    V[0, 0, 0] = bf16([4.0, 0.0, 0.0, 8.0]); V[0, 0, 1] = bf16([0.0, 4.0, 0.0, 0.0])
    out = _att(Q, K, V)
    e = math.e
    np.testing.assert_allclose(out[0], [4.0, 0.0, 0.0, 8.0], atol=1e-15)
    np.testing.assert_allclose(out[1], [4 / (1 + e), 4 * e / (1 + e), 0.0, 8 / (1 + e)], rtol=1e-14)
    # without the mask row 0 sees both keys with score 0: the plain mean
    out = _att(Q, K, V, causal=False)
    np.testing.assert_allclose(out[0], [2.0, 2.0, 0.0, 4.0], atol=1e-15)


def test_attention_equal_keys_gives_prefix_mean():
    """All keys equal: softmax is uniform over the visible prefix, so row t is
    the mean of V[0..t]; row 0 is V[0] exactly."""
    rng = np.random.default_rng(4)
    S, d = 37, 8
    Q = bf16(rng.standard_normal((1, 1, S, d)))
    K = bf16(np.tile(rng.standard_normal((1, 1, 1, d)), (1, 1, S, 1)))
    V = bf16(rng.standard_normal((1, 1, S, d)))
    out = _att(Q, K, V)
    v = f64(V)[0, 0].numpy()
    ref = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(out[0], v[0])


def test_attention_group_map_markers():
    """Reading R2: query head j reads KV head j // (Hq/Hkv) ([NeoX] "Qwen3-0.6B
    example": each KV head serves 2 query heads; [Part]: preserve the mapping
    from global query heads to their KV group).  Each KV head's values are a
    distinct constant marker, so each query head must return its group's marker."""
    rng = np.random.default_rng(5)
    B, S, Hq, Hkv, d = 2, 9, 8, 2, 4
    markers = np.arange(1, B * Hkv * d + 1, dtype=np.float32).reshape(B, Hkv, 1, d)
    V = bf16(np.tile(markers, (1, 1, S, 1)))
    Q = bf16(rng.standard_normal((B, Hq, S, d)))
    K = bf16(rng.standard_normal((B, Hkv, S, d)))
    out = _att(Q, K, V).reshape(B, S, Hq, d)
    for j in range(Hq):
        for b in range(B):
            np.testing.assert_allclose(out[b, :, j], np.broadcast_to(markers[b, j // 4, 0], (S, d)),
                                       rtol=1e-14)


def test_attention_equals_library_sdpa():
    """Special case that reduces to a library routine: the attention step equals
    torch's scaled_dot_product_attention in float64 with each KV head repeated
    for its contiguous group, causal and non-causal, with a ragged length."""
    rng = np.random.default_rng(6)
    B, S, Hq, Hkv, d = 2, 45, 6, 2, 16
    Q = bf16(rng.standard_normal((B, Hq, S, d)) * 2)
    K = bf16(rng.standard_normal((B, Hkv, S, d)) * 2)
    V = bf16(rng.standard_normal((B, Hkv, S, d)))
    G = Hq // Hkv
    for causal in (True, False):
        ref = F.scaled_dot_product_attention(f64(Q), f64(K).repeat_interleave(G, 1),
                                             f64(V).repeat_interleave(G, 1), is_causal=causal)
        ref = ref.transpose(1, 2).reshape(B * S, Hq * d).numpy()
        np.testing.assert_allclose(_att(Q, K, V, causal=causal), ref, rtol=1e-11, atol=1e-12)
    # the row-sampled path returns exactly the selected rows
    sel = [0, 3, 44, 45, 89]
    np.testing.assert_array_equal(_att(Q, K, V, sel=sel), _att(Q, K, V)[sel])


def test_f16_widening_matches_numpy():
    """The oracle's binary16 decoder agrees with numpy's float16 on all 65536
    bit patterns (normals, subnormals, zeros, infinities, NaN)."""
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_attention_f16_inputs_equal_library_sdpa():
    """The attention step on binary16 Q/K/V equals torch's SDPA on the same
    values widened to float64."""
    rng = np.random.default_rng(8)
    B, S, Hq, Hkv, d = 1, 70, 4, 2, 32
    Q = torch.from_numpy(rng.standard_normal((B, Hq, S, d)) * 2).half()
    K = torch.from_numpy(rng.standard_normal((B, Hkv, S, d)) * 2).half()
    V = torch.from_numpy(rng.standard_normal((B, Hkv, S, d))).half()
    ref = F.scaled_dot_product_attention(Q.double(), K.double().repeat_interleave(2, 1),
                                         V.double().repeat_interleave(2, 1), is_causal=True)
    ref = ref.transpose(1, 2).reshape(B * S, Hq * d).numpy()
    np.testing.assert_allclose(_att(Q, K, V), ref, rtol=1e-11, atol=1e-12)


def test_attention_no_future_leak():
    """[Part]: a causal test with a nontrivial length.  A huge value planted in V
    at position 50 must leave rows < 50 untouched and move rows >= 50."""
    rng = np.random.default_rng(7)
    S, d = 130, 8
    Q = bf16(rng.standard_normal((1, 2, S, d)))
    K = bf16(rng.standard_normal((1, 1, S, d)))
    V = bf16(rng.standard_normal((1, 1, S, d)))
    base = _att(Q, K, V)
    V2 = V.clone(); V2[0, 0, 50] = 1e4
    spiked = _att(Q, K, V2)
    np.testing.assert_array_equal(spiked[:50], base[:50])
    assert np.all(np.abs(spiked[50:] - base[50:]).max(axis=1) > 1e-3)


# ----------------------------------------------------------------- whole layer

def _tiny(qk_norm=True, **kw):
    cfg = LayerConfig("tiny", B=2, S=19, hidden=24, Hq=4, Hkv=2, head_dim=8, qk_norm=qk_norm,
                      rope_theta=1e4, eps=1e-6)
    return cfg.with_(**kw) if kw else cfg


def _fwd(cfg, t, **kw):
    return oracle.forward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta,
                          cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                          causal=cfg.causal, threads=T, **kw)


def test_forward_equals_library_composition():
    """The whole layer ([T07] §4 steps 1-7, residual as in [NeoX] "Qwen3-0.6B
    example") equals a float64 composition of torch library routines:
    F.linear, F.rms_norm, complex-multiplication RoPE, scaled_dot_product_attention.
    The last case has five query heads per KV head ([Part]: each KV head serves
    Hq/Hkv contiguous query heads, a group size that is no power of two)."""
    for qk, Hq, Hkv in ((True, 4, 2), (False, 4, 2), (True, 10, 2)):
        cfg = _tiny(qk_norm=qk, Hq=Hq, Hkv=Hkv)
        t = make_layer_inputs(cfg, seed=11, w_std=0.3)
        B, S, h, Hq, Hkv, d = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
        x, W, Wo = f64(t["x"]), f64(t["Wqkv"]), f64(t["Wo"])
        q = F.linear(x, W[:Hq * d]).view(B, S, Hq, d)
        k = F.linear(x, W[Hq * d:(Hq + Hkv) * d]).view(B, S, Hkv, d)
        v = F.linear(x, W[(Hq + Hkv) * d:]).view(B, S, Hkv, d)
        if qk:
            q = F.rms_norm(q, (d,), weight=f64(t["q_norm_w"]), eps=cfg.eps)
            k = F.rms_norm(k, (d,), weight=f64(t["k_norm_w"]), eps=cfg.eps)

        def rope(a):
            half = d // 2
            z = torch.complex(a[..., :half], a[..., half:])
            ang = torch.arange(S, dtype=torch.float64)[:, None] * \
                cfg.rope_theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
            z = z * torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
            return torch.cat([z.real, z.imag], -1)

        q, k = rope(q).transpose(1, 2), rope(k).transpose(1, 2)
        v = v.transpose(1, 2)
        a = F.scaled_dot_product_attention(q, k.repeat_interleave(Hq // Hkv, 1),
                                           v.repeat_interleave(Hq // Hkv, 1), is_causal=True)
        a = a.transpose(1, 2).reshape(B, S, Hq * d)
        ref = (x + F.linear(a, Wo)).reshape(B * S, h).numpy()
        got = _fwd(cfg, t, want_stages=True)
        np.testing.assert_allclose(got["out"], ref, rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(got["attn"], a.reshape(B * S, -1).numpy(), rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(got["k"], k.numpy(), rtol=1e-11, atol=1e-11)


def test_forward_stages_agree_with_stage_functions():
    """oracle.forward and the three stage functions compute the same layer, and
    the row-sampled forward returns exactly the selected rows."""
    cfg = _tiny()
    t = make_layer_inputs(cfg, seed=12, w_std=0.3)
    full = _fwd(cfg, t, want_stages=True)
    q, k, v = oracle.qkv_stage(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta,
                               cfg.eps, cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                               threads=T)
    np.testing.assert_allclose(full["k"], k, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(full["q"], q.transpose(0, 2, 1, 3).reshape(-1, cfg.Hq, cfg.head_dim),
                               rtol=1e-13, atol=1e-14)
    sel = [0, 5, 18, 19, 37]
    part = _fwd(cfg, t, sel=sel)
    np.testing.assert_allclose(part, full["out"][sel], rtol=0, atol=0)


def test_forward_head_sum_decomposition():
    """[Knob] "Why the cost does not move": the layer is the sum over heads of
    head_i @ W_O_i, so zeroing all of W_O but head j's slice keeps exactly
    head j's term, and the terms add up to the full output minus x."""
    cfg = _tiny()
    t = make_layer_inputs(cfg, seed=13, w_std=0.3)
    d = cfg.head_dim
    full = _fwd(cfg, t) - f64(t["x"]).reshape(-1, cfg.hidden).numpy()
    total = np.zeros_like(full)
    for j in range(cfg.Hq):
        t2 = dict(t)
        wo = torch.zeros_like(t["Wo"]); wo[:, j * d:(j + 1) * d] = t["Wo"][:, j * d:(j + 1) * d]
        t2["Wo"] = wo
        term = _fwd(cfg, t2) - f64(t["x"]).reshape(-1, cfg.hidden).numpy()
        assert np.abs(term).max() > 1e-3
        total += term
    np.testing.assert_allclose(total, full, rtol=1e-11, atol=1e-12)
    # Wo = 0 leaves the residual alone
    t3 = dict(t); t3["Wo"] = torch.zeros_like(t["Wo"])
    np.testing.assert_array_equal(_fwd(cfg, t3), f64(t["x"]).reshape(-1, cfg.hidden).numpy())


def test_forward_permutation_tests():
    """[Part]: distinguishable heads so a permutation cannot hide.  Permuting the
    query heads inside a KV group (their Wqkv rows and the matching Wo columns)
    leaves the output unchanged; permuting only the Q rows permutes attn by head;
    swapping two KV groups together with their query heads changes nothing."""
    cfg = _tiny()
    t = make_layer_inputs(cfg, seed=14, w_std=0.3)
    d, Hq, Hkv = cfg.head_dim, cfg.Hq, cfg.Hkv
    base = _fwd(cfg, t, want_stages=True)

    def permuted(qperm, gperm):
        rows = [np.arange(qperm[j] * d, qperm[j] * d + d) for j in range(Hq)]
        rows += [Hq * d + np.arange(gperm[g] * d, gperm[g] * d + d) for g in range(Hkv)]
        rows += [(Hq + Hkv) * d + np.arange(gperm[g] * d, gperm[g] * d + d) for g in range(Hkv)]
        W = t["Wqkv"][torch.from_numpy(np.concatenate(rows))]
        cols = np.concatenate([np.arange(qperm[j] * d, qperm[j] * d + d) for j in range(Hq)])
        Wo = t["Wo"][:, torch.from_numpy(cols)]
        return W, Wo

    # within-group swap of heads 0 and 1 (both in group 0)
    W, Wo = permuted([1, 0, 2, 3], [0, 1])
    t2 = dict(t, Wqkv=W, Wo=Wo)
    got = _fwd(cfg, t2, want_stages=True)
    np.testing.assert_allclose(got["out"], base["out"], rtol=1e-12, atol=1e-13)
    a = got["attn"].reshape(-1, Hq, d)
    np.testing.assert_allclose(a[:, [1, 0, 2, 3]], base["attn"].reshape(-1, Hq, d), rtol=1e-12, atol=1e-13)
    # swap the two KV groups and carry their query heads along
    W, Wo = permuted([2, 3, 0, 1], [1, 0])
    got = _fwd(cfg, dict(t, Wqkv=W, Wo=Wo))
    np.testing.assert_allclose(got, base["out"], rtol=1e-12, atol=1e-13)
    # a cross-group swap of query heads alone is NOT a symmetry: it must change attn
    W, _ = permuted([2, 1, 0, 3], [0, 1])
    got = _fwd(cfg, dict(t, Wqkv=W), want_stages=True)
    a = got["attn"].reshape(-1, Hq, d)
    assert np.abs(a[:, 0] - base["attn"].reshape(-1, Hq, d)[:, 2]).max() > 1e-3


def test_forward_value_only_weights():
    """Reading R1 (fused rows Q, then K, then V): with the Q and K blocks zero
    every score is 0, the softmax is uniform over the prefix, and attn is the
    prefix mean of V = x @ W_v^T, whatever RoPE and QK-norm do to zeros."""
    cfg = _tiny(qk_norm=False)
    t = make_layer_inputs(cfg, seed=15, w_std=0.3)
    d, Hq, Hkv = cfg.head_dim, cfg.Hq, cfg.Hkv
    W = t["Wqkv"].clone(); W[:(Hq + Hkv) * d] = 0
    got = _fwd(cfg, dict(t, Wqkv=W), want_stages=True)
    v = (f64(t["x"]) @ f64(W[(Hq + Hkv) * d:]).T).numpy().reshape(cfg.B, cfg.S, Hkv, d)
    pm = np.cumsum(v, axis=1) / np.arange(1, cfg.S + 1)[None, :, None, None]
    ref = np.repeat(pm, Hq // Hkv, axis=2).reshape(cfg.B * cfg.S, Hq * d)
    np.testing.assert_allclose(got["attn"], ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------- decode

def test_round_bf16_is_nearest_even():
    """R21: a new key or value enters a bf16 cache as the nearest bf16 value,
    ties to even.  Against torch's binary32 -> bf16 conversion on values that
    binary32 holds exactly, the numpy restatement on arbitrary doubles, and
    closed forms: halfway cases go to the even neighbour, a double just above
    a halfway point rounds up (directly, not through binary32, which would make
    it a tie), bf16 subnormals keep the 2^-133 spacing, and a value past the
    largest finite bf16 by half a step or more becomes infinite."""
    rng = np.random.default_rng(41)
    f32 = (rng.standard_normal(4096) * np.exp2(rng.integers(-30, 30, 4096))).astype(np.float32).astype(np.float64)
    lib = torch.from_numpy(f32).float().to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(f32), lib)
    x = rng.standard_normal(4096) * 3.0
    np.testing.assert_array_equal(oracle.round_bf16(x), _bf16_rne(x))
    one = 1.0
    cases = {
        one + 2.0 ** -8: one,                             # halfway between 1 and 1 + 2^-7: even is 1
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,             # halfway, odd below: up to 1 + 2^-6
        one + 2.0 ** -8 + 2.0 ** -40: one + 2.0 ** -7,    # just above halfway (not a binary32 value)
        -(one + 2.0 ** -8 + 2.0 ** -40): -(one + 2.0 ** -7),
        3.0 * 2.0 ** -135: 2.0 ** -133,                   # subnormal range: 0.75 of the 2^-133 spacing rounds up
        2.0 ** -135: 0.0,                                  # and 0.25 of it rounds down to zero
        0.0: 0.0,
        (2 - 2.0 ** -7) * 2.0 ** 127: (2 - 2.0 ** -7) * 2.0 ** 127,
        (2 - 2.0 ** -8) * 2.0 ** 127: math.inf,           # halfway to 2^128: ties to even overflow
    }
    got = oracle.round_bf16(np.array(list(cases)))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))


def test_decode_matches_prefill_last_token():
    """[T07] §4 step 5 (the cache returns the whole history) and the RoPE
    offset: decoding token S-1 over a cache holding the prefill's keys and
    values of tokens 0..S-2 reproduces the prefill's last row.  The cached
    entries are bf16-rounded, so agreement is to bf16 accuracy; a wrong
    position or a dropped new key misses by far more."""
    cfg = _tiny(S=23, B=3)
    t = make_layer_inputs(cfg, seed=16, w_std=0.3)
    B, S, d, Hq, Hkv = cfg.B, cfg.S, cfg.head_dim, cfg.Hq, cfg.Hkv
    pre = _fwd(cfg, t, want_stages=True)
    Lmax = S + 5
    kc = torch.zeros((B, Hkv, Lmax, d), dtype=torch.bfloat16); vc = torch.zeros_like(kc)
    kc[:, :, :S - 1] = torch.from_numpy(pre["k"][:, :, :S - 1]).to(torch.bfloat16)
    vc[:, :, :S - 1] = torch.from_numpy(pre["v"][:, :, :S - 1]).to(torch.bfloat16)
    dec = oracle.decode(t["x"][:, S - 1], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"],
                        cfg.rope_theta, cfg.eps, B, cfg.hidden, Hq, Hkv, d, kc, vc,
                        [S - 1] * B, Lmax, threads=T)
    last = pre["out"].reshape(B, S, -1)[:, S - 1]
    np.testing.assert_allclose(dec["out"], last, rtol=0, atol=2e-2 * np.abs(last).max())
    # the new key as the bf16 cache stores it (R21)
    np.testing.assert_allclose(dec["k"], _bf16_rne(pre["k"][:, :, S - 1]), rtol=1e-12, atol=1e-13)
    # a decode at the wrong position (S instead of S-1) must disagree clearly
    wrong = oracle.decode(t["x"][:, S - 1], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"],
                          cfg.rope_theta, cfg.eps, B, cfg.hidden, Hq, Hkv, d, kc, vc,
                          [S] * B, Lmax, threads=T)
    assert np.abs(wrong["k"] - pre["k"][:, :, S - 1]).max() > 1e-2


def test_decode_attention_stage_matches_prefill_rows():
    """Decode attention of the new token over keys [0, L) equals the prefill
    attention row L-1 computed from the same bf16 Q/K/V."""
    rng = np.random.default_rng(17)
    B, S, Hq, Hkv, d = 2, 31, 4, 2, 16
    Q = bf16(rng.standard_normal((B, Hq, S, d)))
    K = bf16(rng.standard_normal((B, Hkv, S, d)))
    V = bf16(rng.standard_normal((B, Hkv, S, d)))
    lens = [S, 17]
    q = torch.stack([Q[b, :, lens[b] - 1] for b in range(B)])
    got = oracle.decode_attention_stage(q, K, V, lens, B, Hq, Hkv, d, S, threads=T)
    full = _att(Q, K, V).reshape(B, S, -1)
    for b in range(B):
        np.testing.assert_allclose(got[b], full[b, lens[b] - 1], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 2), (32, 2)])
def test_decode_attention_f16_query_equals_library_sdpa(Hq, Hkv):
    """Decode attention with a binary16 query over bf16 caches equals torch's
    SDPA (float64) of the widened values over each sequence's prefix, at groups
    of four, three and sixteen query heads per KV head."""
    rng = np.random.default_rng(18)
    B, d, Lmax = 3, 32, 40
    q = torch.from_numpy(rng.standard_normal((B, Hq, d)) * 1.5).half()
    kc = bf16(rng.standard_normal((B, Hkv, Lmax, d)))
    vc = bf16(rng.standard_normal((B, Hkv, Lmax, d)))
    lens = [40, 1, 17]
    got = oracle.decode_attention_stage(q, kc, vc, lens, B, Hq, Hkv, d, Lmax, threads=T)
    for b in range(B):
        L = lens[b]
        k = f64(kc[b, :, :L]).repeat_interleave(Hq // Hkv, 0)
        v = f64(vc[b, :, :L]).repeat_interleave(Hq // Hkv, 0)
        ref = F.scaled_dot_product_attention(q[b].double()[:, None], k, v)[:, 0].reshape(-1).numpy()
        np.testing.assert_allclose(got[b], ref, rtol=1e-11, atol=1e-12)


def _empty_cache(B, Hkv, Lmax, d):
    return torch.zeros((B, Hkv, Lmax, d), dtype=torch.bfloat16), torch.zeros((B, Hkv, Lmax, d), dtype=torch.bfloat16)


def test_prefill_cached_at_offset_zero_is_the_plain_prefill():
    """With nothing cached (p0 = 0) the cached prefill is the plain layer whose
    keys and values pass through the bf16 cache (R21: attention reads what the
    cache holds): the float64 torch composition with K and V rounded to bf16
    after RoPE.  Without the rounding the two differ by far more than the
    composition's own error."""
    cfg = _tiny(S=21)
    t = make_layer_inputs(cfg, seed=19, w_std=0.3)
    kc, vc = _empty_cache(cfg.B, cfg.Hkv, 32, cfg.head_dim)
    got = oracle.prefill_cached(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, [0] * cfg.B, 32,
                                threads=T)
    keep = {}
    _, out = _torch_layer(cfg, t, keep=keep, kv_round=lambda a: torch.from_numpy(_bf16_rne(a.detach().numpy())))
    B, S, h = cfg.B, cfg.S, cfg.hidden
    np.testing.assert_allclose(got["out"], out.detach().reshape(B * S, h).numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(got["attn"], keep["attn"].detach().reshape(B * S, -1).numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(got["k"], keep["k"].detach().numpy(), rtol=0, atol=0)
    np.testing.assert_allclose(got["v"], keep["v"].detach().numpy(), rtol=0, atol=0)
    plain = _fwd(cfg, t, want_stages=True)
    assert np.abs(got["attn"] - plain["attn"]).max() > 1e-5


def test_prefill_cached_single_token_is_the_decode_step():
    """One new token per sequence is exactly the decode step."""
    cfg = _tiny(S=1, B=3)
    t = make_layer_inputs(cfg, seed=20, w_std=0.3)
    rng = np.random.default_rng(20)
    Lmax = 40
    kc = bf16(rng.standard_normal((cfg.B, cfg.Hkv, Lmax, cfg.head_dim)))
    vc = bf16(rng.standard_normal((cfg.B, cfg.Hkv, Lmax, cfg.head_dim)))
    p0 = [5, 0, 39]
    got = oracle.prefill_cached(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                cfg.B, 1, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, p0, Lmax, threads=T)
    dec = oracle.decode(t["x"][:, 0], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                        cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, kc, vc, p0, Lmax, threads=T)
    np.testing.assert_allclose(got["out"], dec["out"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(got["k"][:, :, 0], dec["k"], rtol=1e-13, atol=1e-13)


def test_prefill_in_two_chunks_matches_one_prefill():
    """Chunked prefill: the first S1 tokens prefilled, their keys/values cached
    (bf16), then the next S2 tokens at offset S1 reproduce the one-shot
    prefill's last S2 rows to bf16 accuracy ([Part]: global positions)."""
    cfg = _tiny(S=30, B=2)
    t = make_layer_inputs(cfg, seed=21, w_std=0.3)
    S1, S2, Lmax = 17, 13, 32
    full = _fwd(cfg, t, want_stages=True)
    kc, vc = _empty_cache(cfg.B, cfg.Hkv, Lmax, cfg.head_dim)
    kc[:, :, :S1] = torch.from_numpy(full["k"][:, :, :S1]).to(torch.bfloat16)
    vc[:, :, :S1] = torch.from_numpy(full["v"][:, :, :S1]).to(torch.bfloat16)
    got = oracle.prefill_cached(t["x"][:, S1:].contiguous(), t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"],
                                cfg.rope_theta, cfg.eps, cfg.B, S2, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                                kc, vc, [S1] * cfg.B, Lmax, threads=T)
    ref = full["out"].reshape(cfg.B, cfg.S, -1)[:, S1:].reshape(-1, cfg.hidden)
    np.testing.assert_allclose(got["out"], ref, rtol=0, atol=2e-2 * np.abs(ref).max())
    np.testing.assert_allclose(got["k"], _bf16_rne(full["k"][:, :, S1:]), rtol=1e-12, atol=1e-13)
    # the wrong offset is caught
    bad = oracle.prefill_cached(t["x"][:, S1:].contiguous(), t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"],
                                cfg.rope_theta, cfg.eps, cfg.B, S2, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim,
                                kc, vc, [S1 - 1] * cfg.B, Lmax, threads=T)
    assert np.abs(bad["k"] - full["k"][:, :, S1:]).max() > 1e-2


def test_oracle_rejects_bad_arguments():
    with pytest.raises(RuntimeError):
        oracle.rope_rows(np.zeros((1, 3)), [0.0], 1e4)     # odd head_dim
    rng = np.random.default_rng(0)
    Q = bf16(rng.standard_normal((1, 3, 4, 8)))
    K = bf16(rng.standard_normal((1, 2, 4, 8)))
    with pytest.raises(RuntimeError):
        oracle.attention_stage(Q, K, K, 1, 4, 3, 2, 8)     # Hq % Hkv != 0


# ----------------------------------------------------------------- partial rotary (reading R16)

def _complex_rope(a, pos, theta, rd):
    """Rotate-half RoPE on the first rd features as complex multiplication of
    z_i = a_i + i*a_{i+rd/2} by exp(i*pos*theta^(-2i/rd)); the rest unchanged."""
    a = torch.as_tensor(a, dtype=torch.float64)
    if rd == 0:
        return a.clone()
    half = rd // 2
    z = torch.complex(a[..., :half], a[..., half:rd])
    ang = torch.as_tensor(pos, dtype=torch.float64)[..., None] * \
        theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / rd)
    z = z * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag, a[..., rd:]], dim=-1)


def test_partial_rope_equals_complex_rotation_of_leading_features():
    """[NeoX] "Scaling and RoPE": rotary_pct < 1 rotates only the leading
    features, with frequencies over the rotary width; rd = d is the full
    rotation and rd = 0 the identity."""
    rng = np.random.default_rng(31)
    d, theta = 64, 1e4
    v = rng.standard_normal((6, d))
    pos = np.array([0.0, 1.0, 7.0, 129.0, 4095.0, 8192.0])
    for rd in (0, 16, 32, 48, 64):
        out = oracle.rope_rows(v, pos, theta, rotary_dim=rd)
        ref = _complex_rope(v, pos, theta, rd).numpy()
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.rope_rows(v, pos, theta, rotary_dim=d), oracle.rope_rows(v, pos, theta),
                               rtol=0, atol=0)
    # a slip that uses d instead of rd for the frequencies is caught
    wrong = _complex_rope(v, pos, theta ** (16 / d), 16).numpy()  # theta^(-2i/d) = (theta^(rd/d))^(-2i/rd)
    assert np.abs(oracle.rope_rows(v, pos, theta, rotary_dim=16) - wrong).max() > 1e-3


def test_partial_rope_invariants():
    """The rotated part keeps its norm, the tail is untouched, and the score of
    two rotated vectors depends only on the position difference."""
    rng = np.random.default_rng(32)
    d, rd, theta = 32, 8, 1e6
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    a = oracle.rope_rows(np.stack([q] * 3), [0.0, 5.0, 1000.0], theta, rotary_dim=rd)
    np.testing.assert_allclose(np.linalg.norm(a[:, :rd], axis=1), np.linalg.norm(q[:rd]), rtol=1e-12)
    np.testing.assert_allclose(a[:, rd:], np.stack([q[rd:]] * 3), rtol=0, atol=0)
    np.testing.assert_allclose(a[0], q, rtol=0, atol=1e-15)
    dots = []
    for m, n in ((3, 1), (10, 8), (1002, 1000)):
        qm = oracle.rope_rows(q[None], [float(m)], theta, rotary_dim=rd)[0]
        kn = oracle.rope_rows(k[None], [float(n)], theta, rotary_dim=rd)[0]
        dots.append(qm @ kn)
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


def test_forward_partial_rotary_equals_library_composition():
    """The layer with rotary_dim = d/4 and d/2 equals the float64 torch
    composition (F.linear, F.rms_norm, complex RoPE on the leading features,
    SDPA); the cached prefill at offset 0 and the decode step of the last token
    agree with it."""
    for rd in (2, 4):
        cfg = _tiny()
        t = make_layer_inputs(cfg, seed=33, w_std=0.3)
        B, S, h, Hq, Hkv, d = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
        x, W, Wo = f64(t["x"]), f64(t["Wqkv"]), f64(t["Wo"])
        q = F.linear(x, W[:Hq * d]).view(B, S, Hq, d)
        k = F.linear(x, W[Hq * d:(Hq + Hkv) * d]).view(B, S, Hkv, d)
        v = F.linear(x, W[(Hq + Hkv) * d:]).view(B, S, Hkv, d)
        q = F.rms_norm(q, (d,), weight=f64(t["q_norm_w"]), eps=cfg.eps)
        k = F.rms_norm(k, (d,), weight=f64(t["k_norm_w"]), eps=cfg.eps)
        pos = torch.arange(S, dtype=torch.float64)[:, None]
        q = _complex_rope(q, pos, cfg.rope_theta, rd).transpose(1, 2)
        k = _complex_rope(k, pos, cfg.rope_theta, rd).transpose(1, 2)
        v = v.transpose(1, 2)
        a = F.scaled_dot_product_attention(q, k.repeat_interleave(Hq // Hkv, 1),
                                           v.repeat_interleave(Hq // Hkv, 1), is_causal=True)
        a = a.transpose(1, 2).reshape(B, S, Hq * d)
        ref = (x + F.linear(a, Wo)).reshape(B * S, h).numpy()
        got = _fwd(cfg, t, want_stages=True, rotary_dim=rd)
        np.testing.assert_allclose(got["out"], ref, rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(got["k"], k.numpy(), rtol=1e-11, atol=1e-11)
        qs, ks, vs = oracle.qkv_stage(t["x"], t["Wqkv"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                                      B, S, h, Hq, Hkv, d, threads=T, rotary_dim=rd)
        np.testing.assert_allclose(qs, q.numpy(), rtol=1e-11, atol=1e-11)
        kc, vc = _empty_cache(B, Hkv, 32, d)
        pc = oracle.prefill_cached(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta,
                                   cfg.eps, B, S, h, Hq, Hkv, d, kc, vc, [0] * B, 32, threads=T, rotary_dim=rd)
        # the cached prefill attends over K and V as the bf16 cache stores them (R21)
        kr, vr = torch.from_numpy(_bf16_rne(k.numpy())), torch.from_numpy(_bf16_rne(v.numpy()))
        ar = F.scaled_dot_product_attention(q, kr.repeat_interleave(Hq // Hkv, 1),
                                            vr.repeat_interleave(Hq // Hkv, 1), is_causal=True)
        ref_c = (x + F.linear(ar.transpose(1, 2).reshape(B, S, Hq * d), Wo)).reshape(B * S, h).numpy()
        np.testing.assert_allclose(pc["out"], ref_c, rtol=1e-11, atol=1e-11)
        kc[:, :, :S - 1] = torch.from_numpy(got["k"][:, :, :S - 1]).to(torch.bfloat16)
        vc[:, :, :S - 1] = torch.from_numpy(got["v"][:, :, :S - 1]).to(torch.bfloat16)
        dec = oracle.decode(t["x"][:, S - 1], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta,
                            cfg.eps, B, h, Hq, Hkv, d, kc, vc, [S - 1] * B, 32, threads=T, rotary_dim=rd)
        np.testing.assert_allclose(dec["k"], _bf16_rne(got["k"][:, :, S - 1]), rtol=1e-12, atol=1e-13)
        last = got["out"].reshape(B, S, -1)[:, S - 1]
        np.testing.assert_allclose(dec["out"], last, rtol=0, atol=2e-2 * np.abs(last).max())


@pytest.mark.parametrize("d,rd", [(80, 80), (80, 20), (96, 96), (96, 48)])
def test_forward_at_widths_80_96_equals_library_composition(d, rd):
    """At head widths that are not a power of two ([Knob] "Where the invariance
    breaks": 80 is Qwen3-4B's hidden/heads quotient, 96 the width it names) the
    layer still equals the float64 torch composition; the RoPE pairs are
    (i, i + rd/2), so a dropped or shifted pair at these offsets fails here."""
    cfg = _tiny(head_dim=d, S=7, hidden=32, Hq=2, Hkv=1)
    t = make_layer_inputs(cfg, seed=51 + d + rd, w_std=0.3)
    B, S, h, Hq, Hkv = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv
    x, W, Wo = f64(t["x"]), f64(t["Wqkv"]), f64(t["Wo"])
    q = F.linear(x, W[:Hq * d]).view(B, S, Hq, d)
    k = F.linear(x, W[Hq * d:(Hq + Hkv) * d]).view(B, S, Hkv, d)
    v = F.linear(x, W[(Hq + Hkv) * d:]).view(B, S, Hkv, d)
    q = F.rms_norm(q, (d,), weight=f64(t["q_norm_w"]), eps=cfg.eps)
    k = F.rms_norm(k, (d,), weight=f64(t["k_norm_w"]), eps=cfg.eps)
    pos = torch.arange(S, dtype=torch.float64)[:, None]
    q = _complex_rope(q, pos, cfg.rope_theta, rd).transpose(1, 2)
    k = _complex_rope(k, pos, cfg.rope_theta, rd).transpose(1, 2)
    v = v.transpose(1, 2)
    a = F.scaled_dot_product_attention(q, k.repeat_interleave(Hq // Hkv, 1),
                                       v.repeat_interleave(Hq // Hkv, 1), is_causal=True)
    a = a.transpose(1, 2).reshape(B, S, Hq * d)
    ref = (x + F.linear(a, Wo)).reshape(B * S, h).numpy()
    got = _fwd(cfg, t, want_stages=True, rotary_dim=rd)
    np.testing.assert_allclose(got["out"], ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(got["q"].reshape(B, S, Hq, d).transpose(0, 2, 1, 3), q.numpy(), rtol=1e-11,
                               atol=1e-11)
    np.testing.assert_allclose(got["k"], k.numpy(), rtol=1e-11, atol=1e-11)


def test_partial_rotary_rejects_bad_widths():
    v = np.zeros((1, 8))
    for rd in (-2, 3, 10):
        with pytest.raises(RuntimeError):
            oracle.rope_rows(v, [0.0], 1e4, rotary_dim=rd)


# ----------------------------------------------------------------- FP8 KV cache (reading R17)

def test_e4m3_decode_matches_library_on_every_code():
    """All 256 E4M3 codes widen to the values torch's float8_e4m3fn gives
    (NaN for S.1111.111, no infinities)."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.isnan(got).sum() == 2
    np.testing.assert_array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])


def test_e4m3_encode_matches_library_and_saturates():
    """In range, the nearest code with ties to even equals torch's conversion;
    beyond +-448 the code saturates to +-448 (closed forms)."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal(200000) * np.exp(rng.uniform(-14.0, 6.0, 200000))
    x = x[np.abs(x) < 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x), ref)
    # ties: 1 + 1/16 lies halfway between 1 and 1.125 -> even mantissa (1.0);
    # 1 + 3/16 -> 1.25; 2^-10 halfway between 0 and the smallest subnormal -> 0
    got = oracle.e4m3_decode(oracle.e4m3_encode([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, -1.0625]))
    np.testing.assert_array_equal(got, [1.0, 1.25, 0.0, 2.0 ** -8, -1.0])
    sat = oracle.e4m3_encode([448.0, 463.99, 464.0, 1e30, -1e30, float("inf")])
    np.testing.assert_array_equal(sat, [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E])
    assert oracle.e4m3_encode([float("nan")])[0] == 0x7F


def test_fp8_decode_attention_equals_bf16_path_on_exact_codes():
    """With power-of-two scales every dequantised entry is a bf16 value, so
    attention over the FP8 cache equals attention over the bf16 cache holding
    those values (two independent code paths of the oracle)."""
    rng = np.random.default_rng(42)
    B, Hq, Hkv, d, Lmax = 3, 8, 2, 32, 50
    ks, vs = 2.0 ** -5, 2.0 ** -3
    kc8 = rng.integers(0, 256, (B, Hkv, Lmax, d), dtype=np.uint8)
    vc8 = rng.integers(0, 256, (B, Hkv, Lmax, d), dtype=np.uint8)
    kc8[(kc8 & 0x7F) == 0x7F] = 0x10  # no NaN codes
    vc8[(vc8 & 0x7F) == 0x7F] = 0x10
    q = torch.from_numpy(rng.standard_normal((B, Hq, d))).half()
    lens = [50, 1, 23]
    got = oracle.decode_attention_stage_fp8(q, kc8, vc8, ks, vs, lens, B, Hq, Hkv, d, Lmax, threads=T)
    kb = bf16(oracle.e4m3_decode(kc8) * ks)
    vb = bf16(oracle.e4m3_decode(vc8) * vs)
    assert np.array_equal(f64(kb).numpy(), oracle.e4m3_decode(kc8) * ks)  # exact in bf16
    ref = oracle.decode_attention_stage(q, kb, vb, lens, B, Hq, Hkv, d, Lmax, threads=T)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_fp8_decode_step_equals_library_composition():
    """The FP8 decode step: the appended codes are the nearest codes of the new
    key / value over their scales, and the output is x + SDPA(q, cache with the
    new entries, all dequantised) @ Wo^T, evaluated with torch in float64."""
    cfg = _tiny(B=3)
    t = make_layer_inputs(cfg, seed=43, w_std=0.3)
    rng = np.random.default_rng(43)
    B, h, Hq, Hkv, d = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
    Lmax, ks, vs = 30, 0.05, 0.02
    kc8 = oracle.e4m3_encode(rng.standard_normal((B, Hkv, Lmax, d)) / ks)
    vc8 = oracle.e4m3_encode(rng.standard_normal((B, Hkv, Lmax, d)) / vs)
    cl = [0, 7, 29]
    x1 = t["x"][:, 0].contiguous()
    got = oracle.decode_fp8(x1, t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps, B, h,
                            Hq, Hkv, d, kc8, vc8, ks, vs, cl, Lmax, threads=T)
    np.testing.assert_array_equal(got["k_code"], oracle.e4m3_encode(got["k"] / ks))
    np.testing.assert_array_equal(got["v_code"], oracle.e4m3_encode(got["v"] / vs))
    # the bf16 decode computes the same q, k, v before its cache's bf16 rounding (R21)
    ref_bf = oracle.decode(x1, t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps, B, h,
                           Hq, Hkv, d, bf16(np.zeros((B, Hkv, Lmax, d))), bf16(np.zeros((B, Hkv, Lmax, d))), cl,
                           Lmax, threads=T)
    np.testing.assert_allclose(got["q"], ref_bf["q"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(_bf16_rne(got["k"]), ref_bf["k"], rtol=1e-13, atol=1e-14)
    kd = oracle.e4m3_decode(kc8) * ks
    vd = oracle.e4m3_decode(vc8) * vs
    for b in range(B):
        p = cl[b]
        k = np.concatenate([kd[b, :, :p], (oracle.e4m3_decode(got["k_code"][b]) * ks)[:, None]], axis=1)
        v = np.concatenate([vd[b, :, :p], (oracle.e4m3_decode(got["v_code"][b]) * vs)[:, None]], axis=1)
        k = torch.from_numpy(k).repeat_interleave(Hq // Hkv, 0)
        v = torch.from_numpy(v).repeat_interleave(Hq // Hkv, 0)
        qb = torch.from_numpy(got["q"][b])[:, None]
        a = F.scaled_dot_product_attention(qb, k, v)[:, 0].reshape(-1)
        np.testing.assert_allclose(got["attn"][b], a.numpy(), rtol=1e-11, atol=1e-12)
        o = f64(t["x"][b, 0]) + F.linear(a, f64(t["Wo"]))
        np.testing.assert_allclose(got["out"][b], o.numpy(), rtol=1e-11, atol=1e-11)


# ----------------------------------------------------------------- backward

def _torch_layer(cfg, t, causal=True, keep=None, kv_round=None, rd=None):
    """The layer as a float64 torch composition (F.linear, F.rms_norm, complex
    RoPE, SDPA); parameters are leaves with requires_grad.  keep (a dict)
    receives the attention's q, k, v and attn with retained gradients.
    kv_round (forward only): applied to K and V after RoPE.  rd: rotary width
    (default head_dim)."""
    B, S, h, Hq, Hkv, d = cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim
    leaves = {k: f64(v).requires_grad_(True) for k, v in t.items() if v is not None}
    x, W, Wo = leaves["x"], leaves["Wqkv"], leaves["Wo"]
    q = F.linear(x, W[:Hq * d]).view(B, S, Hq, d)
    k = F.linear(x, W[Hq * d:(Hq + Hkv) * d]).view(B, S, Hkv, d)
    v = F.linear(x, W[(Hq + Hkv) * d:]).view(B, S, Hkv, d)
    if "q_norm_w" in leaves:
        q = F.rms_norm(q, (d,), weight=leaves["q_norm_w"], eps=cfg.eps)
        k = F.rms_norm(k, (d,), weight=leaves["k_norm_w"], eps=cfg.eps)
    pos = torch.arange(S, dtype=torch.float64)[:, None]
    q = _complex_rope(q, pos, cfg.rope_theta, d if rd is None else rd).transpose(1, 2)
    k = _complex_rope(k, pos, cfg.rope_theta, d if rd is None else rd).transpose(1, 2)
    v = v.transpose(1, 2)
    if kv_round is not None:
        k, v = kv_round(k), kv_round(v)
    if keep is not None and kv_round is None:
        for name, tt in (("q", q), ("k", k), ("v", v)):
            tt.retain_grad()
            keep[name] = tt
    elif keep is not None:
        keep.update(q=q, k=k, v=v)
    a = F.scaled_dot_product_attention(q, k.repeat_interleave(Hq // Hkv, 1), v.repeat_interleave(Hq // Hkv, 1),
                                       is_causal=causal)
    a = a.transpose(1, 2).reshape(B, S, Hq * d)
    if keep is not None:
        if a.requires_grad:
            a.retain_grad()
        keep["attn"] = a
    return leaves, x + F.linear(a, Wo)


@pytest.mark.parametrize("qk,causal,Hq", [(True, True, 4), (False, True, 4), (True, False, 4), (True, True, 10)])
def test_backward_equals_library_autograd(qk, causal, Hq):
    """Every gradient of the layer (x, Wqkv, Wo, both norm weights, and the
    attention's inputs/outputs) equals torch's float64 autograd through the
    library composition; K/V gradients include the sum over a group's heads
    (two heads per group, and five in the last case)."""
    cfg = _tiny(qk_norm=qk, Hq=Hq)
    t = make_layer_inputs(cfg, seed=51, w_std=0.3)
    dout = bf16(np.random.default_rng(51).standard_normal((cfg.B * cfg.S, cfg.hidden)))
    keep = {}
    leaves, out = _torch_layer(cfg, t, causal, keep)
    (out.reshape(-1, cfg.hidden) * f64(dout)).sum().backward()
    got = oracle.backward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                          cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, dout, causal=causal,
                          want_stages=True, threads=T)
    tol = dict(rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(got["dx"], leaves["x"].grad.reshape(-1, cfg.hidden).numpy(), **tol)
    np.testing.assert_allclose(got["dWqkv"], leaves["Wqkv"].grad.numpy(), **tol)
    np.testing.assert_allclose(got["dWo"], leaves["Wo"].grad.numpy(), **tol)
    np.testing.assert_allclose(got["d_attn"], keep["attn"].grad.reshape(cfg.B * cfg.S, -1).numpy(), **tol)
    np.testing.assert_allclose(got["dq"], keep["q"].grad.numpy(), **tol)
    np.testing.assert_allclose(got["dk"], keep["k"].grad.numpy(), **tol)
    np.testing.assert_allclose(got["dv"], keep["v"].grad.numpy(), **tol)
    if qk:
        np.testing.assert_allclose(got["dq_norm_w"], leaves["q_norm_w"].grad.numpy(), **tol)
        np.testing.assert_allclose(got["dk_norm_w"], leaves["k_norm_w"].grad.numpy(), **tol)
    else:
        assert not got["dq_norm_w"].any() and not got["dk_norm_w"].any()


@pytest.mark.parametrize("rd", [4, 2, 0])
def test_backward_partial_rotary_equals_library_autograd(rd):
    """The backward with RoPE on the first rd features only (R16: [NeoX]
    "Scaling and RoPE", rotary_pct): every gradient equals float64 autograd
    through the composition rotating those features; the unrotated features'
    gradients pass the inverse rotation unchanged (rd = 0: no rotation)."""
    cfg = _tiny()
    t = make_layer_inputs(cfg, seed=53, w_std=0.3)
    dout = bf16(np.random.default_rng(53).standard_normal((cfg.B * cfg.S, cfg.hidden)))
    keep = {}
    leaves, out = _torch_layer(cfg, t, True, keep, rd=rd)
    (out.reshape(-1, cfg.hidden) * f64(dout)).sum().backward()
    got = oracle.backward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                          cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, dout, want_stages=True, threads=T,
                          rotary_dim=rd)
    tol = dict(rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(got["dx"], leaves["x"].grad.reshape(-1, cfg.hidden).numpy(), **tol)
    np.testing.assert_allclose(got["dWqkv"], leaves["Wqkv"].grad.numpy(), **tol)
    np.testing.assert_allclose(got["dq_norm_w"], leaves["q_norm_w"].grad.numpy(), **tol)
    np.testing.assert_allclose(got["dk_norm_w"], leaves["k_norm_w"].grad.numpy(), **tol)
    np.testing.assert_allclose(got["dk"], keep["k"].grad.numpy(), **tol)
    full = oracle.backward(t["x"], t["Wqkv"], t["Wo"], t["q_norm_w"], t["k_norm_w"], cfg.rope_theta, cfg.eps,
                           cfg.B, cfg.S, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.head_dim, dout, threads=T)
    assert np.abs(full["dx"] - got["dx"]).max() > 1e-6  # the rotary width matters


def test_attention_backward_stage_equals_library_autograd():
    """The attention backward alone (16-bit inputs widened exactly) equals
    torch float64 autograd of SDPA with repeated KV heads."""
    rng = np.random.default_rng(52)
    B, S, Hq, Hkv, d = 2, 23, 6, 2, 16
    Q = torch.from_numpy(rng.standard_normal((B, Hq, S, d))).half()
    K = torch.from_numpy(rng.standard_normal((B, Hkv, S, d))).half()
    V = torch.from_numpy(rng.standard_normal((B, Hkv, S, d))).half()
    dO = torch.from_numpy(rng.standard_normal((B, S, Hq * d))).half()
    for causal in (True, False):
        q, k, v = (a.double().requires_grad_(True) for a in (Q, K, V))
        a = F.scaled_dot_product_attention(q, k.repeat_interleave(Hq // Hkv, 1), v.repeat_interleave(Hq // Hkv, 1),
                                           is_causal=causal)
        (a.transpose(1, 2).reshape(B, S, -1) * dO.double()).sum().backward()
        dq, dk, dv = oracle.attention_backward(Q, K, V, dO, B, S, Hq, Hkv, d, causal=causal, threads=T)
        np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_backward_closed_forms():
    """A single key: the softmax is the constant 1, so dq = dk = 0 and dv = dO
    summed over the group's heads; with dO = 0 every gradient vanishes."""
    rng = np.random.default_rng(53)
    B, S, Hq, Hkv, d = 1, 1, 4, 2, 8
    Q = bf16(rng.standard_normal((B, Hq, S, d)))
    K = bf16(rng.standard_normal((B, Hkv, S, d)))
    V = bf16(rng.standard_normal((B, Hkv, S, d)))
    dO = bf16(rng.standard_normal((B, S, Hq * d)))
    dq, dk, dv = oracle.attention_backward(Q, K, V, dO, B, S, Hq, Hkv, d, threads=T)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    do = f64(dO).reshape(B, S, Hq, d).numpy()
    np.testing.assert_allclose(dv[0, :, 0], do[0, 0].reshape(Hkv, Hq // Hkv, d).sum(1), rtol=1e-14, atol=0)
    Z = bf16(np.zeros((1, 7, Hq * d)))
    dq, dk, dv = oracle.attention_backward(bf16(rng.standard_normal((1, Hq, 7, d))),
                                           bf16(rng.standard_normal((1, Hkv, 7, d))),
                                           bf16(rng.standard_normal((1, Hkv, 7, d))), Z, 1, 7, Hq, Hkv, d, threads=T)
    assert not dq.any() and not dk.any() and not dv.any()
