"""Python wrapper of the fp64 CPU oracle (``gqa_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product library never
imports, links or runs anything under ``oracle/``.

Inputs are bf16 torch tensors (or numpy uint16 bit patterns); the C code
widens them to double exactly.  Outputs are float64 numpy arrays.

Every function here has a pin in ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_long)
_i32p = ctypes.POINTER(ctypes.c_int)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_L = ctypes.c_long
_D = ctypes.c_double
_I = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP) next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    lib.oracle_effective_head_dim.restype = _L
    lib.oracle_effective_head_dim.argtypes = [_L, _L, _L]
    lib.oracle_widths.restype = None
    lib.oracle_widths.argtypes = [_L, _L, _L, _L, _i64p]
    for f in ("oracle_attn_param_count", "oracle_proj_macs_per_token"):
        getattr(lib, f).restype = ctypes.c_longlong
        getattr(lib, f).argtypes = [_L, _L, _L, _L]
    lib.oracle_score_value_macs_per_token.restype = ctypes.c_longlong
    lib.oracle_score_value_macs_per_token.argtypes = [_L, _L, _L]
    lib.oracle_rmsnorm_rows.restype = _I
    lib.oracle_rmsnorm_rows.argtypes = [_f64p, _L, _L, _u16p, _D, _f64p]
    lib.oracle_rope_rows.restype = _I
    lib.oracle_rope_rows.argtypes = [_f64p, _L, _L, _f64p, _D, _f64p]
    lib.oracle_linear.restype = _I
    lib.oracle_linear.argtypes = [_u16p, _u16p, _L, _L, _L, _f64p, _I]
    lib.oracle_qkv_stage.restype = _I
    lib.oracle_qkv_stage.argtypes = [_u16p, _u16p, _u16p, _u16p, _D, _D,
                                     _L, _L, _L, _L, _L, _L, _f64p, _f64p, _f64p, _I]
    lib.oracle_attention_stage.restype = _I
    lib.oracle_attention_stage.argtypes = [_u16p, _u16p, _u16p, _I, _L, _L, _L, _L, _L, _I,
                                           _i64p, _L, _f64p, _I]
    lib.oracle_round_bf16.restype = _I
    lib.oracle_round_bf16.argtypes = [_f64p, _L, _f64p]
    lib.oracle_f16_to_double.restype = None
    lib.oracle_f16_to_double.argtypes = [_u16p, _L, _f64p]
    lib.oracle_oproj_stage.restype = _I
    lib.oracle_oproj_stage.argtypes = [_u16p, _u16p, _u16p, _L, _L, _L, _i64p, _L, _f64p, _I]
    lib.oracle_forward.restype = _I
    lib.oracle_forward.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, _D, _D,
                                   _L, _L, _L, _L, _L, _L, _I, _i64p, _L,
                                   _f64p, _f64p, _f64p, _f64p, _f64p, _I]
    lib.oracle_decode_attention_stage.restype = _I
    lib.oracle_decode_attention_stage.argtypes = [_u16p, _I, _u16p, _u16p, _i32p,
                                                  _L, _L, _L, _L, _L, _f64p, _I]
    lib.oracle_prefill_cached.restype = _I
    lib.oracle_prefill_cached.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, _D, _D,
                                          _L, _L, _L, _L, _L, _L, _I, _u16p, _u16p, _i32p, _L,
                                          _f64p, _f64p, _f64p, _f64p, _I]
    lib.oracle_decode.restype = _I
    lib.oracle_decode.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, _D, _D,
                                  _L, _L, _L, _L, _L, _u16p, _u16p, _i32p, _L,
                                  _f64p, _f64p, _f64p, _f64p, _f64p, _I]
    _u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_e4m3_decode.restype = None
    lib.oracle_e4m3_decode.argtypes = [_u8p, _L, _f64p]
    lib.oracle_e4m3_encode.restype = None
    lib.oracle_e4m3_encode.argtypes = [_f64p, _L, _u8p]
    lib.oracle_decode_attention_stage_fp8.restype = _I
    lib.oracle_decode_attention_stage_fp8.argtypes = [_u16p, _I, _u8p, _u8p, _D, _D, _i32p,
                                                      _L, _L, _L, _L, _L, _f64p, _I]
    lib.oracle_decode_fp8.restype = _I
    lib.oracle_decode_fp8.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, _D, _D,
                                      _L, _L, _L, _L, _L, _u8p, _u8p, _D, _D, _i32p, _L,
                                      _f64p, _f64p, _f64p, _f64p, _u8p, _u8p, _f64p, _I]
    lib.oracle_backward.restype = _I
    lib.oracle_backward.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, _D, _D, _L, _L, _L, _L, _L, _L, _I,
                                    _u16p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _I]
    lib.oracle_backward_rd.restype = _I
    lib.oracle_backward_rd.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, _D, _D, _L, _L, _L, _L, _L, _L, _L, _I,
                                       _u16p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _I]
    lib.oracle_attention_backward.restype = _I
    lib.oracle_attention_backward.argtypes = [_u16p, _u16p, _u16p, _u16p, _I, _L, _L, _L, _L, _L, _I,
                                              _f64p, _f64p, _f64p, _I]
    # the *_rd forms take the rotary width (reading R16) after eps
    lib.oracle_rope_rows_rd.restype = _I
    lib.oracle_rope_rows_rd.argtypes = [_f64p, _L, _L, _L, _f64p, _D, _f64p]
    for name in ("oracle_qkv_stage", "oracle_forward", "oracle_decode", "oracle_prefill_cached"):
        base = getattr(lib, name).argtypes
        f = getattr(lib, name + "_rd")
        f.restype = _I
        f.argtypes = base[:7] + [_L] + base[7:]
    _lib = lib
    return lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------- marshalling

def _bits(t, allow_f16=False):
    """bf16 (or, where allowed, float16) torch tensor, or uint16 numpy array
    -> contiguous uint16 numpy array of the 16-bit patterns."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16 or (allow_f16 and t.dtype == torch.float16), t.dtype
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _is_f16(t):
    import torch
    return isinstance(t, torch.Tensor) and t.dtype == torch.float16


def _p16(a):
    return None if a is None else a.ctypes.data_as(_u16p)


def _pf(a):
    return None if a is None else a.ctypes.data_as(_f64p)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with status {rc}")


def _sel(sel, total):
    if sel is None:
        return None, total
    a = np.ascontiguousarray(np.asarray(sel, dtype=np.int64))
    return a, a.shape[0]


# ---------------------------------------------------------------- public API

def effective_head_dim(hidden, heads, head_dim=None) -> int:
    return int(_load().oracle_effective_head_dim(hidden, heads, head_dim or 0))


def widths(hidden, Hq, Hkv, d) -> dict:
    out = (ctypes.c_long * 5)()
    _load().oracle_widths(hidden, Hq, Hkv, d, out)
    return {"query_hidden": out[0], "kv_hidden": out[1], "qkv_out": out[2],
            "o_in": out[3], "o_out": out[4]}


def attn_param_count(hidden, Hq, Hkv, d) -> int:
    return int(_load().oracle_attn_param_count(hidden, Hq, Hkv, d))


def proj_macs_per_token(hidden, Hq, Hkv, d) -> int:
    return int(_load().oracle_proj_macs_per_token(hidden, Hq, Hkv, d))


def score_value_macs_per_token(n, Hq, d) -> int:
    return int(_load().oracle_score_value_macs_per_token(n, Hq, d))


def rmsnorm_rows(rows: np.ndarray, w, eps: float) -> np.ndarray:
    rows = np.ascontiguousarray(rows, dtype=np.float64)
    n, d = rows.shape
    out = np.empty_like(rows)
    wb = _bits(w)
    _check(_load().oracle_rmsnorm_rows(_pf(rows), n, d, _p16(wb), eps, _pf(out)), "rmsnorm")
    return out


def _rd(rotary_dim, d):
    return d if rotary_dim is None else int(rotary_dim)


def rope_rows(rows: np.ndarray, pos, theta: float, rotary_dim=None) -> np.ndarray:
    """RoPE of each row at its position; rotary_dim (default: the row
    length) rotates only the first rotary_dim features (reading R16)."""
    rows = np.ascontiguousarray(rows, dtype=np.float64)
    n, d = rows.shape
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.float64), (n,)))
    out = np.empty_like(rows)
    _check(_load().oracle_rope_rows_rd(_pf(rows), n, d, _rd(rotary_dim, d), _pf(p), theta, _pf(out)), "rope")
    return out


def linear(x, W, threads=None) -> np.ndarray:
    xb, wb = _bits(x), _bits(W)
    K = xb.shape[-1]
    M = xb.size // K
    N = wb.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_linear(_p16(xb), _p16(wb), M, N, K, _pf(y), threads or default_threads()),
           "linear")
    return y.reshape(*xb.shape[:-1], N)


def qkv_stage(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, d,
              threads=None, rotary_dim=None):
    """Q [B,Hq,S,d], K/V [B,Hkv,S,d] after projection, QK-norm and RoPE."""
    q = np.empty((B, Hq, S, d)); k = np.empty((B, Hkv, S, d)); v = np.empty((B, Hkv, S, d))
    xb, wb, qn, kn = _bits(x), _bits(Wqkv), _bits(q_norm_w), _bits(k_norm_w)
    _check(_load().oracle_qkv_stage_rd(_p16(xb), _p16(wb), _p16(qn), _p16(kn), rope_theta, eps,
                                       _rd(rotary_dim, d), B, S, hidden, Hq, Hkv, d, _pf(q), _pf(k), _pf(v),
                                    threads or default_threads()), "qkv_stage")
    return q, k, v


def round_bf16(x) -> np.ndarray:
    """x (float64) rounded to the nearest bf16 value, ties to even: how a bf16
    KV cache stores a new key or value (reading R21)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(a)
    _check(_load().oracle_round_bf16(_pf(a), a.size, _pf(out)), "round_bf16")
    return out


def f16_to_double(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).reshape(-1)
    out = np.empty(b.shape[0])
    _load().oracle_f16_to_double(_p16(b), b.shape[0], _pf(out))
    return out.reshape(np.shape(bits))


def attention_stage(Q, K, V, B, S, Hq, Hkv, d, causal=True, sel=None, threads=None):
    """attn [n_sel, Hq*d] from Q [B,Hq,S,d], K/V [B,Hkv,S,d], all bf16 or all float16."""
    s, n = _sel(sel, B * S)
    out = np.empty((n, Hq * d))
    f16 = _is_f16(Q)
    assert _is_f16(K) == f16 and _is_f16(V) == f16, "Q, K and V must share one 16-bit format"
    qb, kb, vb = _bits(Q, True), _bits(K, True), _bits(V, True)
    _check(_load().oracle_attention_stage(_p16(qb), _p16(kb), _p16(vb), int(f16), B, S, Hq, Hkv, d,
                                          int(causal), None if s is None else s.ctypes.data_as(_i64p),
                                          n, _pf(out), threads or default_threads()),
           "attention_stage")
    return out


def oproj_stage(attn, Wo, x, M, hidden, QW, sel=None, threads=None):
    """out [n_sel, hidden] = x + attn @ Wo^T from bf16 attn [M,QW], Wo, x."""
    s, n = _sel(sel, M)
    out = np.empty((n, hidden))
    ab, wb, xb = _bits(attn), _bits(Wo), _bits(x)
    _check(_load().oracle_oproj_stage(_p16(ab), _p16(wb), _p16(xb), M, hidden, QW,
                                      None if s is None else s.ctypes.data_as(_i64p), n,
                                      _pf(out), threads or default_threads()), "oproj_stage")
    return out


def forward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, d,
            causal=True, sel=None, want_stages=False, threads=None, rotary_dim=None):
    """The whole layer.  Returns out [n_sel, hidden]; with want_stages also
    q [n_sel,Hq,d], attn [n_sel,Hq*d], k/v [B,Hkv,S,d] (all float64)."""
    s, n = _sel(sel, B * S)
    out = np.empty((n, hidden))
    q = np.empty((n, Hq, d)) if want_stages else None
    a = np.empty((n, Hq * d)) if want_stages else None
    k = np.empty((B, Hkv, S, d)) if want_stages else None
    v = np.empty((B, Hkv, S, d)) if want_stages else None
    xb, wb, ob, qn, kn = _bits(x), _bits(Wqkv), _bits(Wo), _bits(q_norm_w), _bits(k_norm_w)
    _check(_load().oracle_forward_rd(_p16(xb), _p16(wb), _p16(ob), _p16(qn), _p16(kn), rope_theta,
                                     eps, _rd(rotary_dim, d), B, S, hidden, Hq, Hkv, d, int(causal),
                                  None if s is None else s.ctypes.data_as(_i64p), n,
                                  _pf(q), _pf(a), _pf(out), _pf(k), _pf(v),
                                  threads or default_threads()), "forward")
    if want_stages:
        return {"out": out, "q": q, "attn": a, "k": k, "v": v}
    return out


def decode_attention_stage(q, k_cache, v_cache, kv_len, B, Hq, Hkv, d, Lmax, threads=None):
    """attn [B, Hq*d] of q [B,Hq,d] (bf16 or float16) over keys [0, kv_len[b])
    of the bf16 caches."""
    out = np.empty((B, Hq * d))
    kl = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
    qb, kb, vb = _bits(q, True), _bits(k_cache), _bits(v_cache)
    _check(_load().oracle_decode_attention_stage(_p16(qb), int(_is_f16(q)), _p16(kb), _p16(vb),
                                                 kl.ctypes.data_as(_i32p), B, Hq, Hkv, d, Lmax,
                                                 _pf(out), threads or default_threads()),
           "decode_attention_stage")
    return out


def prefill_cached(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, d,
                   k_cache, v_cache, p0, Lmax, causal=True, threads=None, rotary_dim=None):
    """S new tokens per sequence at positions p0[b].. after p0[b] cached ones.
    Returns dict out [B*S, hidden], k/v [B,Hkv,S,d] (the new tokens'), attn
    [B*S, Hq*d]; the caches are read, not modified."""
    out = np.empty((B * S, hidden)); kn_ = np.empty((B, Hkv, S, d)); vn_ = np.empty((B, Hkv, S, d))
    a = np.empty((B * S, Hq * d))
    p = np.ascontiguousarray(np.asarray(p0, dtype=np.int32))
    xb, wb, ob, qn, kn = _bits(x), _bits(Wqkv), _bits(Wo), _bits(q_norm_w), _bits(k_norm_w)
    kb, vb = _bits(k_cache), _bits(v_cache)
    _check(_load().oracle_prefill_cached_rd(_p16(xb), _p16(wb), _p16(ob), _p16(qn), _p16(kn), rope_theta, eps,
                                            _rd(rotary_dim, d), B, S, hidden, Hq, Hkv, d, int(causal), _p16(kb), _p16(vb),
                                         p.ctypes.data_as(_i32p), Lmax, _pf(out), _pf(kn_), _pf(vn_), _pf(a),
                                         threads or default_threads()), "prefill_cached")
    return {"out": out, "k": kn_, "v": vn_, "attn": a}


def decode(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, hidden, Hq, Hkv, d,
           k_cache, v_cache, cache_len, Lmax, threads=None, rotary_dim=None):
    """One decode step.  Returns dict out [B,hidden], q [B,Hq,d], k/v [B,Hkv,d]
    (the new token's), attn [B,Hq*d]; the caches are read, not modified."""
    out = np.empty((B, hidden)); q = np.empty((B, Hq, d))
    kn_ = np.empty((B, Hkv, d)); vn_ = np.empty((B, Hkv, d)); a = np.empty((B, Hq * d))
    cl = np.ascontiguousarray(np.asarray(cache_len, dtype=np.int32))
    xb, wb, ob, qn, kn = _bits(x), _bits(Wqkv), _bits(Wo), _bits(q_norm_w), _bits(k_norm_w)
    kb, vb = _bits(k_cache), _bits(v_cache)
    _check(_load().oracle_decode_rd(_p16(xb), _p16(wb), _p16(ob), _p16(qn), _p16(kn), rope_theta, eps,
                                    _rd(rotary_dim, d), B, hidden, Hq, Hkv, d, _p16(kb), _p16(vb), cl.ctypes.data_as(_i32p),
                                 Lmax, _pf(out), _pf(q), _pf(kn_), _pf(vn_), _pf(a),
                                 threads or default_threads()), "decode")
    return {"out": out, "q": q, "k": kn_, "v": vn_, "attn": a}


# ------------------------------------------------------------- FP8 KV cache (reading R17)

def _codes(a):
    """uint8 E4M3 codes: a numpy uint8 array or a torch uint8 / float8_e4m3fn tensor."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint8
        return np.ascontiguousarray(a)
    import torch
    t = a.detach().cpu().contiguous()
    if t.dtype != torch.uint8:
        t = t.view(torch.uint8)
    return t.numpy()


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes -> float64 (exact)."""
    c = _codes(codes)
    flat = c.reshape(-1)
    out = np.empty(flat.shape[0])
    _load().oracle_e4m3_decode(flat.ctypes.data_as(_u8p), flat.shape[0], _pf(out))
    return out.reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    """float64 values -> nearest E4M3 codes (ties to even, saturating at +-448)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    flat = a.reshape(-1)
    out = np.empty(flat.shape[0], dtype=np.uint8)
    _load().oracle_e4m3_encode(_pf(flat), flat.shape[0], out.ctypes.data_as(_u8p))
    return out.reshape(a.shape)


def decode_attention_stage_fp8(q, k_codes, v_codes, k_scale, v_scale, kv_len, B, Hq, Hkv, d, Lmax,
                               threads=None):
    """attn [B, Hq*d] of q [B,Hq,d] (bf16 or float16) over keys [0, kv_len[b])
    of FP8 caches [B,Hkv,Lmax,d] worth code * scale."""
    out = np.empty((B, Hq * d))
    kl = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
    qb, kb, vb = _bits(q, True), _codes(k_codes), _codes(v_codes)
    _check(_load().oracle_decode_attention_stage_fp8(_p16(qb), int(_is_f16(q)), kb.ctypes.data_as(_u8p),
                                                     vb.ctypes.data_as(_u8p), k_scale, v_scale,
                                                     kl.ctypes.data_as(_i32p), B, Hq, Hkv, d, Lmax,
                                                     _pf(out), threads or default_threads()),
           "decode_attention_stage_fp8")
    return out


def decode_fp8(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, hidden, Hq, Hkv, d,
               k_codes, v_codes, k_scale, v_scale, cache_len, Lmax, threads=None):
    """One decode step over FP8 caches.  Returns dict out [B,hidden], q
    [B,Hq,d], k/v [B,Hkv,d] (the new token's, before quantisation), k_code /
    v_code [B,Hkv,d] (uint8, as appended), attn [B,Hq*d]; the caches are read,
    not modified."""
    out = np.empty((B, hidden)); q = np.empty((B, Hq, d))
    kn_ = np.empty((B, Hkv, d)); vn_ = np.empty((B, Hkv, d)); a = np.empty((B, Hq * d))
    kc_ = np.empty((B, Hkv, d), dtype=np.uint8); vc_ = np.empty((B, Hkv, d), dtype=np.uint8)
    cl = np.ascontiguousarray(np.asarray(cache_len, dtype=np.int32))
    xb, wb, ob, qn, kn = _bits(x), _bits(Wqkv), _bits(Wo), _bits(q_norm_w), _bits(k_norm_w)
    kb, vb = _codes(k_codes), _codes(v_codes)
    _check(_load().oracle_decode_fp8(_p16(xb), _p16(wb), _p16(ob), _p16(qn), _p16(kn), rope_theta, eps,
                                     B, hidden, Hq, Hkv, d, kb.ctypes.data_as(_u8p), vb.ctypes.data_as(_u8p),
                                     k_scale, v_scale, cl.ctypes.data_as(_i32p), Lmax, _pf(out), _pf(q),
                                     _pf(kn_), _pf(vn_), kc_.ctypes.data_as(_u8p), vc_.ctypes.data_as(_u8p),
                                     _pf(a), threads or default_threads()), "decode_fp8")
    return {"out": out, "q": q, "k": kn_, "v": vn_, "k_code": kc_, "v_code": vc_, "attn": a}


# ------------------------------------------------------------- backward

def backward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, d, dout,
             causal=True, want_stages=False, threads=None, rotary_dim=None):
    """Gradients of the layer given dout = dL/dout [B*S, hidden] (bf16).
    Returns dict dx [B*S, hidden], dWqkv [(Hq+2Hkv)d, hidden], dWo [hidden,
    Hq*d], dq_norm_w / dk_norm_w [d]; with want_stages also d_attn [B*S,
    Hq*d] and the attention-input gradients dq [B,Hq,S,d], dk/dv [B,Hkv,S,d]."""
    lib = _load()
    N = (Hq + 2 * Hkv) * d
    dx = np.empty((B * S, hidden)); dW = np.empty((N, hidden)); dWo = np.empty((hidden, Hq * d))
    dqn = np.empty(d); dkn = np.empty(d)
    da = np.empty((B * S, Hq * d)) if want_stages else None
    dq = np.empty((B, Hq, S, d)) if want_stages else None
    dk = np.empty((B, Hkv, S, d)) if want_stages else None
    dv = np.empty((B, Hkv, S, d)) if want_stages else None
    xb, wb, ob, qn, kn, gb = _bits(x), _bits(Wqkv), _bits(Wo), _bits(q_norm_w), _bits(k_norm_w), _bits(dout)
    _check(lib.oracle_backward_rd(_p16(xb), _p16(wb), _p16(ob), _p16(qn), _p16(kn), rope_theta, eps,
                                  _rd(rotary_dim, d), B, S, hidden, Hq, Hkv, d, int(causal), _p16(gb), _pf(dx),
                                  _pf(dW), _pf(dWo), _pf(dqn), _pf(dkn), _pf(da), _pf(dq), _pf(dk), _pf(dv),
                                  threads or default_threads()), "backward")
    res = {"dx": dx, "dWqkv": dW, "dWo": dWo, "dq_norm_w": dqn, "dk_norm_w": dkn}
    if want_stages:
        res.update({"d_attn": da, "dq": dq, "dk": dk, "dv": dv})
    return res


def attention_backward(Q, K, V, dO, B, S, Hq, Hkv, d, causal=True, threads=None):
    """dq [B,Hq,S,d], dk/dv [B,Hkv,S,d] of the attention alone, from 16-bit
    Q [B,Hq,S,d], K/V [B,Hkv,S,d], dO [B,S,Hq*d] (all bf16 or all float16)."""
    lib = _load()
    f16 = _is_f16(Q)
    assert all(_is_f16(t) == f16 for t in (K, V, dO)), "Q, K, V and dO must share one 16-bit format"
    dq = np.empty((B, Hq, S, d)); dk = np.empty((B, Hkv, S, d)); dv = np.empty((B, Hkv, S, d))
    qb, kb, vb, gb = _bits(Q, True), _bits(K, True), _bits(V, True), _bits(dO, True)
    _check(lib.oracle_attention_backward(_p16(qb), _p16(kb), _p16(vb), _p16(gb), int(f16), B, S, Hq, Hkv, d,
                                         int(causal), _pf(dq), _pf(dk), _pf(dv), threads or default_threads()),
           "attention_backward")
    return dq, dk, dv
