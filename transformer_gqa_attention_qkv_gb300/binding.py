"""ctypes binding of ``libgqa_attn.so`` (declared in ``include/gqa_attn.h``).

Argument marshalling only: every function takes torch tensors on the current
CUDA device, checks dtype/contiguity, and passes raw pointers, sizes and the
current torch stream to the C entry point of the same name.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If the
library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_attn.so")

GQA_OK = 0
GQA_ERR_ARG = -1
GQA_ERR_UNSUPPORTED = -2
GQA_ERR_CUDA = -3
GQA_ERR_TIMEOUT = -4
GQA_ERR_WORKSPACE = -5
GQA_ERR_RANGE = -6

# every symbol include/gqa_attn.h declares
EXPORTS = (
    "gqa_attn_workspace_size", "gqa_attn_forward_ex", "gqa_attn_forward", "gqa_qkv_proj",
    "gqa_attention", "gqa_oproj_residual", "gqa_attn_decode_workspace_size", "gqa_attn_decode",
    "gqa_decode_qkv", "gqa_decode_attention_workspace_size", "gqa_decode_attention",
    "gqa_attn_cost", "gqa_last_error", "gqa_check_device_error", "gqa_selftest_bounded_wait",
    "gqa_last_launch_count", "gqa_set_cta_pairs", "gqa_decode_attention_noalloc", "gqa_check_stream_error",
    "gqa_attn_prefill_cached_workspace_size", "gqa_attn_prefill_cached", "gqa_attention_cached",
    "gqa_attention_cached_workspace_size",
    "gqa_attn_forward_rd", "gqa_qkv_proj_rd", "gqa_attn_prefill_cached_rd", "gqa_attn_decode_rd",
    "gqa_decode_qkv_rd", "gqa_attn_decode_fp8", "gqa_decode_qkv_fp8", "gqa_decode_attention_fp8",
    "gqa_attn_backward_workspace_size", "gqa_attn_backward", "gqa_attention_backward_workspace_size",
    "gqa_attention_backward", "gqa_attn_forward_host_workspace_size", "gqa_attn_forward_host",
    "gqa_attn_forward_train", "gqa_attn_backward_saved", "gqa_attn_backward_rd", "gqa_attn_forward_train_rd",
    "gqa_attn_backward_saved_rd",
)


class GqaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (status {code})")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t
_LLP = ctypes.POINTER(ctypes.c_longlong)


def lib():
    """Load the library once; raise if it is missing (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m transformer_gqa_attention_qkv_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    sig = {
        "gqa_attn_workspace_size": (_Z, [_I] * 6),
        "gqa_attn_forward_ex": (_I, [_P] * 5 + [_F, _F] + [_I] * 7 + [_P, _P, _Z, _P]),
        "gqa_attn_forward": (_I, [_P] * 5 + [_F, _F] + [_I] * 7 + [_P]),
        "gqa_attn_forward_host_workspace_size": (_Z, [_I] * 6),
        "gqa_attn_forward_host": (_I, [_P] * 5 + [_F, _F] + [_I] * 7 + [_P, _P, _Z, _P]),
        "gqa_qkv_proj": (_I, [_P] * 4 + [_F, _F] + [_I] * 6 + [_P] * 4),
        "gqa_attention": (_I, [_P] * 3 + [_I] * 6 + [_P, _P]),
        "gqa_oproj_residual": (_I, [_P] * 3 + [_I] * 3 + [_P, _P]),
        "gqa_attn_decode_workspace_size": (_Z, [_I] * 6),
        "gqa_attn_decode": (_I, [_P] * 5 + [_F, _F] + [_I] * 5 + [_P, _P, _P, _I, _P, _P, _Z, _P]),
        "gqa_decode_qkv": (_I, [_P] * 4 + [_F, _F] + [_I] * 5 + [_P, _P, _P, _I, _P, _P]),
        "gqa_decode_attention_workspace_size": (_Z, [_I] * 5),
        "gqa_decode_attention": (_I, [_P] * 4 + [_I] * 5 + [_P, _P, _Z, _P]),
        "gqa_attn_cost": (_I, [_I] * 7 + [_LLP] * 4),
        "gqa_last_error": (ctypes.c_char_p, []),
        "gqa_check_device_error": (_I, []),
        "gqa_check_stream_error": (_I, [_P]),
        "gqa_selftest_bounded_wait": (_I, [_I]),
        "gqa_last_launch_count": (_I, []),
        "gqa_set_cta_pairs": (_I, [_I]),
        "gqa_decode_attention_noalloc": (_I, [_P] * 4 + [_I] * 5 + [_P, _P]),
        "gqa_attn_prefill_cached_workspace_size": (_Z, [_I] * 6),
        "gqa_attention_cached_workspace_size": (_Z, [_I] * 4),
        "gqa_attn_prefill_cached": (_I, [_P] * 5 + [_F, _F] + [_I] * 7 + [_P, _P, _P, _I, _P, _P, _Z, _P]),
        "gqa_attention_cached": (_I, [_P] * 4 + [_I] * 7 + [_P, _P, _Z, _P]),
    }
    # the *_rd forms: rotary_dim (int) right after rope_theta and eps
    for base, name in (("gqa_attn_forward_ex", "gqa_attn_forward_rd"), ("gqa_qkv_proj", "gqa_qkv_proj_rd"),
                       ("gqa_attn_prefill_cached", "gqa_attn_prefill_cached_rd"),
                       ("gqa_attn_decode", "gqa_attn_decode_rd"), ("gqa_decode_qkv", "gqa_decode_qkv_rd")):
        res, args = sig[base]
        k = args.index(_F) + 2
        sig[name] = (res, args[:k] + [_I] + args[k:])
    sig["gqa_attn_decode_fp8"] = (_I, [_P] * 5 + [_F, _F] + [_I] * 5 + [_P, _P, _F, _F, _P, _I, _P, _P, _Z, _P])
    sig["gqa_decode_qkv_fp8"] = (_I, [_P] * 4 + [_F, _F] + [_I] * 5 + [_P, _P, _F, _F, _P, _I, _P, _P])
    sig["gqa_decode_attention_fp8"] = (_I, [_P] * 3 + [_F, _F, _P] + [_I] * 5 + [_P, _P, _Z, _P])
    sig["gqa_attn_backward_workspace_size"] = (_Z, [_I] * 6)
    sig["gqa_attn_backward"] = (_I, [_P] * 5 + [_F, _F] + [_I] * 7 + [_P] * 6 + [_P, _Z, _P])
    sig["gqa_attn_backward_saved"] = sig["gqa_attn_backward"]
    sig["gqa_attn_forward_train"] = (_I, [_P] * 5 + [_F, _F] + [_I] * 7 + [_P, _P, _Z, _P])
    for base in ("gqa_attn_backward", "gqa_attn_backward_saved", "gqa_attn_forward_train"):
        res, args = sig[base]
        k = args.index(_F) + 2
        sig[base + "_rd"] = (res, args[:k] + [_I] + args[k:])
    sig["gqa_attention_backward_workspace_size"] = (_Z, [_I] * 4)
    sig["gqa_attention_backward"] = (_I, [_P] * 4 + [_I] * 6 + [_P] * 3 + [_P, _Z, _P])
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(rc: int):
    if rc != GQA_OK:
        msg = lib().gqa_last_error().decode(errors="replace")
        raise GqaError(rc, msg)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _bf16(t):
    if t is not None and t.dtype != torch.bfloat16:
        raise TypeError(f"expected bfloat16, got {t.dtype}")
    return _ptr(t)


def _f16(t):
    if t is not None and t.dtype != torch.float16:
        raise TypeError(f"expected float16, got {t.dtype}")
    return _ptr(t)


def _i32(t):
    if t.dtype != torch.int32:
        raise TypeError(f"expected int32, got {t.dtype}")
    return _ptr(t)


def _u8(t):
    """E4M3 codes: a uint8 or float8_e4m3fn tensor."""
    if t is not None and t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"expected uint8 or float8_e4m3fn codes, got {t.dtype}")
    return _ptr(t)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------------- prefill

def gqa_attn_workspace_size(B, S, hidden, Hq, Hkv, head_dim) -> int:
    return int(lib().gqa_attn_workspace_size(B, S, hidden, Hq, Hkv, head_dim))


def gqa_attn_forward_ex(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv,
                        head_dim, causal, out, workspace, stream=None):
    _check(lib().gqa_attn_forward_ex(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                     rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim, int(causal),
                                     _bf16(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))
    return out


def _host_bf16(t):
    """A contiguous bf16 tensor in host memory (page-locked for asynchronous copies)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.is_cuda:
        raise ValueError("tensor must be in host memory")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"expected bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def gqa_attn_forward_host_workspace_size(B, S, hidden, Hq, Hkv, head_dim) -> int:
    return int(lib().gqa_attn_forward_host_workspace_size(B, S, hidden, Hq, Hkv, head_dim))


def gqa_attn_forward_host(x_host, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv,
                          head_dim, causal, out_host, workspace, stream=None):
    """x_host / out_host: host tensors (pinned for overlap); out_host is complete once `stream` is."""
    _check(lib().gqa_attn_forward_host(_host_bf16(x_host), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w),
                                       _bf16(k_norm_w), rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim,
                                       int(causal), _host_bf16(out_host), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))
    return out_host


def gqa_attn_forward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv,
                     head_dim, causal, out):
    """Runs on the legacy default stream with the library's own workspace."""
    _check(lib().gqa_attn_forward(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                  rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim, int(causal), _bf16(out)))
    return out


def gqa_qkv_proj(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim,
                 q_out, k_out, v_out, stream=None):
    """q_out/k_out/v_out are float16 (binary16) tensors."""
    _check(lib().gqa_qkv_proj(_bf16(x), _bf16(Wqkv), _bf16(q_norm_w), _bf16(k_norm_w), rope_theta, eps,
                              B, S, hidden, Hq, Hkv, head_dim, _f16(q_out), _f16(k_out), _f16(v_out),
                              _stream(stream)))


# ------------------------------------------- partial rotary (rotary_dim < head_dim)

def gqa_attn_forward_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv,
                        head_dim, causal, out, workspace, stream=None):
    _check(lib().gqa_attn_forward_rd(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                     rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim, int(causal),
                                     _bf16(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))
    return out


def gqa_qkv_proj_rd(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim,
                    q_out, k_out, v_out, stream=None):
    _check(lib().gqa_qkv_proj_rd(_bf16(x), _bf16(Wqkv), _bf16(q_norm_w), _bf16(k_norm_w), rope_theta, eps,
                                 rotary_dim, B, S, hidden, Hq, Hkv, head_dim, _f16(q_out), _f16(k_out),
                                 _f16(v_out), _stream(stream)))


def gqa_attn_prefill_cached_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq,
                               Hkv, head_dim, causal, k_cache, v_cache, cache_len, Lmax, out, workspace,
                               stream=None):
    _check(lib().gqa_attn_prefill_cached_rd(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                            rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim,
                                            int(causal), _bf16(k_cache), _bf16(v_cache), _i32(cache_len), Lmax,
                                            _bf16(out), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def gqa_attn_decode_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, hidden, Hq, Hkv,
                       head_dim, k_cache, v_cache, cache_len, Lmax, out, workspace, stream=None):
    _check(lib().gqa_attn_decode_rd(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                    rope_theta, eps, rotary_dim, B, hidden, Hq, Hkv, head_dim, _bf16(k_cache),
                                    _bf16(v_cache), _i32(cache_len), Lmax, _bf16(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def gqa_decode_qkv_rd(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, hidden, Hq, Hkv, head_dim,
                      k_cache, v_cache, cache_len, Lmax, q_out, stream=None):
    _check(lib().gqa_decode_qkv_rd(_bf16(x), _bf16(Wqkv), _bf16(q_norm_w), _bf16(k_norm_w), rope_theta, eps,
                                   rotary_dim, B, hidden, Hq, Hkv, head_dim, _bf16(k_cache), _bf16(v_cache),
                                   _i32(cache_len), Lmax, _f16(q_out), _stream(stream)))


def gqa_attention(q, k, v, B, S, Hq, Hkv, head_dim, causal, attn_out, stream=None):
    """q/k/v are float16 (binary16) tensors; attn_out is bfloat16."""
    _check(lib().gqa_attention(_f16(q), _f16(k), _f16(v), B, S, Hq, Hkv, head_dim, int(causal),
                               _bf16(attn_out), _stream(stream)))


def gqa_oproj_residual(attn, Wo, x, M, hidden, q_width, out, stream=None):
    _check(lib().gqa_oproj_residual(_bf16(attn), _bf16(Wo), _bf16(x), M, hidden, q_width, _bf16(out),
                                    _stream(stream)))


# ------------------------------------------------------ prefill into a cache

def gqa_attn_prefill_cached_workspace_size(B, S, Hq, Hkv, head_dim, Lmax) -> int:
    return int(lib().gqa_attn_prefill_cached_workspace_size(B, S, Hq, Hkv, head_dim, Lmax))


def gqa_attention_cached_workspace_size(B, Hkv, head_dim, Lmax) -> int:
    return int(lib().gqa_attention_cached_workspace_size(B, Hkv, head_dim, Lmax))


def gqa_attn_prefill_cached(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim,
                            causal, k_cache, v_cache, cache_len, Lmax, out, workspace, stream=None):
    _check(lib().gqa_attn_prefill_cached(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                         rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim, int(causal),
                                         _bf16(k_cache), _bf16(v_cache), _i32(cache_len), Lmax, _bf16(out),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)))
    return out


def gqa_attention_cached(q, k_cache, v_cache, cache_len, B, S, Hq, Hkv, head_dim, Lmax, causal, attn_out,
                         workspace=None, stream=None):
    """workspace: None allocates one of gqa_attention_cached_workspace_size bytes."""
    if workspace is None:
        workspace = new_workspace(gqa_attention_cached_workspace_size(B, Hkv, head_dim, Lmax), q.device)
    _check(lib().gqa_attention_cached(_f16(q), _bf16(k_cache), _bf16(v_cache), _i32(cache_len), B, S, Hq, Hkv,
                                      head_dim, Lmax, int(causal), _bf16(attn_out), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)))


# -------------------------------------------------------------------- decode

def gqa_attn_decode_workspace_size(B, hidden, Hq, Hkv, head_dim, Lmax) -> int:
    return int(lib().gqa_attn_decode_workspace_size(B, hidden, Hq, Hkv, head_dim, Lmax))


def gqa_attn_decode(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, hidden, Hq, Hkv, head_dim,
                    k_cache, v_cache, cache_len, Lmax, out, workspace, stream=None):
    _check(lib().gqa_attn_decode(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                 rope_theta, eps, B, hidden, Hq, Hkv, head_dim, _bf16(k_cache),
                                 _bf16(v_cache), _i32(cache_len), Lmax, _bf16(out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def gqa_decode_qkv(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, B, hidden, Hq, Hkv, head_dim,
                   k_cache, v_cache, cache_len, Lmax, q_out, stream=None):
    _check(lib().gqa_decode_qkv(_bf16(x), _bf16(Wqkv), _bf16(q_norm_w), _bf16(k_norm_w), rope_theta, eps,
                                B, hidden, Hq, Hkv, head_dim, _bf16(k_cache), _bf16(v_cache),
                                _i32(cache_len), Lmax, _f16(q_out), _stream(stream)))


def gqa_decode_attention_workspace_size(B, Hq, Hkv, head_dim, Lmax) -> int:
    return int(lib().gqa_decode_attention_workspace_size(B, Hq, Hkv, head_dim, Lmax))


def gqa_decode_attention(q, k_cache, v_cache, kv_len, B, Hq, Hkv, head_dim, Lmax, attn_out, workspace,
                         stream=None):
    _check(lib().gqa_decode_attention(_f16(q), _bf16(k_cache), _bf16(v_cache), _i32(kv_len), B, Hq, Hkv,
                                      head_dim, Lmax, _bf16(attn_out), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)))


def gqa_decode_attention_noalloc(q, k_cache, v_cache, kv_len, B, Hq, Hkv, head_dim, Lmax, attn_out,
                                 stream=None):
    """Decode attention without a workspace, for callers that cannot allocate
    device memory: the split partials live in a fixed array inside the
    library.  Calls that overlap on the GPU race on that array."""
    _check(lib().gqa_decode_attention_noalloc(_f16(q), _bf16(k_cache), _bf16(v_cache), _i32(kv_len), B, Hq,
                                              Hkv, head_dim, Lmax, _bf16(attn_out), _stream(stream)))


# ---------------------------------------------------------------- accounting

def resolve_head_dim(hidden: int, Hq: int, head_dim: int | None = None) -> int:
    """The head width a model configuration implies ([NeoX] "Proposed
    configuration behavior"): an explicit head_dim wins and needs no relation
    to hidden (Qwen3-4B: hidden 2560, 32 heads, head_dim 128); without one it
    is hidden / Hq, and only then must Hq divide hidden.  Every entry point
    of the library takes the resolved value explicitly."""
    if head_dim is not None:
        if int(head_dim) <= 0:
            raise ValueError(f"head_dim={head_dim} must be positive")
        return int(head_dim)
    if Hq <= 0 or hidden <= 0 or hidden % Hq:
        raise ValueError(f"hidden={hidden} is not a positive multiple of Hq={Hq}: give head_dim explicitly")
    return hidden // Hq


def gqa_attn_cost(B, S, hidden, Hq, Hkv, head_dim, causal=True) -> dict:
    vals = [ctypes.c_longlong() for _ in range(4)]
    _check(lib().gqa_attn_cost(B, S, hidden, Hq, Hkv, head_dim, int(causal), *[ctypes.byref(v) for v in vals]))
    return {"weights": vals[0].value, "proj_macs_per_token": vals[1].value,
            "attn_macs": vals[2].value, "flops": vals[3].value}


def gqa_last_error() -> str:
    return lib().gqa_last_error().decode(errors="replace")


def gqa_check_device_error() -> int:
    return int(lib().gqa_check_device_error())


def gqa_check_stream_error(stream=None) -> int:
    """The device error check, waiting only for `stream` (default: the current stream)."""
    return int(lib().gqa_check_stream_error(_stream(stream)))


def gqa_selftest_bounded_wait(limit_ms: int) -> int:
    return int(lib().gqa_selftest_bounded_wait(limit_ms))


def gqa_last_launch_count() -> int:
    return int(lib().gqa_last_launch_count())


def gqa_set_cta_pairs(enable: bool) -> bool:
    """Use (True, the default) or avoid the 2-CTA-cluster kernel forms; returns the previous setting."""
    return bool(lib().gqa_set_cta_pairs(1 if enable else 0))


# --------------------------------------------------------- tensor helpers

def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A uint8 device buffer (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# --------------------------------------------------------- FP8 (E4M3) KV cache

def gqa_attn_decode_fp8(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, hidden, Hq, Hkv, head_dim,
                        k_cache, v_cache, k_scale, v_scale, cache_len, Lmax, out, workspace, stream=None):
    """k_cache / v_cache: E4M3 codes (uint8 or float8_e4m3fn) worth code * scale."""
    _check(lib().gqa_attn_decode_fp8(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                     rope_theta, eps, B, hidden, Hq, Hkv, head_dim, _u8(k_cache), _u8(v_cache),
                                     k_scale, v_scale, _i32(cache_len), Lmax, _bf16(out), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def gqa_decode_qkv_fp8(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, B, hidden, Hq, Hkv, head_dim,
                       k_cache, v_cache, k_scale, v_scale, cache_len, Lmax, q_out, stream=None):
    _check(lib().gqa_decode_qkv_fp8(_bf16(x), _bf16(Wqkv), _bf16(q_norm_w), _bf16(k_norm_w), rope_theta, eps,
                                    B, hidden, Hq, Hkv, head_dim, _u8(k_cache), _u8(v_cache), k_scale, v_scale,
                                    _i32(cache_len), Lmax, _f16(q_out), _stream(stream)))


def gqa_decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, kv_len, B, Hq, Hkv, head_dim, Lmax,
                             attn_out, workspace, stream=None):
    _check(lib().gqa_decode_attention_fp8(_f16(q), _u8(k_cache), _u8(v_cache), k_scale, v_scale, _i32(kv_len),
                                          B, Hq, Hkv, head_dim, Lmax, _bf16(attn_out), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


# ----------------------------------------------------------------- backward

def _f32(t):
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"expected float32, got {t.dtype}")
    return _ptr(t)


def gqa_attn_backward_workspace_size(B, S, hidden, Hq, Hkv, head_dim) -> int:
    return int(lib().gqa_attn_backward_workspace_size(B, S, hidden, Hq, Hkv, head_dim))


def gqa_attn_forward_train(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim,
                           causal, out, workspace, stream=None):
    """The forward, keeping in `workspace` (gqa_attn_backward_workspace_size bytes) what
    gqa_attn_backward_saved needs."""
    _check(lib().gqa_attn_forward_train(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                        rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim, int(causal), _bf16(out),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)))
    return out


def gqa_attn_backward_saved(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim,
                            causal, dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, stream=None):
    """gqa_attn_backward from the workspace gqa_attn_forward_train filled (nothing recomputed)."""
    _check(lib().gqa_attn_backward_saved(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                         rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim, int(causal), _bf16(dout),
                                         _bf16(dx), _f32(dWqkv), _f32(dWo), _f32(dq_norm_w), _f32(dk_norm_w),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)))


def gqa_attn_backward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim, causal,
                      dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, stream=None):
    """dx bf16; dWqkv, dWo, dq_norm_w, dk_norm_w float32."""
    _check(lib().gqa_attn_backward(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w), rope_theta,
                                   eps, B, S, hidden, Hq, Hkv, head_dim, int(causal), _bf16(dout), _bf16(dx),
                                   _f32(dWqkv), _f32(dWo), _f32(dq_norm_w), _f32(dk_norm_w), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def gqa_attention_backward_workspace_size(B, S, Hq, head_dim) -> int:
    return int(lib().gqa_attention_backward_workspace_size(B, S, Hq, head_dim))


def gqa_attention_backward(q, k, v, dO, B, S, Hq, Hkv, head_dim, causal, dq, dk, dv, workspace, stream=None):
    """q, k, v, dO float16 head-major; dq, dk, dv float32."""
    _check(lib().gqa_attention_backward(_f16(q), _f16(k), _f16(v), _f16(dO), B, S, Hq, Hkv, head_dim, int(causal),
                                        _f32(dq), _f32(dk), _f32(dv), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)))


# ----------------------------------------------- backward with partial rotary

def gqa_attn_backward_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv,
                         head_dim, causal, dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, stream=None):
    _check(lib().gqa_attn_backward_rd(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                      rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim, int(causal),
                                      _bf16(dout), _bf16(dx), _f32(dWqkv), _f32(dWo), _f32(dq_norm_w),
                                      _f32(dk_norm_w), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)))


def gqa_attn_forward_train_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv,
                              head_dim, causal, out, workspace, stream=None):
    _check(lib().gqa_attn_forward_train_rd(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                           rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim, int(causal),
                                           _bf16(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)))
    return out


def gqa_attn_backward_saved_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv,
                               head_dim, causal, dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, stream=None):
    _check(lib().gqa_attn_backward_saved_rd(_bf16(x), _bf16(Wqkv), _bf16(Wo), _bf16(q_norm_w), _bf16(k_norm_w),
                                            rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim,
                                            int(causal), _bf16(dout), _bf16(dx), _f32(dWqkv), _f32(dWo),
                                            _f32(dq_norm_w), _f32(dk_norm_w), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream(stream)))
