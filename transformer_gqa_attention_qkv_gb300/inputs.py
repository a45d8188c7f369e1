"""Seeded synthetic inputs for the attention layer and its decode step.

This module only draws random numbers and names workload shapes.  It holds
none of the layer's arithmetic, so both the CUDA path and the CPU oracle can be
fed from it without sharing any computation.

Workloads (shapes of the Qwen3 geometries and the Vaswani layer named on the
pages; value recipe: x ~ N(0,1), projection weights ~ N(0, 0.02), QK-norm
weights ~ 1 + N(0, 0.1), KV-cache entries ~ N(0,1); every draw is fp32 from a
seeded ``torch.Generator`` and then rounded to bf16):

* ``qwen3_0p6b``  B=1,  S=128,   hidden=1024, Hq=16, Hkv=8, d=128, QK-norm, theta 1e6
* ``vaswani_mha`` B=8,  S=2048,  hidden=512,  Hq=8,  Hkv=8, d=64,  no QK-norm, theta 1e4
* ``qwen3_4b``    B=4,  S=4096,  hidden=2560, Hq=32, Hkv=8, d=128, QK-norm, theta 1e6
* ``qwen3_32b``   B=1,  S=16384, hidden=5120, Hq=64, Hkv=8, d=128, QK-norm, theta 1e6
* ``qwen3_8b_decode`` 64 sequences x 1 new token over 8192 cached tokens,
  hidden=4096, Hq=32, Hkv=8, d=128, QK-norm, theta 1e6
* ``gemma3_d256`` B=4, S=4096, hidden=640, Hq=4, Hkv=1, d=256, QK-norm, theta 1e6
* ``qwen3_4b_d80`` the Qwen3-4B widths with head_dim = hidden / Hq = 80
* ``knob_d96``    B=4, S=4096, hidden=3072, Hq=32, Hkv=8, d=96 (= hidden / Hq)
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerConfig:
    name: str
    B: int
    S: int
    hidden: int
    Hq: int
    Hkv: int
    head_dim: int
    qk_norm: bool
    rope_theta: float
    eps: float = 1e-6
    causal: bool = True

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    cache_len: int
    hidden: int
    Hq: int
    Hkv: int
    head_dim: int
    qk_norm: bool
    rope_theta: float
    eps: float = 1e-6
    Lmax: int = 0  # 0: cache_len + 1

    @property
    def lmax(self) -> int:
        return self.Lmax if self.Lmax > 0 else self.cache_len + 1

    def with_(self, **kw) -> "DecodeConfig":
        return replace(self, **kw)


PREFILL_CONFIGS = {
    "qwen3_0p6b": LayerConfig("qwen3_0p6b", 1, 128, 1024, 16, 8, 128, True, 1e6),
    "vaswani_mha": LayerConfig("vaswani_mha", 8, 2048, 512, 8, 8, 64, False, 1e4),
    "qwen3_4b": LayerConfig("qwen3_4b", 4, 4096, 2560, 32, 8, 128, True, 1e6),
    "qwen3_32b": LayerConfig("qwen3_32b", 1, 16384, 5120, 64, 8, 128, True, 1e6),
    # head_dim 256 at the Gemma-3 example's width (hidden 640, four query heads);
    # one KV head, batch and length are this workload's own choice
    "gemma3_d256": LayerConfig("gemma3_d256", 4, 4096, 640, 4, 1, 256, True, 1e6),
    # head widths that are not a power of two: Qwen3-4B's hidden / heads quotient
    # (80) and the width 96; hidden 3072 makes 96 the quotient of 32 heads
    "qwen3_4b_d80": LayerConfig("qwen3_4b_d80", 4, 4096, 2560, 32, 8, 80, True, 1e6),
    "knob_d96": LayerConfig("knob_d96", 4, 4096, 3072, 32, 8, 96, True, 1e6),
}
DECODE_CONFIGS = {
    "qwen3_8b_decode": DecodeConfig("qwen3_8b_decode", 64, 8192, 4096, 32, 8, 128, True, 1e6),
}
# seeds: 1000 + position of the workload in the list above
SEEDS = {"qwen3_0p6b": 1000, "vaswani_mha": 1001, "qwen3_4b": 1002,
         "qwen3_32b": 1003, "qwen3_8b_decode": 1004, "gemma3_d256": 1005,
         "qwen3_4b_d80": 1006, "knob_d96": 1007}


def _normal(shape, gen, std, mean=0.0, device="cpu"):
    t = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_layer_inputs(cfg: LayerConfig, seed: int, *, w_std: float = 0.02,
                      x_std: float = 1.0, norm_std: float = 0.1, wo_std: float | None = None,
                      device: str = "cpu") -> dict:
    """bf16 tensors x [B,S,hidden], Wqkv [(Hq+2Hkv)d, hidden] (rows: W_q, W_k,
    W_v), Wo [hidden, Hq d], q_norm_w / k_norm_w [d] (None without QK-norm).
    wo_std defaults to w_std."""
    g = _gen(seed, device)
    d = cfg.head_dim
    n_qkv = (cfg.Hq + 2 * cfg.Hkv) * d
    x = _normal((cfg.B, cfg.S, cfg.hidden), g, x_std, device=device)
    wqkv = _normal((n_qkv, cfg.hidden), g, w_std, device=device)
    wo = _normal((cfg.hidden, cfg.Hq * d), g, w_std if wo_std is None else wo_std, device=device)
    if cfg.qk_norm:
        qn = _normal((d,), g, norm_std, 1.0, device=device)
        kn = _normal((d,), g, norm_std, 1.0, device=device)
    else:
        qn = kn = None
    return {"x": x, "Wqkv": wqkv, "Wo": wo, "q_norm_w": qn, "k_norm_w": kn}


def make_decode_inputs(cfg: DecodeConfig, seed: int, *, w_std: float = 0.02,
                       norm_std: float = 0.1, device: str = "cpu") -> dict:
    """bf16 x [B,hidden], Wqkv, Wo, norm weights, and caches k_cache/v_cache
    [B,Hkv,Lmax,d] whose entries [0, cache_len) are N(0,1) (standing for
    already normed and rotated keys) and whose remaining slots are zero;
    cache_len is an int32 tensor [B]."""
    g = _gen(seed, device)
    d = cfg.head_dim
    n_qkv = (cfg.Hq + 2 * cfg.Hkv) * d
    x = _normal((cfg.B, cfg.hidden), g, 1.0, device=device)
    wqkv = _normal((n_qkv, cfg.hidden), g, w_std, device=device)
    wo = _normal((cfg.hidden, cfg.Hq * d), g, w_std, device=device)
    if cfg.qk_norm:
        qn = _normal((d,), g, norm_std, 1.0, device=device)
        kn = _normal((d,), g, norm_std, 1.0, device=device)
    else:
        qn = kn = None
    L, Lmax = cfg.cache_len, cfg.lmax
    kc = torch.zeros((cfg.B, cfg.Hkv, Lmax, d), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    if L > 0:
        kc[:, :, :L].copy_(_normal((cfg.B, cfg.Hkv, L, d), g, 1.0, device=device))
        vc[:, :, :L].copy_(_normal((cfg.B, cfg.Hkv, L, d), g, 1.0, device=device))
    cache_len = torch.full((cfg.B,), L, dtype=torch.int32, device=device)
    return {"x": x, "Wqkv": wqkv, "Wo": wo, "q_norm_w": qn, "k_norm_w": kn,
            "k_cache": kc, "v_cache": vc, "cache_len": cache_len}


def sample_rows(B: int, S: int, n_per_batch: int, seed: int, tile: int = 128) -> torch.Tensor:
    """Flattened token indices b*S+t for a sampled check: the first, second,
    last rows, the rows on both sides of every tile edge, and seeded random
    rows; sorted and unique."""
    g = torch.Generator().manual_seed(seed)
    rows = []
    for b in range(B):
        fixed = {0, 1, S - 1}
        for e in range(tile, S, tile * max(1, S // (tile * 8))):
            fixed.update({e - 1, e})
        fixed = {t for t in fixed if 0 <= t < S}
        n_rand = max(0, n_per_batch - len(fixed))
        rnd = torch.randint(0, S, (n_rand,), generator=g).tolist() if n_rand else []
        rows.extend(b * S + t for t in sorted(fixed.union(rnd)))
    return torch.tensor(sorted(set(rows)), dtype=torch.int64)
