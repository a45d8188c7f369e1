"""Shared helpers of the parity tests: the tolerance and bf16 <-> float64.

Tolerance (stated for the layer's outputs in bf16 with fp32 accumulation):
  max|gpu - ref| <= 1e-2 * max|ref|   and   sum|gpu - ref| / sum|ref| <= 2e-3
where ref is the fp64 oracle on the same bf16 inputs.
"""
import numpy as np
import torch

TOL_MAX = 1e-2
TOL_REL = 2e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def errors(gpu: np.ndarray, ref: np.ndarray):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    err = np.abs(gpu - ref)
    max_ref = float(np.abs(ref).max()) if ref.size else 0.0
    den = float(np.abs(ref).sum())
    rel = float(err.sum() / den) if den > 0 else float(err.sum())
    return float(err.max()) if err.size else 0.0, max_ref, rel


def assert_parity(name: str, gpu, ref, tol_max: float = TOL_MAX, tol_rel: float = TOL_REL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values in GPU output"
    emax, rmax, rel = errors(gpu, ref)
    msg = f"{name}: max|err|={emax:.3e} (limit {tol_max * rmax:.3e}), rel-L1={rel:.3e} (limit {tol_rel:.1e})"
    print(msg)
    assert emax <= tol_max * rmax and rel <= tol_rel, msg
