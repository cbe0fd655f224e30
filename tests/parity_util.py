"""Shared helpers for the GPU parity tests: tolerances and error metrics.

Tolerances (written here once, used by every parity test): for bf16 inputs with fp32
accumulation the GPU result must be within max-abs 2e-2 and relative L2 1e-2 of the oracle;
with the FP8 latent cache both bounds are 5e-2.  Metrics are taken in float64 over the whole
compared tensor.
"""
import math

import numpy as np
import torch

TOL_BF16 = dict(max_abs=2e-2, rel_l2=1e-2)
TOL_FP8 = dict(max_abs=5e-2, rel_l2=5e-2)
SCALE = 1.0 / math.sqrt(192.0)


def to_f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def errors(got, ref):
    g, r = to_f64(got), to_f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    d = g - r
    return float(np.abs(d).max()), float(np.linalg.norm(d) / max(np.linalg.norm(r), 1e-300))


def assert_close(got, ref, tol=TOL_BF16, what=""):
    g = to_f64(got)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    max_abs, rel = errors(g, ref)
    assert max_abs <= tol["max_abs"] and rel <= tol["rel_l2"], (
        f"{what}: max_abs {max_abs:.3e} (tol {tol['max_abs']}), rel_l2 {rel:.3e} (tol {tol['rel_l2']})")
    return max_abs, rel


def bf16_round(x: np.ndarray) -> torch.Tensor:
    """Round float64 values to bf16 (round to nearest even), as a CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float32).to(torch.bfloat16)
