"""Shared helpers of the GPU parity tests: device copies and error norms."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances stated for this path: exact-fp32 storage must match the fp64 oracle
# to max-abs 1e-4; bf16 storage to relative L2 2e-2 per output tensor.
F32_MAX_ABS = 1e-4
BF16_REL_L2 = 2e-2


def to_dev(x: np.ndarray, dtype: str, dev="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return t.to(torch.bfloat16) if dtype == "bf16" else t.float()


def graph_to_dev(g, dev="cuda"):
    return torch.from_numpy(g.indptr).to(dev), torch.from_numpy(g.indices).to(dev)


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def max_abs(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, dtype: str):
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    if dtype == "f32":
        e = max_abs(got, ref)
        assert e <= F32_MAX_ABS, f"{name}: max-abs error {e:.3e} > {F32_MAX_ABS}"
    else:
        e = rel_l2(got, ref)
        assert e <= BF16_REL_L2, f"{name}: relative L2 error {e:.3e} > {BF16_REL_L2}"
    return e
