"""Shared helpers of the GPU parity tests: device copies and error norms."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances stated for this path: exact-fp32 storage must match the fp64 oracle
# to max-abs 1e-4; bf16 storage to relative L2 2e-2 per output tensor.
F32_MAX_ABS = 1e-4
BF16_REL_L2 = 2e-2
# lse is an fp32 output near ln N + max_j s_ij (about 10 here), so relative L2
# alone would let it drift by about 0.2, which scales every p_ij by 20 %.  bf16
# storage rounds only q, k, v (exact inputs of the oracle as well); lse itself
# comes from fp32 sums, so it is also held to an absolute bound.
BF16_LSE_MAX_ABS = 1e-3


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
        if name.startswith("lse"):
            a = max_abs(got, ref)
            assert a <= BF16_LSE_MAX_ABS, f"{name}: max-abs error {a:.3e} > {BF16_LSE_MAX_ABS}"
    return e


def stored_o_dT_bound(ref_o: np.ndarray, got_o: np.ndarray, dO: np.ndarray) -> np.ndarray:
    """Per head, the largest change of any dT entry that comes from the backward
    being given the stored (bf16-rounded) o' rather than the exact o.

    D_i = <dO_i, o_i> enters every dS_ij = p_ij (dP_ij - D_i) of row i; with o'
    in its place each dS_ij moves by p_ij <dO_i, o_i - o_i'>, and since the p_ij of
    a row sum to 1, a bucket's sum moves by at most sum_i |<dO_i, o_i - o_i'>|."""
    dO = np.asarray(dO, np.float64)
    return np.abs(((ref_o - got_o) * dO).sum(-1)).sum(0)           # [h]


def assert_dT_stored_o(got_dT, ref_dT, ref_o, got_o, dO, rel=BF16_REL_L2, floor=1e-5):
    """bf16 end-to-end dT against the oracle: within the stored-o bound above,
    plus rel of each entry (the kernels' own rounding) and a small floor."""
    bound = stored_o_dT_bound(ref_o, got_o, dO)
    err = np.abs(got_dT - ref_dT)
    lim = bound[:, None] * 1.05 + rel * np.abs(ref_dT) + floor
    assert np.all(err <= lim), ("dT beyond the stored-o bound", err.max(), bound)
    return float(err.max()), float(bound.max())

