"""Device memory of one biased-attention layer: materialised against blockwise.

MegaGraph ("Towards Efficient Training of Large-Scale Graph Transformers with
Automated Hybrid Parallelism"), abstract: in every GT layer the attention score
matrix and its topology-aware bias matrix are N x N per head, and that memory is
what bounds the graph a GPU can train on.  This module counts the device bytes
of one layer's forward and backward both ways, for the sizes of a workload:

* materialised: the plain computation builds, per head, the bias matrix
  T[h][spd] (fp32), the score matrix and its softmax P (kept for the backward),
  and in the backward dP = dO V^T and dS; every one of them is N x N per head.
* blockwise (this library): the int8 bucket matrix (N x ld bytes, shared by the
  heads and by every layer), the [N][H][d] tensors, lse [H][N] fp32, T and dT,
  and the library workspace; no N x N object per head.

`blockwise_layer_bytes` follows the allocations the Python binding makes (one
workspace per call, sized by gt_bias_attn_workspace_size), so it predicts the
peak that torch's allocator reports for a forward + backward, up to the
allocator's 512-byte rounding.
"""
from __future__ import annotations

_ELEM = {"f32": 4, "bf16": 2}


def _ld(n: int) -> int:
    return (n + 15) // 16 * 16


def materialised_layer_bytes(n: int, h: int, d: int, dtype: str = "bf16") -> dict:
    """Bytes of the N x N per-head objects of a materialised forward + backward.

    `peak_min` is the largest set that must coexist whatever the order of the
    steps: bias and scores (scores = scale q k^T + bias), scores and P (the
    softmax), or P, dP and dS (dS = P (dP - D) needs P and dP) -- plus the
    [N][H][d] tensors.  `peak_max` keeps every one of them at once."""
    e = _ELEM[dtype]
    nn = n * n * h
    parts = {
        "bias": 4 * nn,          # T[h][spd[i][j]] gathered per head, fp32
        "scores": e * nn,        # scale q k^T + bias
        "probs": e * nn,         # softmax, saved for the backward
        "dprobs": e * nn,        # dO V^T
        "dscores": e * nn,       # P (dP - D)
    }
    dense = 8 * n * h * d * e    # q, k, v, o, dO, dq, dk, dv
    parts["dense"] = dense
    parts["peak_min"] = dense + max(parts["bias"] + parts["scores"], parts["scores"] + parts["probs"],
                                    parts["probs"] + parts["dprobs"] + parts["dscores"])
    parts["peak_max"] = dense + sum(parts[k] for k in ("bias", "scores", "probs", "dprobs", "dscores"))
    return parts


def blockwise_layer_bytes(n: int, h: int, d: int, nb: int, dtype: str = "bf16", kv_block: int = 0,
                          workspace_bytes=None) -> dict:
    """Bytes of one blockwise forward + backward through this library.

    base: the caller's inputs (bucket matrix, q, k, v, dO, T); fwd: + o, lse and
    the forward workspace; bwd: + o, lse, dq, dk, dv, dT and the backward
    workspace.  `workspace_bytes(dtype_code, n, h, d, kv_block)` defaults to the
    library's gt_bias_attn_workspace_size."""
    if workspace_bytes is None:
        from . import gt_bias_attn_workspace_size as workspace_bytes
    e = _ELEM[dtype]
    code = 0 if dtype == "f32" else 1
    dense = n * h * d * e
    base = {"spd": n * _ld(n), "q": dense, "k": dense, "v": dense, "dO": dense, "T": 4 * h * nb}
    base_total = sum(base.values())
    o_lse = dense + 4 * h * n
    ws_fwd = max(int(workspace_bytes(code, n, h, d, kv_block)), 256)
    ws_bwd = max(int(workspace_bytes(code, n, h, d, 0)), 256)
    fwd = base_total + o_lse + ws_fwd
    bwd = base_total + o_lse + 3 * dense + 4 * h * nb + ws_bwd
    return {**base, "base": base_total, "workspace_fwd": ws_fwd, "workspace_bwd": ws_bwd,
            "fwd_phase": fwd, "bwd_phase": bwd, "peak": max(fwd, bwd)}
