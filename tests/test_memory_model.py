"""The memory model of one biased-attention layer (host arithmetic, no GPU).

The model itself is checked against measured peak memory in
test_gpu_memory.py; here its closed forms and the orders of magnitude the
five workloads give."""
import pytest

import gt_inputs as gi
from graph_transformer_attention_gb300 import memory as M


def test_materialised_closed_forms():
    n, h, d = 1000, 8, 16
    m = M.materialised_layer_bytes(n, h, d, "bf16")
    assert m["bias"] == 4 * h * n * n
    assert m["scores"] == m["probs"] == m["dprobs"] == m["dscores"] == 2 * h * n * n
    assert m["dense"] == 8 * n * h * d * 2
    # the largest coexisting set: bias + scores (6 h n^2) vs P + dP + dS (6 h n^2)
    assert m["peak_min"] == m["dense"] + 6 * h * n * n
    assert m["peak_max"] == m["dense"] + 12 * h * n * n
    f = M.materialised_layer_bytes(n, h, d, "f32")
    assert f["peak_min"] == f["dense"] + 12 * h * n * n      # P + dP + dS at 4 bytes


def test_blockwise_arithmetic_with_a_given_workspace():
    n, h, d, nb = 1000, 8, 8, 18
    ws = lambda code, n_, h_, d_, kvb: 5000 if kvb else 3000
    b = M.blockwise_layer_bytes(n, h, d, nb, "bf16", kv_block=256, workspace_bytes=ws)
    dense = n * h * d * 2
    assert b["spd"] == n * 1008                     # rows padded to 16 bytes
    assert b["base"] == n * 1008 + 4 * dense + 4 * h * nb
    assert b["fwd_phase"] == b["base"] + dense + 4 * h * n + 5000
    assert b["bwd_phase"] == b["base"] + dense + 4 * h * n + 3 * dense + 4 * h * nb + 3000
    assert b["peak"] == max(b["fwd_phase"], b["bwd_phase"])


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_blockwise_is_far_below_materialised(cfg):
    w = gi.CONFIGS[cfg]
    ws = lambda code, n_, h_, d_, kvb: 64 * n_ * h_       # order of the real workspace
    b = M.blockwise_layer_bytes(w.n, w.heads, w.head_dim, w.nb, w.dtype, w.kv_block, workspace_bytes=ws)
    m = M.materialised_layer_bytes(w.n, w.heads, w.head_dim, w.dtype)
    # the per-head N x N objects are what the blockwise form removes: the bucket
    # matrix is 1 byte per pair for all heads, against >= 6 H bytes per pair
    assert b["peak"] * 10 < m["peak_min"]
    assert b["spd"] >= w.n * w.n
