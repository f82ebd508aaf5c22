"""Launch statistics of libgt on the GPU: every kernel of a call is counted
under its name, and with timing on each gets a positive device time."""
import numpy as np
import pytest
import torch

import gt_inputs as gi
from tests.helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gt():
    import graph_transformer_attention_gb300 as m
    from graph_transformer_attention_gb300 import build
    build.build()
    m.load_library()
    return m


@pytest.mark.parametrize("timing", [False, True])
def test_counts_and_times_of_one_layer(gt, timing):
    n, h, d, nb = 300, 8, 16, 26
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=5)
    q, k, v, dO = (to_dev(x[a], "bf16") for a in ("q", "k", "v", "dO"))
    T = torch.from_numpy(x["T"]).cuda()
    codes = np.random.default_rng(5).integers(0, nb, size=(n, gt.spd_ld(n))).astype(np.int8)
    spd = torch.from_numpy(codes).cuda()
    torch.cuda.synchronize()
    gt.gt_kernel_stats_reset(timing)
    o, lse = gt.gt_bias_attn_fwd(q, k, v, spd, T)
    gt.gt_bias_attn_bwd(q, k, v, o, dO, lse, spd, T)
    gt.gt_check_device_status()
    stats = gt.gt_kernel_stats()
    gt.gt_kernel_stats_reset(False)
    # first-launch order (the forward may balance its work and merge shared
    # tiles; the backward may split its streams, and its last launch converts the
    # fp32 sums and the bucket sums)
    per = gt.launches_per_call("bf16", h, d, n, nb=nb)
    names = [m for m in stats if m != "fwd_merge"]
    assert names == ["fwd_tc", "bwd_prep", "bwd_dq", "bwd_dkdv", "bwd_finish"]
    assert ("fwd_merge" in stats) == (per["fwd"] == 2)
    assert per["bwd"] == 4
    assert sum(c for c, _ in stats.values()) == per["fwd"] + per["bwd"]
    for name, (launches, ms) in stats.items():
        assert launches == 1
        if timing:
            assert 0.0 < ms < 1000.0, (name, ms)
        else:
            assert ms == -1.0


def test_splits_fill_the_last_waves(gt):
    """The dq split on a GB300 (152 SMs, two dq CTAs each): 4096 nodes give 64
    tasks, split 4 ways (256 CTAs, one wave); 16384 nodes give 256 tasks, split
    7 ways (1792 CTAs in six waves); 19456 nodes give 304 tasks, exactly one
    wave, unsplit.  The forward makes no uniform KV split of its own (it
    balances its work instead), and an explicit kv_block is kept."""
    lib = gt.load_library()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert lib.gt_bias_attn_bwd_split(1, 4096, 8, 8, 18) == 4
        assert lib.gt_bias_attn_bwd_split(1, 16384, 8, 16, 26) == 7
        assert lib.gt_bias_attn_bwd_split(1, 19456, 8, 16, 26) == 1
    assert lib.gt_bias_attn_bwd_split(1, 4096, 8, 8, 18) >= 2
    assert lib.gt_bias_attn_fwd_kv_block(1, 4096, 8, 8, 0) == 0
    assert lib.gt_bias_attn_fwd_kv_block(1, 4096, 8, 8, 1024) == 1024
    assert lib.gt_bias_attn_fwd_kv_block(1, 16384, 8, 16, 0) == 0


def test_counts_of_a_graph_past_one_wave(gt):
    """n = 16384 (128 tiles): the balanced forward merges its split tiles, and the
    backward splits the dq tasks and dk/dv groups past their last full wave,
    with one fp32-to-bf16 conversion at the end; the library's own launch count
    matches what ran."""
    n, h, d, nb = 16384, 8, 16, 26
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=6)
    q, k, v, dO = (to_dev(x[a], "bf16") for a in ("q", "k", "v", "dO"))
    T = torch.from_numpy(x["T"]).cuda()
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    spd = torch.randint(0, nb, (n, gt.spd_ld(n)), dtype=torch.int8, device="cuda", generator=g)
    torch.cuda.synchronize()
    gt.gt_kernel_stats_reset(False)
    o, lse = gt.gt_bias_attn_fwd(q, k, v, spd, T)
    gt.gt_bias_attn_bwd(q, k, v, o, dO, lse, spd, T)
    gt.gt_check_device_status()
    stats = gt.gt_kernel_stats()
    gt.gt_kernel_stats_reset(False)
    per = gt.launches_per_call("bf16", h, d, n, nb=nb)
    assert sum(c for c, _ in stats.values()) == per["fwd"] + per["bwd"], (stats, per)
    assert ("fwd_merge" in stats) == (per["fwd"] == 2)
    if gt.load_library().gt_bias_attn_fwd_ctas(1, n, h, d, 0) > 0:
        assert stats["fwd_merge"][0] == 1
