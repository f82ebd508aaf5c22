"""Peak device memory of a forward + backward, measured, against the model.

blockwise: this library through its Python binding; the model predicts the
peak of the bytes requested from torch's allocator exactly (its
`requested_bytes` statistic: tensor sizes before the allocator rounds them).
materialised: the plain N x N computation in eager torch must hold at least the
model's `peak_min`."""
import math

import numpy as np
import pytest
import torch

from graph_transformer_attention_gb300 import memory as M

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gt():
    import graph_transformer_attention_gb300 as m
    from graph_transformer_attention_gb300 import build
    build.build()
    m.load_library()
    return m


def _requested():
    st = torch.cuda.memory_stats()
    return st["requested_bytes.all.current"], st["requested_bytes.all.peak"]


def _inputs(n, h, d, nb, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    dev = torch.device("cuda")
    q, k, v, dO = (torch.randn((n, h, d), generator=g, dtype=torch.float32).to(dtype).to(dev) for _ in range(4))
    T = (0.1 * torch.randn((h, nb), generator=g, dtype=torch.float32)).to(dev)
    ld = (n + 15) // 16 * 16
    spd = torch.randint(0, nb, (n, ld), generator=g, dtype=torch.int8).to(dev)
    return q, k, v, dO, T, spd


def _measure_blockwise(n, d, dtype, kv_block, out):
    """In a fresh process (so no earlier test's allocator state can show up in the
    window): the peak of the requested bytes during one forward + backward."""
    import graph_transformer_attention_gb300 as m
    m.load_library()
    h, nb = 8, 18
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v, dO, T, spd = _inputs(n, h, d, nb, tdt, seed=n + d)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before, _ = _requested()
    o, lse = m.gt_bias_attn_fwd(q, k, v, spd, T, kv_block=kv_block)
    dq, dk, dv, dT = m.gt_bias_attn_bwd(q, k, v, o, dO, lse, spd, T)
    m.gt_check_device_status()
    out["measured"] = _requested()[1] - before


@pytest.mark.parametrize("n,d,dtype,kv_block", [(4096, 8, "bf16", 0), (6000, 16, "bf16", 0),
                                                (8192, 8, "bf16", 2048), (1000, 8, "f32", 0)])
def test_blockwise_peak_matches_the_model(gt, n, d, dtype, kv_block):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        p = ctx.Process(target=_measure_blockwise, args=(n, d, dtype, kv_block, out))
        p.start()
        p.join(300)
        assert p.exitcode == 0
        measured = out["measured"]
    model = M.blockwise_layer_bytes(n, 8, d, 18, dtype, kv_block)
    predicted = model["peak"] - model["base"]            # the inputs were live before
    assert measured == predicted, (measured, predicted)


def test_materialised_peak_is_at_least_the_model(gt):
    n, h, d, nb = 1024, 8, 8, 18
    q, k, v, dO, T, spd = _inputs(n, h, d, nb, torch.float32, seed=7)
    dev = q.device
    qh, kh, vh = (x.permute(1, 0, 2).contiguous().requires_grad_(True) for x in (q, k, v))
    Tg = T.clone().requires_grad_(True)
    idx = spd[:, :n].long()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before, _ = _requested()
    S = (qh @ kh.transpose(1, 2)) * (1.0 / math.sqrt(d)) + Tg[:, idx]
    P = torch.softmax(S, dim=-1)
    del S
    O = P @ vh
    O.backward(dO.permute(1, 0, 2))
    torch.cuda.synchronize()
    measured = _requested()[1] - before
    model = M.materialised_layer_bytes(n, h, d, "f32")
    per_head_nn = model["peak_min"] - model["dense"]
    assert measured >= per_head_nn, (measured, per_head_nn)
    # and the blockwise form of the same layer needs a small fraction of it
    blk = M.blockwise_layer_bytes(n, h, d, nb, "f32")
    assert blk["peak"] - blk["base"] < measured / 10
