"""GPU parity of the GT encoder layer (gt_layer_fwd / gt_layer_bwd) against the
fp64 layer oracle: every output and gradient within the bf16 tolerance
(relative L2 <= 2e-2 per tensor; the attention runs in bf16)."""
import numpy as np
import pytest
import torch

import gt_inputs as gi
from oracle import layer as L
from oracle import oracle as O

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def gt():
    import graph_transformer_attention_gb300 as m
    from graph_transformer_attention_gb300 import build
    build.build()
    m.load_library()
    return m


def _rel(a, b):
    a = a.detach().float().cpu().numpy().astype(np.float64) if torch.is_tensor(a) else np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a.ravel() - b.ravel()) / max(np.linalg.norm(b.ravel()), 1e-30))


@pytest.mark.parametrize("n,graph,D", [(300, "ba", 6), (1000, "dba", 12), (2049, "er", 5), (1, "empty", 3),
                                       (129, "path", 4), (128, "path", 5), (256, "er", 4), (383, "ba", 5),
                                       (6800, "ba6800", 20)])
def test_layer_forward_and_backward_match_the_oracle(gt, n, graph, D):
    if graph == "empty":
        g = gi.csr_from_edges(n, np.zeros(0, np.int64), np.zeros(0, np.int64))
    elif graph == "path":
        g = gi.csr_from_edges(n, np.arange(n - 1), np.arange(1, n))
    elif graph == "ba":
        g = gi.barabasi_albert(n, 3, seed=21)
    elif graph == "ba6800":
        g = gi.config_graph(gi.CONFIGS[3])      # one layer of the 16-layer workload, full size
    elif graph == "dba":
        g = gi.disjoint_ba(4, n // 4, 2, seed=22)
    else:
        g = gi.erdos_renyi(n, 4.0 / n, seed=23)
    n = g.n
    nb = D + 2
    spd = O.spd(n, g.indptr, g.indices, D)
    p = gi.make_gt_layer_params(64, 64, nb, 8, seed=30 + n)
    io = gi.make_gt_layer_io(n, 64, seed=40 + n)
    dev = torch.device("cuda")
    ld = gt.spd_ld(n)
    spd_d = torch.zeros((n, ld), dtype=torch.int8)
    spd_d[:, :n] = torch.from_numpy(spd)
    spd_d = spd_d.to(dev)
    params = {k: torch.from_numpy(v).to(dev) for k, v in p.items() if k != "T"}
    T = torch.from_numpy(p["T"]).to(dev)
    x = torch.from_numpy(io["x"]).to(dev)
    dy = torch.from_numpy(io["dy"]).to(dev)
    y, saved = gt.gt_layer_fwd(x, params, spd_d, T)
    dx, grads, dT = gt.gt_layer_bwd(x, params, spd_d, T, saved, dy)
    gt.gt_check_device_status()

    fw = L.layer_fwd(io["x"], p, spd, 8)
    gr = L.layer_bwd(io["x"], p, spd, 8, fw, io["dy"])
    errs = {"y": _rel(y, fw["y"]), "q": _rel(saved["q"], fw["q"]), "k": _rel(saved["k"], fw["k"]),
            "v": _rel(saved["v"], fw["v"]), "o": _rel(saved["o"], fw["o"]), "lse": _rel(saved["lse"], fw["lse"]),
            "dx": _rel(dx, gr["x"]), "dT": _rel(dT, gr["T"])}
    for name in L_PARAMS:
        errs["d" + name] = _rel(grads[name], gr[name])
    print(f"layer n={n}: " + ", ".join(f"{k} {v:.1e}" for k, v in errs.items()))
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, f"relative L2 above {TOL}: {bad} (all: {errs})"


L_PARAMS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2")


def test_layer_rejects_unsupported_shapes(gt):
    import ctypes
    lib = gt.load_library()
    fake = ctypes.c_void_p(0x1000)
    assert lib.gt_layer_fwd(100, 4, 8, 64, fake, fake, fake, 112, fake, 8, fake, fake, fake, fake, fake, fake,
                            fake, 1 << 20, None) == -2
    assert lib.gt_layer_workspace_size(100, 8, 16, 64) == 0
