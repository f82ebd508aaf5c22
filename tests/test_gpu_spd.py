"""GPU parity of gt_spd_build against the CPU oracle: bit-exact bucket codes."""
import numpy as np
import pytest
import torch

import gt_inputs as gi
from oracle import oracle as O
from tests.helpers import graph_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gt():
    import graph_transformer_attention_gb300 as m
    from graph_transformer_attention_gb300 import build
    build.build()
    m.load_library()
    return m


ALGOS = [0, 1, 2, 3, 4]     # auto, scan32, scan16, queue32, global64


def _gpu_spd(gt, g, D, algo=0):
    ip, ix = graph_to_dev(g)
    out = gt.gt_spd_build(ip, ix, g.n, D, algo=algo)
    gt.gt_check_device_status()
    return out[:, :g.n].cpu().numpy()


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_spd_full_config(gt, cfg):
    w = gi.CONFIGS[cfg]
    g = gi.config_graph(w)
    got = _gpu_spd(gt, g, w.D)
    ref = O.spd(g.n, g.indptr, g.indices, w.D)
    assert np.array_equal(got, ref), f"config {cfg}: {int((got != ref).sum())} codes differ"


def _path(n):
    return gi.csr_from_edges(n, np.arange(n - 1), np.arange(1, n))


def _empty(n):
    return gi.csr_from_edges(n, np.zeros(0, np.int64), np.zeros(0, np.int64))


@pytest.mark.parametrize("name,g,D", [
    ("n1", _empty(1), 3),
    ("n2_edge", gi.csr_from_edges(2, [0], [1]), 1),
    ("n2_none", _empty(2), 5),
    ("empty_77", _empty(77), 16),
    ("path_300_D5", _path(300), 5),
    ("path_1000_D126", _path(1000), 126),
    ("path_129_D1", _path(129), 1),
    ("complete_65", gi.csr_from_edges(65, *np.triu_indices(65, 1)), 16),
    ("star_200", gi.csr_from_edges(200, np.zeros(199, np.int64), np.arange(1, 200)), 2),
    ("er_333", gi.erdos_renyi(333, 0.004, seed=5), 7),
    ("dba_5x70", gi.disjoint_ba(5, 70, 2, seed=3), 24),
    ("ba_1000_tree", gi.barabasi_albert(1000, 1, seed=9), 32),
])
@pytest.mark.parametrize("algo", ALGOS)
def test_spd_edge_cases(gt, name, g, D, algo):
    got = _gpu_spd(gt, g, D, algo)
    ref = O.spd(g.n, g.indptr, g.indices, D)
    assert np.array_equal(got, ref), f"{name}, algo {algo}: {int((got != ref).sum())} codes differ"


@pytest.mark.parametrize("name,g,D", [
    ("cm_3001", gi.configuration_model(3001, 2.1, 2, 300, seed=11), 32),
    ("rgg_2500", gi.random_geometric(2500, 0.03, seed=12), 16),
    ("dba_9x333", gi.disjoint_ba(9, 333, 3, seed=13), 24),
    ("ba_4095", gi.barabasi_albert(4095, 4, seed=14), 20),
])
@pytest.mark.parametrize("algo", ALGOS)
def test_spd_every_algorithm_mid_size(gt, name, g, D, algo):
    """Every search algorithm on graphs of a few thousand vertices (several
    batches per CTA, blocks of hubs and of leaves, odd n for the packed words)."""
    got = _gpu_spd(gt, g, D, algo)
    ref = O.spd(g.n, g.indptr, g.indices, D)
    assert np.array_equal(got, ref), f"{name}, algo {algo}: {int((got != ref).sum())} codes differ"


def test_spd_algorithm_limits(gt):
    """Each algorithm takes the sizes it documents; asking for more is refused."""
    assert gt.gt_spd_workspace_size(18000, 10, 8, algo=1) > 0
    assert gt.gt_spd_workspace_size(20000, 10, 8, algo=1) == 0
    assert gt.gt_spd_workspace_size(36000, 10, 8, algo=2) > 0
    assert gt.gt_spd_workspace_size(40000, 10, 8, algo=2) == 0
    assert gt.gt_spd_workspace_size(1 << 20, 10, 8, algo=4) > 0
    g = _path(300)
    ip, ix = graph_to_dev(g)
    with pytest.raises(gt.GtError):
        gt.gt_spd_build(ip, ix, 20000, 8, algo=1)


def test_spd_tolerates_self_loops_and_repeats(gt):
    g = gi.erdos_renyi(150, 0.03, seed=1)
    # rebuild the CSR with a self-loop on every vertex and every edge twice
    rows = np.repeat(np.arange(g.n), np.diff(g.indptr))
    cols = g.indices.astype(np.int64)
    r2 = np.concatenate([rows, rows, np.arange(g.n)])
    c2 = np.concatenate([cols, cols, np.arange(g.n)])
    order = np.lexsort((c2, r2))
    r2, c2 = r2[order], c2[order]
    indptr = np.zeros(g.n + 1, np.int64)
    np.add.at(indptr, r2 + 1, 1)
    indptr = np.cumsum(indptr)
    messy = gi.Graph(g.n, indptr, c2.astype(np.int32))
    got = _gpu_spd(gt, messy, 9)
    assert np.array_equal(got, O.spd(g.n, g.indptr, g.indices, 9))


@pytest.mark.parametrize("n", [100, 77])
def test_spd_respects_row_stride(gt, n):
    g = gi.erdos_renyi(n, 0.05, seed=2)
    ip, ix = graph_to_dev(g)
    out = torch.full((n, 144), 77, dtype=torch.int8, device="cuda")
    gt.gt_spd_build(ip, ix, g.n, 6, out=out)
    gt.gt_check_device_status()
    got = out.cpu().numpy()
    assert np.array_equal(got[:, :n], O.spd(g.n, g.indptr, g.indices, 6))
    assert np.all(got[:, n:] == 77)   # columns n..ld-1 are left alone


def test_spd_repeat_calls_reuse_workspace(gt):
    g = gi.barabasi_albert(500, 2, seed=4)
    ip, ix = graph_to_dev(g)
    ws = torch.empty(gt.gt_spd_workspace_size(g.n, g.nnz, 12), dtype=torch.uint8, device="cuda")
    a = gt.gt_spd_build(ip, ix, g.n, 12, workspace=ws)
    b = gt.gt_spd_build(ip, ix, g.n, 12, workspace=ws)
    gt.gt_check_device_status()
    assert torch.equal(a[:, :g.n], b[:, :g.n])      # columns >= n are padding
    assert np.array_equal(a[:, :g.n].cpu().numpy(), O.spd(g.n, g.indptr, g.indices, 12))
