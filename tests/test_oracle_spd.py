"""Pins for the oracle's clipped shortest-path buckets (CPU only).

The SPD code of a pair is min(dist(i,j), D) for reachable pairs and D+1 for
unreachable ones (MegaGraph abstract: topology-aware bias; the bucket rule is
Graphormer's spatial encoding).  Each pin below is independent of the oracle's
breadth-first search: Floyd-Warshall on tiny graphs, scipy's csgraph routine,
closed forms of textbook graphs, and structural invariants.
"""
import os

import numpy as np
import pytest

import gt_inputs as gi
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _codes_from_dist(dist: np.ndarray, D: int) -> np.ndarray:
    out = np.where(np.isfinite(dist), np.minimum(dist, D), D + 1)
    return out.astype(np.int8)


def _floyd_warshall(g: gi.Graph) -> np.ndarray:
    n = g.n
    dist = np.full((n, n), np.inf)
    np.fill_diagonal(dist, 0.0)
    for u in range(n):
        for e in range(g.indptr[u], g.indptr[u + 1]):
            dist[u, g.indices[e]] = 1.0
    for k in range(n):
        dist = np.minimum(dist, dist[:, k:k + 1] + dist[k:k + 1, :])
    return dist


@pytest.mark.parametrize("seed", range(12))
def test_spd_matches_floyd_warshall(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 65))
    p = float(rng.choice([0.0, 0.02, 0.05, 0.1, 0.3, 1.0]))
    g = gi.erdos_renyi(n, p, seed=100 + seed)
    D = int(rng.choice([1, 2, 3, 5, 16, 126]))
    ref = _codes_from_dist(_floyd_warshall(g), D)
    got = O.spd(g.n, g.indptr, g.indices, D)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("cfg", [1, 2])
def test_spd_matches_scipy_on_configs(cfg):
    from scipy.sparse import csr_matrix
    from scipy.sparse.csgraph import shortest_path
    w = gi.CONFIGS[cfg]
    g = gi.config_graph(w)
    A = csr_matrix((np.ones(g.nnz), g.indices, g.indptr), shape=(g.n, g.n))
    dist = shortest_path(A, directed=False, unweighted=True)
    ref = _codes_from_dist(dist, w.D)
    got = O.spd(g.n, g.indptr, g.indices, w.D)
    assert np.array_equal(got, ref)


def test_spd_scipy_disjoint_ba_prefix():
    """First 8 components of the 64-component workload: cross-component pairs are D+1."""
    from scipy.sparse import csr_matrix
    from scipy.sparse.csgraph import shortest_path
    g = gi.disjoint_ba(8, 256, 3, seed=7)
    A = csr_matrix((np.ones(g.nnz), g.indices, g.indptr), shape=(g.n, g.n))
    ref = _codes_from_dist(shortest_path(A, directed=False, unweighted=True), 24)
    got = O.spd(g.n, g.indptr, g.indices, 24)
    assert np.array_equal(got, ref)
    comp = np.arange(g.n) // 256
    assert np.all(got[comp[:, None] != comp[None, :]] == 25)


def _grid(rows, cols):
    idx = np.arange(rows * cols).reshape(rows, cols)
    u = np.concatenate([idx[:, :-1].ravel(), idx[:-1, :].ravel()])
    v = np.concatenate([idx[:, 1:].ravel(), idx[1:, :].ravel()])
    return gi.csr_from_edges(rows * cols, u, v)


@pytest.mark.parametrize("n,D", [(1, 4), (2, 1), (17, 5), (40, 100)])
def test_spd_closed_form_path(n, D):
    g = gi.csr_from_edges(n, np.arange(n - 1), np.arange(1, n))
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    assert np.array_equal(O.spd(n, g.indptr, g.indices, D), np.minimum(abs(i - j), D))


@pytest.mark.parametrize("n,D", [(3, 4), (10, 3), (31, 20)])
def test_spd_closed_form_cycle(n, D):
    g = gi.csr_from_edges(n, np.arange(n), (np.arange(n) + 1) % n)
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    a = abs(i - j)
    assert np.array_equal(O.spd(n, g.indptr, g.indices, D), np.minimum(np.minimum(a, n - a), D))


def test_spd_closed_form_complete_star_empty_grid():
    n = 9
    iu, ju = np.triu_indices(n, 1)
    g = gi.csr_from_edges(n, iu, ju)
    expect = np.ones((n, n), np.int8); np.fill_diagonal(expect, 0)
    assert np.array_equal(O.spd(n, g.indptr, g.indices, 16), expect)

    star = gi.csr_from_edges(n, np.zeros(n - 1, np.int64), np.arange(1, n))
    expect = np.full((n, n), 2, np.int8); expect[0, :] = 1; expect[:, 0] = 1
    np.fill_diagonal(expect, 0)
    assert np.array_equal(O.spd(n, star.indptr, star.indices, 16), expect)

    empty = gi.csr_from_edges(n, np.zeros(0, np.int64), np.zeros(0, np.int64))
    expect = np.full((n, n), 17, np.int8); np.fill_diagonal(expect, 0)
    assert np.array_equal(O.spd(n, empty.indptr, empty.indices, 16), expect)

    r, c = 5, 7
    grid = _grid(r, c)
    y, x = np.divmod(np.arange(r * c), c)
    man = abs(y[:, None] - y[None, :]) + abs(x[:, None] - x[None, :])
    assert np.array_equal(O.spd(r * c, grid.indptr, grid.indices, 4), np.minimum(man, 4))


def test_spd_disjoint_union_unreachable():
    a = gi.csr_from_edges(6, np.arange(5), np.arange(1, 6))           # path on 0..5
    u = np.concatenate([np.arange(5), 6 + np.arange(3)])
    v = np.concatenate([np.arange(1, 6), 6 + (np.arange(3) + 1) % 3])  # plus a triangle
    g = gi.csr_from_edges(9, u, v)
    got = O.spd(9, g.indptr, g.indices, 3)
    assert np.all(got[:6, 6:] == 4) and np.all(got[6:, :6] == 4)
    ref_path = O.spd(6, a.indptr, a.indices, 3)
    assert np.array_equal(got[:6, :6], ref_path)
    tri = np.ones((3, 3), np.int8); np.fill_diagonal(tri, 0)
    assert np.array_equal(got[6:, 6:], tri)


@pytest.mark.parametrize("cfg", [1, 3])
def test_spd_invariants(cfg):
    w = gi.CONFIGS[cfg]
    g = gi.config_graph(w)
    big_D = 126
    s = O.spd(g.n, g.indptr, g.indices, big_D).astype(np.int32)
    assert np.array_equal(s, s.T)
    assert np.all(np.diag(s) == 0)
    adj = np.zeros((g.n, g.n), bool)
    rows = np.repeat(np.arange(g.n), np.diff(g.indptr))
    adj[rows, g.indices] = True
    assert np.array_equal(s == 1, adj)
    # along an edge (u,v) the distance to any target changes by at most one
    reach = s <= big_D
    su, sv = s[rows], s[g.indices]
    both = reach[rows] & reach[g.indices]
    assert np.all(np.abs(su - sv)[both] <= 1)
    # clipping at the workload's D is a pure min() of the unclipped distances
    clipped = O.spd(g.n, g.indptr, g.indices, w.D).astype(np.int32)
    assert np.array_equal(clipped, np.where(s <= big_D, np.minimum(s, w.D), w.D + 1))


def test_spd_golden_fixture():
    """Hand-worked 8-node graph (two components) in tests/golden/spd_two_components.txt."""
    path = os.path.join(GOLDEN, "spd_two_components.txt")
    lines = [ln for ln in open(path) if ln.strip() and not ln.startswith("#")]
    n, D = map(int, lines[0].split())
    edges = np.array([list(map(int, ln.split())) for ln in lines[1:] if len(ln.split()) == 2])
    mat = np.array([list(map(int, ln.split())) for ln in lines[1:] if len(ln.split()) == n])
    g = gi.csr_from_edges(n, edges[:, 0], edges[:, 1])
    assert np.array_equal(O.spd(n, g.indptr, g.indices, D), mat.astype(np.int8))
