"""Seeded synthetic inputs for biased graph attention.

This module only draws random graphs and random tensors.  It holds none of the
attention or shortest-path arithmetic: both the CPU oracle (``oracle/``) and the
CUDA library consume what it returns, and neither is imported from here.

Graphs come back as an undirected simple graph in CSR form with both directions
stored (``indptr`` int64[N+1], ``indices`` int32[nnz], neighbours sorted, no
self-loops, no multi-edges).

The five workloads follow the MegaGraph paper's GT shape (Fig. 8: 16 layers,
8 heads, hidden 64; batch of 6800 nodes) and its blockwise KV streaming (Fig. 4).
The paper names no dataset, so every graph here is a seeded random graph of a
textbook family; the recipe of each is in ``CONFIGS``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Graph", "Workload", "CONFIGS", "make_graph", "make_layer_tensors",
    "erdos_renyi", "random_geometric", "barabasi_albert", "disjoint_ba",
    "configuration_model", "csr_from_edges", "round_to_bf16", "make_gt_layer_params",
    "make_gt_layer_io",
]


@dataclass
class Graph:
    n: int
    indptr: np.ndarray   # int64 [n+1]
    indices: np.ndarray  # int32 [nnz]

    @property
    def nnz(self) -> int:
        return int(self.indices.shape[0])


def csr_from_edges(n: int, u: np.ndarray, v: np.ndarray) -> Graph:
    """Symmetric CSR of the simple undirected graph with edges (u[k], v[k])."""
    u = np.asarray(u, dtype=np.int64).ravel()
    v = np.asarray(v, dtype=np.int64).ravel()
    keep = u != v
    u, v = u[keep], v[keep]
    a = np.concatenate([u, v])
    b = np.concatenate([v, u])
    if a.size:
        key = np.unique(a * n + b)
        a, b = key // n, key % n
    indptr = np.zeros(n + 1, dtype=np.int64)
    np.add.at(indptr, a + 1, 1)
    np.cumsum(indptr, out=indptr)
    return Graph(n, indptr, b.astype(np.int32))


def erdos_renyi(n: int, p: float, seed: int) -> Graph:
    """G(n, p): each unordered pair i<j is an edge with probability p."""
    rng = np.random.Generator(np.random.PCG64(seed))
    iu, ju = np.triu_indices(n, 1)
    hit = rng.random(iu.shape[0]) < p
    return csr_from_edges(n, iu[hit], ju[hit])


def random_geometric(n: int, radius: float, seed: int) -> Graph:
    """Points uniform in the unit square (no torus); edge iff distance < radius."""
    rng = np.random.Generator(np.random.PCG64(seed))
    pos = rng.random((n, 2))
    us, vs = [], []
    step = 512
    for s in range(0, n, step):
        blk = pos[s:s + step]
        d2 = ((blk[:, None, :] - pos[None, :, :]) ** 2).sum(-1)
        ii, jj = np.nonzero(d2 < radius * radius)
        ii = ii + s
        keep = ii < jj
        us.append(ii[keep]); vs.append(jj[keep])
    return csr_from_edges(n, np.concatenate(us), np.concatenate(vs))


def _ba_edges(n: int, m: int, rng: np.random.Generator, offset: int = 0):
    """Barabasi-Albert growth: a star on m+1 nodes, then each new node attaches
    to m distinct existing nodes chosen with probability proportional to degree."""
    us, vs = [], []
    rep = []  # every edge endpoint once: sampling from it is degree-proportional
    for t in range(1, m + 1):
        us.append(0); vs.append(t)
        rep += [0, t]
    for v in range(m + 1, n):
        targets = set()
        while len(targets) < m:
            targets.add(rep[int(rng.integers(len(rep)))])
        for t in sorted(targets):
            us.append(v); vs.append(t)
            rep += [v, t]
    return np.asarray(us, np.int64) + offset, np.asarray(vs, np.int64) + offset


def barabasi_albert(n: int, m: int, seed: int) -> Graph:
    rng = np.random.Generator(np.random.PCG64(seed))
    u, v = _ba_edges(n, m, rng)
    return csr_from_edges(n, u, v)


def disjoint_ba(n_comp: int, comp_size: int, m: int, seed: int) -> Graph:
    """Disjoint union of BA graphs; component c holds node ids [c*size, (c+1)*size)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    us, vs = [], []
    for c in range(n_comp):
        u, v = _ba_edges(comp_size, m, rng, offset=c * comp_size)
        us.append(u); vs.append(v)
    return csr_from_edges(n_comp * comp_size, np.concatenate(us), np.concatenate(vs))


def configuration_model(n: int, gamma: float, kmin: int, kmax: int, seed: int) -> Graph:
    """Degrees k in [kmin, kmax] with P(k) ~ k^-gamma; the last node's degree is
    redrawn until the degree sum is even; stubs are matched by a random
    permutation; self-loops and multi-edges are dropped afterwards."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ks = np.arange(kmin, kmax + 1)
    pk = ks.astype(np.float64) ** (-gamma)
    pk /= pk.sum()
    deg = rng.choice(ks, size=n, p=pk)
    while int(deg.sum()) % 2:
        deg[-1] = rng.choice(ks, p=pk)
    stubs = np.repeat(np.arange(n, dtype=np.int64), deg)
    rng.shuffle(stubs)
    pairs = stubs.reshape(-1, 2)
    return csr_from_edges(n, pairs[:, 0], pairs[:, 1])


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(x)
    out = (rounded & 0xFFFFFFFF).astype(np.uint32).view(np.float32).copy()
    out[nan] = np.nan
    return out


@dataclass
class Workload:
    index: int
    name: str
    n: int
    heads: int
    head_dim: int
    dtype: str          # "f32" or "bf16"
    D: int              # SPD clip; buckets 0..D, plus D+1 for unreachable
    layers: int = 1
    kv_block: int = 0   # 0: one pass over all KV columns
    graph_kind: str = ""
    graph_args: dict = field(default_factory=dict)

    @property
    def nb(self) -> int:
        return self.D + 2

    @property
    def graph_seed(self) -> int:
        return 1000 + self.index

    def tensor_seed(self, layer: int) -> int:
        return 2000 + 100 * self.index + layer


CONFIGS = {
    1: Workload(1, "er512", 512, 8, 8, "f32", 16, graph_kind="er",
                graph_args=dict(p=8.0 / 511.0)),
    2: Workload(2, "rgg4096", 4096, 8, 8, "bf16", 16, graph_kind="rgg",
                graph_args=dict(radius=math.sqrt(10.0 / (math.pi * 4095.0)))),
    3: Workload(3, "ba6800x16", 6800, 8, 8, "bf16", 20, layers=16, graph_kind="ba",
                graph_args=dict(m=4)),
    4: Workload(4, "ba64x256", 16384, 8, 16, "bf16", 24, graph_kind="dba",
                graph_args=dict(n_comp=64, comp_size=256, m=3)),
    5: Workload(5, "cm32768", 32768, 8, 8, "bf16", 32, kv_block=4096, graph_kind="cm",
                graph_args=dict(gamma=2.1, kmin=2, kmax=2000)),
}


def make_graph(kind: str, n: int, seed: int, **args) -> Graph:
    if kind == "er":
        return erdos_renyi(n, args["p"], seed)
    if kind == "rgg":
        return random_geometric(n, args["radius"], seed)
    if kind == "ba":
        return barabasi_albert(n, args["m"], seed)
    if kind == "dba":
        g = disjoint_ba(args["n_comp"], args["comp_size"], args["m"], seed)
        assert g.n == n
        return g
    if kind == "cm":
        return configuration_model(n, args["gamma"], args["kmin"], args["kmax"], seed)
    raise ValueError(f"unknown graph kind {kind!r}")


def config_graph(cfg: Workload) -> Graph:
    return make_graph(cfg.graph_kind, cfg.n, cfg.graph_seed, **cfg.graph_args)


def make_layer_tensors(n: int, heads: int, head_dim: int, nb: int, dtype: str, seed: int,
                       t_std: float = 0.1) -> dict:
    """Q, K, V, T, dO drawn in that order from PCG64(seed).

    Q, K, V, dO ~ N(0,1) of shape [n][heads][head_dim]; T ~ N(0, t_std^2) of shape
    [heads][nb].  For dtype "bf16" Q, K, V and dO are rounded to bfloat16 (the
    arrays stay float32 but hold bf16 values exactly); T is always float32.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    shp = (n, heads, head_dim)
    q = rng.standard_normal(shp, dtype=np.float32)
    k = rng.standard_normal(shp, dtype=np.float32)
    v = rng.standard_normal(shp, dtype=np.float32)
    t = (t_std * rng.standard_normal((heads, nb))).astype(np.float32)
    do = rng.standard_normal(shp, dtype=np.float32)
    if dtype == "bf16":
        q, k, v, do = (round_to_bf16(a) for a in (q, k, v, do))
    elif dtype != "f32":
        raise ValueError(dtype)
    return dict(q=q, k=k, v=v, T=t, dO=do)


def config_layer_tensors(cfg: Workload, layer: int = 0) -> dict:
    return make_layer_tensors(cfg.n, cfg.heads, cfg.head_dim, cfg.nb, cfg.dtype,
                              cfg.tensor_seed(layer))


def make_gt_layer_params(width: int, ffn: int, nb: int, heads: int, seed: int) -> dict:
    """Weights of one GT encoder layer around the biased attention, drawn from
    PCG64(seed) in this order: LayerNorm 1 (gain, shift), W_qkv, b_qkv, W_o, b_o,
    LayerNorm 2, W_1, b_1, W_2, b_2, T.  Matrices ~ N(0, 1/fan_in) (a unit-variance
    input keeps a unit-variance output), biases and shifts ~ N(0, 0.02^2), gains
    ~ 1 + N(0, 0.1^2), T ~ N(0, 0.1^2).  All float32.  W_qkv is [width][3 width]
    (columns: q | k | v, each in (head, channel) order), W_o [width][width],
    W_1 [width][ffn], W_2 [ffn][width]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    f32 = np.float32

    def mat(r, c):
        return (rng.standard_normal((r, c)) / math.sqrt(r)).astype(f32)

    def vec(m, std=0.02):
        return (std * rng.standard_normal(m)).astype(f32)

    p = {}
    p["ln1_g"] = (1.0 + vec(width, 0.1)).astype(f32)
    p["ln1_b"] = vec(width)
    p["w_qkv"] = mat(width, 3 * width)
    p["b_qkv"] = vec(3 * width)
    p["w_o"] = mat(width, width)
    p["b_o"] = vec(width)
    p["ln2_g"] = (1.0 + vec(width, 0.1)).astype(f32)
    p["ln2_b"] = vec(width)
    p["w_1"] = mat(width, ffn)
    p["b_1"] = vec(ffn)
    p["w_2"] = mat(ffn, width)
    p["b_2"] = vec(width)
    p["T"] = (0.1 * rng.standard_normal((heads, nb))).astype(f32)
    return p


def make_gt_layer_io(n: int, width: int, seed: int) -> dict:
    """Layer input x and the gradient dy of the layer output, both N(0, 1)
    float32 [n][width], drawn from PCG64(seed) in that order."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n, width), dtype=np.float32)
    dy = rng.standard_normal((n, width), dtype=np.float32)
    return dict(x=x, dy=dy)
