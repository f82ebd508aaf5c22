"""fp64 CPU oracle of one GT encoder layer around the biased attention.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg may import this module; the library itself never does.  It
shares no code with the CUDA path.

The pages fix the model's shape (MegaGraph, Fig. 8: a 16-layer, 8-head GT with
hidden and FFN dimension 64) but not the order of the operations inside a layer.
The plainest reading, the Graphormer encoder layer (a textbook source, named, not
copied), is used, with LayerNorm before each sublayer:

    u = LN1(x)                      LN(v) = g * (v - mean v) / sqrt(var v + eps) + b
    [q | k | v] = u W_qkv + b_qkv   split into heads: [n][h][d], h d = width
    o = A(q, k, v)                  the biased attention (spd buckets, table T)
    hh = x + o W_o + b_o
    z = LN2(hh)
    a = z W_1 + b_1,  g = GELU(a)   GELU(a) = a Phi(a), Phi the normal CDF
    y = hh + g W_2 + b_2

The backward is derived by hand from these definitions, step by step in reverse;
the attention part calls the attention oracle (oracle.attn_fwd / attn_bwd).
Everything is fp64.  Pinned in tests/test_oracle_layer.py against torch
autograd (fp64, CPU, the same layer written with torch's own layer_norm, gelu and
softmax) and against central finite differences.
"""
from __future__ import annotations

import math

import numpy as np

from . import oracle as O

LN_EPS = 1e-5


def _ln_fwd(v, g, b):
    mu = v.mean(axis=1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=1, keepdims=True)
    r = 1.0 / np.sqrt(var + LN_EPS)
    vh = (v - mu) * r
    return vh * g + b, vh, r


def _ln_bwd(dout, vh, r, g):
    """Given d(LN output), the normalised input vh and 1/std r: d(input), dg, db."""
    dvh = dout * g
    c = dvh.shape[1]
    dv = r * (dvh - dvh.sum(axis=1, keepdims=True) / c - vh * (dvh * vh).sum(axis=1, keepdims=True) / c)
    return dv, (dout * vh).sum(axis=0), dout.sum(axis=0)


def _phi_cdf(a):
    return 0.5 * (1.0 + np.vectorize(math.erf)(a / math.sqrt(2.0)))


def _gelu(a):
    return a * _phi_cdf(a)


def _gelu_grad(a):
    return _phi_cdf(a) + a * np.exp(-0.5 * a * a) / math.sqrt(2.0 * math.pi)


def layer_fwd(x, p, spd_mat, heads: int, nthreads=None) -> dict:
    """Forward of one layer; returns y and the intermediates the backward uses."""
    x = np.asarray(x, np.float64)
    P = {k: np.asarray(v, np.float64) for k, v in p.items()}
    n, c = x.shape
    d = c // heads
    u, uh, r1 = _ln_fwd(x, P["ln1_g"], P["ln1_b"])
    qkv = u @ P["w_qkv"] + P["b_qkv"]
    q, k, v = (qkv[:, i * c:(i + 1) * c].reshape(n, heads, d) for i in range(3))
    o, lse = O.attn_fwd(q, k, v, spd_mat, P["T"], nthreads=nthreads)
    o2 = o.reshape(n, c)
    hh = x + o2 @ P["w_o"] + P["b_o"]
    z, zh, r2 = _ln_fwd(hh, P["ln2_g"], P["ln2_b"])
    a = z @ P["w_1"] + P["b_1"]
    g = _gelu(a)
    y = hh + g @ P["w_2"] + P["b_2"]
    return dict(y=y, u=u, uh=uh, r1=r1, q=q, k=k, v=v, o=o, lse=lse, hh=hh, z=z, zh=zh, r2=r2, a=a, g=g)


def layer_bwd(x, p, spd_mat, heads: int, fw: dict, dy, nthreads=None) -> dict:
    """Backward of one layer given the forward's intermediates and dL/dy."""
    P = {k: np.asarray(v, np.float64) for k, v in p.items()}
    dy = np.asarray(dy, np.float64)
    n, c = dy.shape
    d = c // heads
    gr = {}
    # y = hh + g W_2 + b_2
    gr["w_2"] = fw["g"].T @ dy
    gr["b_2"] = dy.sum(axis=0)
    dg = dy @ P["w_2"].T
    da = dg * _gelu_grad(fw["a"])
    gr["w_1"] = fw["z"].T @ da
    gr["b_1"] = da.sum(axis=0)
    dz = da @ P["w_1"].T
    dhh_ln, gr["ln2_g"], gr["ln2_b"] = _ln_bwd(dz, fw["zh"], fw["r2"], P["ln2_g"])
    dhh = dy + dhh_ln
    # hh = x + o W_o + b_o
    o2 = fw["o"].reshape(n, c)
    gr["w_o"] = o2.T @ dhh
    gr["b_o"] = dhh.sum(axis=0)
    do = (dhh @ P["w_o"].T).reshape(n, heads, d)
    Dv = O.bwd_delta(fw["o"], do)
    ga = O.attn_bwd(fw["q"], fw["k"], fw["v"], do, spd_mat, P["T"], fw["lse"], Dv, nthreads=nthreads)
    gr["T"] = ga["dT"]
    dqkv = np.concatenate([ga["dq"].reshape(n, c), ga["dk"].reshape(n, c), ga["dv"].reshape(n, c)], axis=1)
    gr["w_qkv"] = fw["u"].T @ dqkv
    gr["b_qkv"] = dqkv.sum(axis=0)
    du = dqkv @ P["w_qkv"].T
    dx_ln, gr["ln1_g"], gr["ln1_b"] = _ln_bwd(du, fw["uh"], fw["r1"], P["ln1_g"])
    gr["x"] = dhh + dx_ln
    gr["do"] = do
    return gr
