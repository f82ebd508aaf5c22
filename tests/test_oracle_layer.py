"""Pins for the oracle of the GT encoder layer around the biased attention (CPU).

The layer (pre-LayerNorm encoder layer, GELU FFN; widths from MegaGraph Fig. 8):
    u = LN1(x); [q|k|v] = u W_qkv + b; o = A(q, k, v); hh = x + o W_o + b_o;
    y = hh + GELU(LN2(hh) W_1 + b_1) W_2 + b_2
Independent pins: torch autograd in fp64 through the same layer written with
torch's own layer_norm, gelu and softmax (the attention bias gathered from T by
indexing, so autograd gives dT), and central finite differences of the oracle's
own forward for single entries of every parameter group.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import gt_inputs as gi
from oracle import layer as L
from oracle import oracle as O

H, D, C, FF, NB = 8, 8, 64, 64, 9


@pytest.fixture(scope="module", autouse=True)
def _built():
    O.build()


def _case(n, seed):
    p = gi.make_gt_layer_params(C, FF, NB, H, seed)
    io = gi.make_gt_layer_io(n, C, seed + 1)
    rng = np.random.default_rng(seed + 2)
    spd = rng.integers(0, NB, size=(n, n)).astype(np.int8)      # not symmetric on purpose
    return p, io["x"].astype(np.float64), io["dy"].astype(np.float64), spd


def _torch_layer(p, x, spd):
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    n = x.shape[0]
    u = F.layer_norm(xt, (C,), t["ln1_g"], t["ln1_b"], eps=L.LN_EPS)
    qkv = u @ t["w_qkv"] + t["b_qkv"]
    q, k, v = (qkv[:, i * C:(i + 1) * C].reshape(n, H, D).transpose(0, 1) for i in range(3))
    bias = t["T"][:, torch.tensor(spd, dtype=torch.long)]                 # [H][n][n]
    s = q @ k.transpose(1, 2) / np.sqrt(D) + bias
    o = (torch.softmax(s, dim=-1) @ v).transpose(0, 1).reshape(n, C)
    hh = xt + o @ t["w_o"] + t["b_o"]
    z = F.layer_norm(hh, (C,), t["ln2_g"], t["ln2_b"], eps=L.LN_EPS)
    y = hh + F.gelu(z @ t["w_1"] + t["b_1"], approximate="none") @ t["w_2"] + t["b_2"]
    return y, t, xt


def test_layer_matches_torch_autograd():
    p, x, dy, spd = _case(37, seed=5)
    fw = L.layer_fwd(x, p, spd, H)
    gr = L.layer_bwd(x, p, spd, H, fw, dy)
    y, t, xt = _torch_layer(p, x, spd)
    assert np.allclose(fw["y"], y.detach().numpy(), rtol=1e-12, atol=1e-12)
    y.backward(torch.tensor(dy))
    for k, v in t.items():
        assert np.allclose(gr[k], v.grad.numpy(), rtol=1e-9, atol=1e-11), k
    assert np.allclose(gr["x"], xt.grad.numpy(), rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("name,idx", [("w_qkv", (3, 70)), ("w_qkv", (10, 140)), ("b_qkv", (5,)),
                                      ("w_o", (7, 9)), ("ln1_g", (4,)), ("ln1_b", (11,)),
                                      ("ln2_g", (2,)), ("w_1", (6, 13)), ("b_1", (8,)),
                                      ("w_2", (1, 50)), ("b_2", (20,)), ("T", (3, 4)), ("x", (5, 17))])
def test_layer_gradients_match_finite_differences(name, idx):
    p, x, dy, spd = _case(12, seed=9)
    fw = L.layer_fwd(x, p, spd, H)
    gr = L.layer_bwd(x, p, spd, H, fw, dy)
    eps = 1e-6

    def loss(pp, xx):
        return float((L.layer_fwd(xx, pp, spd, H)["y"] * dy).sum())

    pp = {k: np.asarray(v, np.float64).copy() for k, v in p.items()}
    xx = x.copy()
    tgt = xx if name == "x" else pp[name]
    old = tgt[idx]
    tgt[idx] = old + eps
    lp = loss(pp, xx)
    tgt[idx] = old - eps
    lm = loss(pp, xx)
    tgt[idx] = old
    fd = (lp - lm) / (2 * eps)
    assert abs(gr[name][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (gr[name][idx], fd)


def test_identity_attention_sublayer_when_w_o_is_zero():
    """W_o = 0 and b_o = 0 remove the attention sublayer: hh = x, and the
    attention receives no gradient (dT, dW_qkv vanish)."""
    p, x, dy, spd = _case(10, seed=3)
    p = dict(p)
    p["w_o"] = np.zeros_like(p["w_o"])
    p["b_o"] = np.zeros_like(p["b_o"])
    fw = L.layer_fwd(x, p, spd, H)
    assert np.allclose(fw["hh"], x)
    gr = L.layer_bwd(x, p, spd, H, fw, dy)
    assert np.abs(gr["T"]).max() == 0.0 and np.abs(gr["w_qkv"]).max() == 0.0
