"""Pins for the oracle's biased attention forward and backward (CPU only).

Definition pinned (MegaGraph abstract and Fig. 4; Graphormer spatial bias):
    s_ij = scale <q_i,k_j> + T[h][spd_ij],  o_i = softmax_j(s_i) V,  lse_i = logsumexp_j s_ij
and its gradients dq, dk, dv, dT for an upstream dO.

Independent pins: torch's scaled_dot_product_attention (fp64, CPU) with the
bias materialised as a float mask; torch autograd through that graph, with T
gathered by indexing so autograd yields dT; torch.logsumexp on the materialised
scores; central finite differences of the oracle's own forward; closed forms.
Bucket matrices here are random and NOT symmetric, so a transposed spd index
cannot hide.  A last group plants mistakes in a copy of the oracle source and
checks that these pins catch each one.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

from oracle import oracle as O



@pytest.fixture(autouse=True)
def _fp64_default():
    """fp64 as torch's default dtype inside this module's tests only (set at
    import it would leak into every test collected after it)."""
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


def _case(n, h, d, nb, seed, t_std=1.0, sym=False, code_hi=None):
    """Random inputs; bucket codes uniform on [0, nb), or on [0, code_hi) when
    given (code_hi up to 256: bytes at or above nb, above 127 included)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, h, d))
    k = rng.standard_normal((n, h, d))
    v = rng.standard_normal((n, h, d))
    dO = rng.standard_normal((n, h, d))
    T = t_std * rng.standard_normal((h, nb))
    spd = rng.integers(0, code_hi or nb, size=(n, n)).astype(np.uint8).view(np.int8)
    if sym:
        spd = np.triu(spd) + np.triu(spd, 1).T
    return q, k, v, dO, T, spd


def _torch_ref(q, k, v, dO, T, spd, scale):
    """SDPA + autograd reference: returns o, lse, dq, dk, dv, dT (numpy fp64).
    The bias of a pair is column `code` of T padded with zero columns to 256
    (every byte value), so a code at or above nb adds 0 and, the padding being a
    constant, receives no gradient."""
    qt = torch.tensor(q).permute(1, 0, 2).contiguous().requires_grad_(True)   # [h][n][d]
    kt = torch.tensor(k).permute(1, 0, 2).contiguous().requires_grad_(True)
    vt = torch.tensor(v).permute(1, 0, 2).contiguous().requires_grad_(True)
    Tt = torch.tensor(T).requires_grad_(True)
    Tpad = torch.cat([Tt, torch.zeros(T.shape[0], 256 - T.shape[1])], dim=1)
    codes = torch.tensor(np.asarray(spd).view(np.uint8).astype(np.int64))
    bias = Tpad[:, codes]                                                     # [h][n][n]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt[None], kt[None], vt[None], attn_mask=bias[None], scale=scale)[0]
    o.backward(torch.tensor(dO).permute(1, 0, 2))
    with torch.no_grad():
        scores = scale * qt @ kt.transpose(-1, -2) + bias
        lse = torch.logsumexp(scores, dim=-1)                                 # [h][n]
    perm = lambda t: t.detach().permute(1, 0, 2).numpy()
    return dict(o=perm(o), lse=lse.numpy(), dq=perm(qt.grad), dk=perm(kt.grad),
                dv=perm(vt.grad), dT=Tt.grad.numpy())


SHAPES = [(1, 1, 1, 1), (5, 2, 4, 3), (33, 3, 8, 7), (130, 8, 8, 18), (70, 8, 16, 26),
          (64, 4, 2, 34)]


@pytest.mark.parametrize("n,h,d,nb", SHAPES)
def test_forward_matches_sdpa(n, h, d, nb):
    q, k, v, dO, T, spd = _case(n, h, d, nb, seed=n * 7 + d)
    scale = 1.0 / np.sqrt(d)
    ref = _torch_ref(q, k, v, dO, T, spd, scale)
    o, lse = O.attn_fwd(q, k, v, spd, T, scale)
    np.testing.assert_allclose(o, ref["o"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref["lse"], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n,h,d,nb", SHAPES)
def test_backward_matches_autograd(n, h, d, nb):
    q, k, v, dO, T, spd = _case(n, h, d, nb, seed=n * 11 + d)
    scale = 0.37 if d == 4 else 1.0 / np.sqrt(d)
    ref = _torch_ref(q, k, v, dO, T, spd, scale)
    got = O.attn_fwd_bwd(q, k, v, dO, spd, T, scale)
    for name in ("o", "lse", "dq", "dk", "dv", "dT"):
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-9, atol=1e-11, err_msg=name)


@pytest.mark.parametrize("n,h,d,nb", [(40, 3, 8, 7), (70, 8, 16, 26), (33, 2, 4, 1)])
def test_codes_at_or_above_nb_match_autograd(n, h, d, nb):
    """Bytes 0..255, most of them at or above nb (and above 127): zero bias,
    nothing in dT -- against SDPA + autograd over T padded with zero columns."""
    q, k, v, dO, T, spd = _case(n, h, d, nb, seed=n * 13 + nb, code_hi=256)
    assert (spd.view(np.uint8) >= nb).mean() > 0.5 and (spd.view(np.uint8) > 127).any()
    scale = 1.0 / np.sqrt(d)
    ref = _torch_ref(q, k, v, dO, T, spd, scale)
    got = O.attn_fwd_bwd(q, k, v, dO, spd, T, scale)
    for name in ("o", "lse", "dq", "dk", "dv", "dT"):
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-9, atol=1e-11, err_msg=name)


def test_codes_at_or_above_nb_all_pairs():
    """Every pair's code at or above nb: plain softmax attention (SDPA without a
    mask) and dT = 0 exactly."""
    q, k, v, dO, T, _ = _case(25, 4, 8, 9, seed=77)
    spd = np.random.default_rng(78).integers(9, 256, size=(25, 25)).astype(np.uint8).view(np.int8)
    g = O.attn_fwd_bwd(q, k, v, dO, spd, T)
    qt, kt, vt = (torch.tensor(a).permute(1, 0, 2) for a in (q, k, v))
    plain = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(g["o"], plain, rtol=1e-10, atol=1e-12)
    assert np.all(g["dT"] == 0.0)


def test_forward_row_subset_matches_full():
    q, k, v, dO, T, spd = _case(50, 3, 4, 6, seed=3)
    o, lse = O.attn_fwd(q, k, v, spd, T)
    rows = np.array([49, 0, 17, 17, 3])
    o2, lse2 = O.attn_fwd(q, k, v, spd, T, rows=rows)
    np.testing.assert_array_equal(o2, o[rows])
    np.testing.assert_array_equal(lse2, lse[:, rows])


def _loss(q, k, v, dO, T, spd, scale):
    o, _ = O.attn_fwd(q, k, v, spd, T, scale, nthreads=1)
    return float((o * dO).sum())


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_finite_differences(seed):
    n, h, d, nb = 9, 2, 3, 5
    q, k, v, dO, T, spd = _case(n, h, d, nb, seed=seed)
    scale = 0.6
    g = O.attn_fwd_bwd(q, k, v, dO, spd, T, scale)
    eps = 1e-6
    rng = np.random.default_rng(seed + 100)
    args = dict(q=q, k=k, v=v, T=T)
    grads = dict(q=g["dq"], k=g["dk"], v=g["dv"], T=g["dT"])
    for name in args:
        for _ in range(6):
            idx = tuple(int(rng.integers(s)) for s in args[name].shape)
            plus = {a: b.copy() for a, b in args.items()}
            minus = {a: b.copy() for a, b in args.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            fd = (_loss(plus["q"], plus["k"], plus["v"], dO, plus["T"], spd, scale)
                  - _loss(minus["q"], minus["k"], minus["v"], dO, minus["T"], spd, scale)) / (2 * eps)
            assert abs(fd - grads[name][idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grads[name][idx])


def test_closed_form_uniform_v():
    """All rows of V equal: o_i = v, and dq = dk = 0 (dS rows sum to zero against a constant V)."""
    n, h, d, nb = 40, 4, 8, 9
    q, k, v, dO, T, spd = _case(n, h, d, nb, seed=5)
    v[:] = v[0]
    g = O.attn_fwd_bwd(q, k, v, dO, spd, T)
    np.testing.assert_allclose(g["o"], np.broadcast_to(v[0], g["o"].shape), atol=1e-13)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dk"], 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dT"], 0.0, atol=1e-11)


def test_closed_form_zero_and_constant_bias():
    """T = 0 is plain softmax attention; a per-head constant T shifts every score of a
    row equally, so o is unchanged, lse shifts by the constant and dT[h] sums to 0."""
    n, h, d, nb = 48, 3, 8, 7
    q, k, v, dO, T, spd = _case(n, h, d, nb, seed=6)
    zero = np.zeros_like(T)
    o0, lse0 = O.attn_fwd(q, k, v, spd, zero)
    qt, kt, vt = (torch.tensor(a).permute(1, 0, 2) for a in (q, k, v))
    plain = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o0, plain, rtol=1e-10, atol=1e-12)
    c = np.array([0.5, -2.0, 3.25])[:, None] * np.ones((1, nb))
    g = O.attn_fwd_bwd(q, k, v, dO, spd, c)
    np.testing.assert_allclose(g["o"], o0, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["lse"], lse0 + c[:, :1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dT"].sum(1), 0.0, atol=1e-11)


def test_closed_form_single_node():
    """N = 1: the only weight is 1, so o = v, lse = s_00, all gradients but dv vanish."""
    q, k, v, dO, T, spd = _case(1, 8, 16, 18, seed=8)
    spd[:] = 0
    g = O.attn_fwd_bwd(q, k, v, dO, spd, T)
    np.testing.assert_allclose(g["o"], v, atol=1e-14)
    s00 = (q * k).sum(-1)[0] / 4.0 + T[:, 0]
    np.testing.assert_allclose(g["lse"][:, 0], s00, atol=1e-13)
    np.testing.assert_allclose(g["dv"], dO, atol=1e-14)
    for name in ("dq", "dk", "dT"):
        np.testing.assert_allclose(g[name], 0.0, atol=1e-13)


def test_closed_form_complete_graph_two_buckets():
    """Complete graph: bucket 0 on the diagonal, 1 elsewhere, so dT[h][1] = -dT[h][0]."""
    n, h, d, nb = 30, 8, 8, 18
    q, k, v, dO, T, _ = _case(n, h, d, nb, seed=9)
    spd = np.ones((n, n), np.int8); np.fill_diagonal(spd, 0)
    g = O.attn_fwd_bwd(q, k, v, dO, spd, T)
    np.testing.assert_allclose(g["dT"][:, 1], -g["dT"][:, 0], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(g["dT"][:, 2:], 0.0, atol=0)
    assert np.all(np.abs(g["dT"][:, 0]) > 1e-6)


def test_dT_sums_to_zero_any_input():
    q, k, v, dO, T, spd = _case(90, 8, 8, 34, seed=10)
    g = O.attn_fwd_bwd(q, k, v, dO, spd, T)
    assert np.all(np.abs(g["dT"].sum(1)) < 1e-10 * np.abs(g["dT"]).sum(1).max())


def test_partial_rows_cols_match_full():
    q, k, v, dO, T, spd = _case(37, 2, 4, 5, seed=12)
    full = O.attn_fwd_bwd(q, k, v, dO, spd, T)
    rows = np.array([36, 1, 5]); cols = np.array([0, 20])
    part = O.attn_bwd(q, k, v, dO, spd, T, full["lse"], full["D"], rows=rows, cols=cols, want_dT=False)
    np.testing.assert_allclose(part["dq"], full["dq"][rows], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(part["dk"], full["dk"][cols], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(part["dv"], full["dv"][cols], rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------- planted mistakes

MUTATIONS = {
    "drop_bias": ("return c->scale * dot + bias;", "return c->scale * dot;"),
    "transpose_spd": ("int code = (int)(uint8_t)c->spd[(int64_t)i * c->ld + j];\n    double bias",
                      "int code = (int)(uint8_t)c->spd[(int64_t)j * c->ld + i];\n    double bias"),
    "bias_head_index": ("double bias = code < c->nb ? c->T[(int64_t)hh * c->nb + code] : 0.0;",
                        "double bias = code < c->nb ? c->T[code] : 0.0;"),
    "scale_dropped": ("return c->scale * dot + bias;", "return dot + bias;"),
    "high_code_clamped": ("double bias = code < c->nb ? c->T[(int64_t)hh * c->nb + code] : 0.0;",
                          "double bias = c->T[(int64_t)hh * c->nb + (code < c->nb ? code : c->nb - 1)];"),
    "high_code_in_dT": ("if (dT && code < c->nb) dT[(int64_t)hh * c->nb + code] += ds;",
                        "if (dT) dT[(int64_t)hh * c->nb + (code < c->nb ? code : c->nb - 1)] += ds;"),
    "ds_sign": ("double ds = p * (dprob(c, i, j, hh) - Di);",
                "double ds = p * (dprob(c, i, j, hh) + Di);"),
    "dk_uses_k": ("dkj[t] += c->scale * ds * qi[t];", "dkj[t] += c->scale * ds * c->k[((int64_t)j * c->h + hh) * c->d + t];"),
    "dv_drops_p": ("dvj[t] += p * gi[t];", "dvj[t] += gi[t];"),
    "dT_wrong_bucket": ("int code = (int)(uint8_t)c->spd[(int64_t)i * c->ld + j];\n                if (dT",
                        "int code = (int)(uint8_t)c->spd[(int64_t)j * c->ld + i];\n                if (dT"),
    "lse_no_max": ("c->lse_out[(int64_t)hh * c->nrows + r] = m + log(l);",
                   "c->lse_out[(int64_t)hh * c->nrows + r] = log(l);"),
    "spd_no_clip": ("(dist[v] < c->D ? dist[v] : c->D)", "dist[v]"),
    "spd_unreach_code": ("int32_t code = dist[v] < 0 ? c->D + 1", "int32_t code = dist[v] < 0 ? c->D"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="gto_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)
    O.use_library(None)


def _pins_pass() -> bool:
    """Run a compact set of the pins above against whatever library is loaded."""
    try:
        for (n, h, d, nb, hi) in [(33, 3, 8, 7, None), (12, 2, 4, 5, None), (20, 2, 4, 5, 256)]:
            q, k, v, dO, T, spd = _case(n, h, d, nb, seed=n + d, code_hi=hi)
            ref = _torch_ref(q, k, v, dO, T, spd, 0.45)
            got = O.attn_fwd_bwd(q, k, v, dO, spd, T, 0.45)
            for name in ("o", "lse", "dq", "dk", "dv", "dT"):
                np.testing.assert_allclose(got[name], ref[name], rtol=1e-9, atol=1e-11)
        import gt_inputs as gi
        g = gi.erdos_renyi(40, 0.05, seed=3)
        from scipy.sparse import csr_matrix
        from scipy.sparse.csgraph import shortest_path
        A = csr_matrix((np.ones(g.nnz), g.indices, g.indptr), shape=(g.n, g.n))
        dist = shortest_path(A, directed=False, unweighted=True)
        ref = np.where(np.isfinite(dist), np.minimum(dist, 3), 4).astype(np.int8)
        np.testing.assert_array_equal(O.spd(g.n, g.indptr, g.indices, 3), ref)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(O.__file__), "gt_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    path = os.path.join(mutant_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = O.compile_source(path, os.path.join(mutant_dir, f"lib{name}.so"))
    O.use_library(lib)
    try:
        assert not _pins_pass(), f"planted mistake {name!r} slipped past the pins"
    finally:
        O.use_library(None)


def test_unmutated_oracle_passes_compact_pins():
    O.use_library(None)
    assert _pins_pass()
