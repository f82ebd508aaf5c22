"""GPU parity of gt_bias_attn_fwd / gt_bias_attn_bwd against the fp64 CPU oracle.

Tolerances: fp32 storage max-abs <= 1e-4; bf16 storage relative L2 <= 2e-2 per
output tensor (o, lse, dq, dk, dv, dT).  The oracle runs on exactly the values
the GPU sees (bf16-rounded inputs upcast to fp64).  Bucket matrices come from
the oracle's own BFS or are drawn at random (not symmetric), never from the GPU.
"""
import numpy as np
import pytest
import torch

import gt_inputs as gi
from oracle import oracle as O
from tests.helpers import assert_close, assert_dT_stored_o, host, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gt():
    import graph_transformer_attention_gb300 as m
    from graph_transformer_attention_gb300 import build
    build.build()
    m.load_library()
    return m


def _spd_dev(spd: np.ndarray) -> torch.Tensor:
    n = spd.shape[0]
    ld = (n + 15) // 16 * 16
    buf = np.zeros((n, ld), np.int8)
    buf[:, :n] = spd
    return torch.from_numpy(buf).cuda()


def _run_gpu(gt, x, spd, dtype, kv_block=0, scale=None):
    q, k, v, dO = (to_dev(x[a], dtype) for a in ("q", "k", "v", "dO"))
    T = torch.from_numpy(x["T"]).cuda()
    sp = _spd_dev(spd)
    o, lse = gt.gt_bias_attn_fwd(q, k, v, sp, T, scale=scale, kv_block=kv_block)
    dq, dk, dv, dT = gt.gt_bias_attn_bwd(q, k, v, o, dO, lse, sp, T, scale=scale)
    gt.gt_check_device_status()
    return dict(o=host(o), lse=host(lse), dq=host(dq), dk=host(dk), dv=host(dv), dT=host(dT))


def _compare_full(got, ref, dtype, names=("o", "lse", "dq", "dk", "dv", "dT")):
    return {nm: assert_close(nm, got[nm], ref[nm], dtype) for nm in names}


SMALL = [
    # n, h, d, dtype, nb, kv_block, graph-or-random
    (1, 8, 8, "f32", 18, 0, "random"),
    (2, 8, 8, "bf16", 18, 0, "random"),
    (37, 8, 8, "f32", 18, 0, "graph"),
    (130, 8, 8, "bf16", 18, 0, "random"),
    (300, 8, 16, "bf16", 26, 0, "graph"),
    (513, 8, 8, "bf16", 34, 128, "graph"),
    (257, 4, 32, "f32", 7, 0, "random"),
    (200, 2, 64, "f32", 5, 0, "random"),
    (1000, 8, 8, "bf16", 22, 256, "random"),
    (640, 8, 16, "bf16", 26, 0, "graph"),
    (129, 4, 16, "bf16", 9, 0, "random"),
    # many buckets: the dT bins of the tensor-core backward shrink to fewer copies
    (700, 8, 8, "bf16", 100, 0, "random"),
    (520, 8, 16, "bf16", 60, 0, "random"),
    (400, 8, 16, "bf16", 128, 0, "random"),
]


@pytest.mark.parametrize("n,h,d,dtype,nb,kv_block,kind", SMALL)
def test_small_parity(gt, n, h, d, dtype, nb, kv_block, kind):
    seed = 10 * n + d
    x = gi.make_layer_tensors(n, h, d, nb, dtype, seed=seed)
    if kind == "graph":
        g = gi.barabasi_albert(n, 2, seed=seed) if n > 3 else gi.erdos_renyi(n, 0.5, seed)
        spd = O.spd(n, g.indptr, g.indices, nb - 2)
    else:
        spd = np.random.default_rng(seed).integers(0, nb, size=(n, n)).astype(np.int8)
    got = _run_gpu(gt, x, spd, dtype, kv_block=kv_block)
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, dtype)


@pytest.mark.parametrize("n,d,dtype,nb,kv_block", [(300, 8, "bf16", 18, 0), (520, 16, "bf16", 26, 0),
                                                    (700, 8, "bf16", 22, 256), (150, 8, "f32", 18, 0),
                                                    (257, 32, "f32", 7, 0)])
def test_codes_at_or_above_nb(gt, n, d, dtype, nb, kv_block):
    """Bucket bytes 0..255 (most at or above nb, many above 127): such a byte adds
    no bias and no dT term, in the kernels as in the oracle.  Half the rows hold
    high codes only, so whole chunks take the uniform paths with such a code."""
    h = 8 if d <= 16 else 4
    x = gi.make_layer_tensors(n, h, d, nb, dtype, seed=60 + n)
    rng = np.random.default_rng(61 + n)
    spd = rng.integers(0, 256, size=(n, n)).astype(np.uint8)
    spd[n // 2:, :] = rng.integers(nb, 256)
    spd = spd.view(np.int8)
    got = _run_gpu(gt, x, spd, dtype, kv_block=kv_block)
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, dtype)


def test_large_bias_values(gt):
    """Bias up to +-30 makes the running max jump between KV blocks."""
    n, h, d, nb = 700, 8, 8, 18
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=3)
    x["T"] = (np.random.default_rng(4).uniform(-30, 30, size=(h, nb))).astype(np.float32)
    spd = np.random.default_rng(5).integers(0, nb, size=(n, n)).astype(np.int8)
    got = _run_gpu(gt, x, spd, "bf16")
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, "bf16")


@pytest.mark.parametrize("d", [8, 16])
def test_growing_scores(gt, d):
    """Scores that keep growing along the row force repeated rescales of the output.
    The growth comes from the bias: bucket codes rise with the column index and the
    table rises with the code, by 24 in total along every row."""
    n, h, nb = 600, 8, 26
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=13 + d)
    x["T"] = (x["T"] + np.arange(nb, dtype=np.float32)[None, :] * (24.0 / (nb - 1))).astype(np.float32)
    cols = (np.arange(n) * nb) // n
    jitter = np.random.default_rng(14).integers(-1, 2, size=(n, n))
    spd = np.clip(cols[None, :] + jitter, 0, nb - 1).astype(np.int8)
    got = _run_gpu(gt, x, spd, "bf16")
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, "bf16")


@pytest.mark.parametrize("d", [8, 16])
def test_growing_scores_uniform_runs(gt, d):
    """The same growth where every row holds code j // 16 at column j: every
    16-column half chunk is uniform across a warp's rows, so the forward forms
    x - m from the bias minus the running maximum there, and each half chunk
    brings a new maximum (the table rises by 4 per bucket), redoing it on shifted
    scores, in both halves of a chunk.  The ragged last block is a mixed half
    chunk (columns past n read code 0).

    Most of the probability sits in the last buckets, whose dT is then a near-zero
    difference: rounding o to bf16 alone (D_i = <dO_i, o_i> comes from the stored
    o) moves dT by a few % in relative L2 in exact arithmetic.  So dT is checked
    twice: at relative L2 2e-2 against the oracle backward given the o the
    backward was given (the kernels' own arithmetic), and end to end against the
    oracle within the bound that rounding o to bf16 sets (tests/helpers.py)."""
    n, h, nb = 600, 8, 40
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=31 + d)
    x["T"] = (x["T"] + np.arange(nb, dtype=np.float32)[None, :] * 4.0).astype(np.float32)
    cols = np.minimum(np.arange(n) // 16, nb - 1)
    spd = np.broadcast_to(cols[None, :], (n, n)).astype(np.int8).copy()
    got = _run_gpu(gt, x, spd, "bf16")
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, "bf16", names=("o", "lse", "dq", "dk", "dv"))
    q, k, v, dO = (np.asarray(x[a], np.float64) for a in ("q", "k", "v", "dO"))
    d_stored = O.bwd_delta(np.asarray(got["o"], np.float64), dO)
    ref_b = O.attn_bwd(q, k, v, dO, spd, x["T"], ref["lse"], d_stored)
    assert_close("dT", got["dT"], ref_b["dT"], "bf16")
    err, bound = assert_dT_stored_o(got["dT"], ref["dT"], ref["o"], got["o"], dO)
    print(f"growing_scores_uniform_runs d={d}: end-to-end dT rel L2 {rel_l2(got['dT'], ref['dT']):.3e}, "
          f"max err {err:.3e}, stored-o bound {bound:.3e}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_unreachable_and_single_bucket(gt, dtype):
    n, h, d, D = 300, 8, 8, 16
    x = gi.make_layer_tensors(n, h, d, D + 2, dtype, seed=21)
    empty = gi.csr_from_edges(n, np.zeros(0, np.int64), np.zeros(0, np.int64))
    spd = O.spd(n, empty.indptr, empty.indices, D)   # 0 on the diagonal, D+1 elsewhere
    got = _run_gpu(gt, x, spd, dtype)
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, dtype, names=("o", "lse", "dq", "dk", "dv") + (("dT",) if dtype == "f32" else ()))
    # Only two buckets are used, and the diagonal bucket holds N tiny terms, so dT
    # is small and its error is set by D_i = <dO_i, o_i> being taken from the
    # stored o: each row's dS then sums to dD_i = <dO_i, o_i - o_i'> instead of 0,
    # and a bucket's error is at most sum_i |dD_i| (p_ij <= 1 summed over j).
    err, bound = assert_dT_stored_o(got["dT"], ref["dT"], ref["o"], got["o"], x["dO"])
    print(f"all_unreachable {dtype}: end-to-end dT rel L2 {rel_l2(got['dT'], ref['dT']):.3e}, "
          f"max err {err:.3e}, stored-o bound {bound:.3e}")
    assert np.all(got["dT"][:, 1:D + 1] == 0.0)
    spd1 = np.full((n, n), 3, np.int8)                  # one bucket everywhere
    got = _run_gpu(gt, x, spd1, dtype)
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd1, x["T"])
    _compare_full(got, ref, dtype, names=("o", "lse", "dq", "dk", "dv"))
    # One bucket holds every pair, so dT[h][3] = sum_ij dS_ij.  Exactly that is
    # sum_i <dO_i, o_i - o_i'> where o' is the output the backward was given: zero
    # for exact o, and the bf16 rounding residual of o otherwise.
    do64 = x["dO"].astype(np.float64)
    predicted = ((ref["o"] - got["o"]) * do64).sum(axis=(0, 2))       # [h]
    assert np.all(np.abs(got["dT"][:, 3] - predicted) <= 1e-3 + 2e-2 * np.abs(predicted))
    assert np.all(got["dT"][:, np.arange(D + 2) != 3] == 0.0)
    err, bound = assert_dT_stored_o(got["dT"], ref["dT"], ref["o"], got["o"], x["dO"])
    print(f"single_bucket {dtype}: end-to-end dT max err {err:.3e}, stored-o bound {bound:.3e}")


@pytest.mark.parametrize("d,mag", [(8, 40.0), (16, 40.0), (16, 1e-3)])
def test_dT_fixed_point_scale_extremes(gt, d, mag):
    """The bf16 backward sums dT in fixed point with a per-CTA scale derived from
    |dO_i| max_j |v_j| + |D_i|.  Large dO and v (dS of hundreds) must not
    overflow; tiny ones must keep their relative accuracy.  Random codes send
    every chunk through the per-element bins."""
    n, h, nb = 520, 8, 30
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=31 + d)
    x["dO"] = gi.round_to_bf16((x["dO"] * mag).astype(np.float32))
    x["v"] = gi.round_to_bf16((x["v"] * (mag if mag > 1 else 1.0)).astype(np.float32))
    spd = np.random.default_rng(32).integers(0, nb, size=(n, n)).astype(np.int8)
    got = _run_gpu(gt, x, spd, "bf16")
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, "bf16")


def test_components_not_aligned_to_tiles(gt):
    """Disjoint graphs of 40 nodes: the 16 x 32 blocks of the bucket matrix mix
    uniform blocks (pairs in other components, one code) with blocks that cut a
    component's diagonal block, so both the per-block and per-element paths of
    the backward run in one launch."""
    n_comp, size = 25, 40
    g = gi.disjoint_ba(n_comp, size, 2, seed=41)
    n, h, d, D = n_comp * size, 8, 16, 12
    spd = O.spd(n, g.indptr, g.indices, D)
    x = gi.make_layer_tensors(n, h, d, D + 2, "bf16", seed=42)
    got = _run_gpu(gt, x, spd, "bf16")
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, "bf16")


@pytest.mark.parametrize("dtype,d", [("bf16", 8), ("bf16", 16), ("f32", 8), ("bf16", 32)])
def test_partial_ranges_and_merge(gt, dtype, d):
    """gt_bias_attn_fwd_partial over three KV ranges, each against the oracle with
    the columns outside the range masked (a bias of -inf through an extra code),
    then gt_bias_attn_merge of the three against the full forward."""
    n, h, nb = 1000, 8, 22
    x = gi.make_layer_tensors(n, h, d, nb, dtype, seed=50 + d)
    spd = np.random.default_rng(51).integers(0, nb, size=(n, n)).astype(np.int8)
    q, k, v = (to_dev(x[a], dtype) for a in ("q", "k", "v"))
    T = torch.from_numpy(x["T"]).cuda()
    sp = _spd_dev(spd)
    t_ext = np.concatenate([x["T"], np.full((h, 1), -np.inf, np.float32)], axis=1)
    ops, lps = [], []
    for a, b in ((0, 384), (384, 640), (640, n)):
        op, lp = gt.gt_bias_attn_fwd_partial(q, k, v, sp, T, a, b)
        gt.gt_check_device_status()
        masked = spd.copy()
        masked[:, :a] = nb
        masked[:, b:] = nb
        ro, rl = O.attn_fwd(x["q"], x["k"], x["v"], masked, t_ext)
        assert_close("o_part", host(op), ro, dtype)
        assert_close("lse_part", host(lp), rl, dtype)
        ops.append(op)
        lps.append(lp)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o, lse = gt.gt_bias_attn_merge(torch.stack(ops), torch.stack(lps), dtype=tdt)
    gt.gt_check_device_status()
    ro, rl = O.attn_fwd(x["q"], x["k"], x["v"], spd, x["T"])
    assert_close("o", host(o), ro, dtype)
    assert_close("lse", host(lse), rl, dtype)


def test_kv_block_matches_single_pass(gt):
    n, h, d, nb = 1100, 8, 8, 34
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=8)
    spd = np.random.default_rng(9).integers(0, nb, size=(n, n)).astype(np.int8)
    a = _run_gpu(gt, x, spd, "bf16", kv_block=0)
    b = _run_gpu(gt, x, spd, "bf16", kv_block=256)
    for nm in ("o", "lse"):
        assert np.linalg.norm(a[nm] - b[nm]) <= 1e-2 * np.linalg.norm(a[nm])


@pytest.mark.parametrize("n,d,kind", [(1000, 16, "random"), (2048, 8, "graph"), (4096, 16, "random")])
def test_balanced_forward_pieces(gt, n, d, kind):
    """The forward's balanced grid: each CTA takes an equal contiguous share of
    the (tile, head half, KV block) work, so one tile's KV range is covered by up
    to six CTAs here (n = 4096), whose pieces are merged through their lse while
    whole ranges are written directly.  Every row against the oracle."""
    tiles = (n + 127) // 128
    assert gt.load_library().gt_bias_attn_fwd_ctas(1, n, 8, d, 0) > 2 * tiles
    nb = 26
    x = gi.make_layer_tensors(n, 8, d, nb, "bf16", seed=60 + d)
    if kind == "graph":
        g = gi.disjoint_ba(n // 64, 64, 2, seed=61)
        spd = O.spd(n, g.indptr, g.indices, nb - 2)
    else:
        spd = np.random.default_rng(62).integers(0, nb, size=(n, n)).astype(np.int8)
    q, k, v = (to_dev(x[a], "bf16") for a in ("q", "k", "v"))
    T = torch.from_numpy(x["T"]).cuda()
    o, lse = gt.gt_bias_attn_fwd(q, k, v, _spd_dev(spd), T)
    gt.gt_check_device_status()
    ro, rl = O.attn_fwd(x["q"], x["k"], x["v"], spd, x["T"])
    assert_close("o", host(o), ro, "bf16")
    assert_close("lse", host(lse), rl, "bf16")
    # no row is left unwritten or written twice over: every row's error is small
    err = np.abs(host(lse) - rl).max(axis=0)
    assert np.all(err < 0.05), np.argsort(err)[-5:]


def test_backward_after_balanced_forward_ragged(gt):
    """The backward at a ragged size (n = 9857: 78 tiles, the last one 1 row):
    its 156 dq tasks fill no wave of two CTAs per SM and are all split along
    their KV blocks, its 156 dk/dv groups fill one wave of one CTA per SM and the
    4 past it are split along their query tiles; fed by the balanced forward (156
    tasks over two waves' worth of CTAs, up to three CTAs per tile).  Rows: the
    first and last of every tile plus random ones, against the oracle; dT by its
    zero-sum property."""
    n, h, d, nb = 9857, 8, 16, 26
    lib = gt.load_library()
    assert lib.gt_bias_attn_bwd_split(1, n, h, d, nb) >= 2
    assert lib.gt_bias_attn_fwd_ctas(1, n, h, d, 0) > 0
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=70)
    spd = np.random.default_rng(71).integers(0, nb, size=(n, n)).astype(np.int8)
    got = _run_gpu(gt, x, spd, "bf16")
    rng = np.random.default_rng(72)
    ends = np.concatenate([np.arange(0, n, 128), np.minimum(np.arange(127, n + 127, 128), n - 1)])
    rows = np.unique(np.concatenate([ends, rng.choice(n, 64, replace=False)]))
    o_r, lse_r = O.attn_fwd(x["q"], x["k"], x["v"], spd, x["T"], rows=rows)
    assert_close("o[rows]", got["o"][rows], o_r, "bf16")
    assert_close("lse[rows]", got["lse"][:, rows], lse_r, "bf16")
    Dv_rows = (o_r * x["dO"][rows].astype(np.float64)).sum(-1).T
    lse_full = np.zeros((h, n)); Dv_full = np.zeros((h, n))
    lse_full[:, rows] = lse_r; Dv_full[:, rows] = Dv_rows
    g = O.attn_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"], lse_full, Dv_full,
                   rows=rows, want_dT=False, want_dkdv=False)
    assert_close("dq[rows]", got["dq"][rows], g["dq"], "bf16")
    dT = got["dT"]
    bound = 2.0 ** -8 * np.abs(x["dO"].astype(np.float64) * got["o"]).sum(axis=(0, 2)) + 1e-4
    assert np.all(np.abs(dT.sum(1)) <= bound), (dT.sum(1), bound)


def test_two_wave_balanced_forward_and_split_dq(gt):
    """n = 20000: 157 tiles, 314 tasks for 304 resident slots, so the forward's
    balanced grid is two waves (608 CTAs) and the dq kernel runs a full wave of
    whole tasks and then the 10 tasks past it split along the KV blocks, that
    launch overlapping the first.  Rows: the first and last of every 16th tile,
    the last tile's, and random ones, against the oracle (o, lse, dq); dT and dv
    by their sum properties."""
    n, h, d, nb = 20000, 8, 16, 26
    lib = gt.load_library()
    tiles = (n + 127) // 128
    assert lib.gt_bias_attn_fwd_ctas(1, n, h, d, 0) >= 2 * tiles
    assert lib.gt_bias_attn_bwd_split(1, n, h, d, nb) >= 2
    x = gi.make_layer_tensors(n, h, d, nb, "bf16", seed=90)
    spd = np.random.default_rng(91).integers(0, nb, size=(n, n), dtype=np.int8)
    got = _run_gpu(gt, x, spd, "bf16")
    rng = np.random.default_rng(92)
    starts = np.arange(0, n, 128 * 16)
    split_rows = [152 * 128, 152 * 128 + 77, 155 * 128 + 5]   # tiles of the split tasks (past 304 tasks)
    rows = np.unique(np.concatenate([starts, np.minimum(starts + 127, n - 1), [n - 1, n - 2, (tiles - 1) * 128],
                                     split_rows, rng.choice(n, 48, replace=False)]))
    o_r, lse_r = O.attn_fwd(x["q"], x["k"], x["v"], spd, x["T"], rows=rows)
    assert_close("o[rows]", got["o"][rows], o_r, "bf16")
    assert_close("lse[rows]", got["lse"][:, rows], lse_r, "bf16")
    Dv_rows = (o_r * x["dO"][rows].astype(np.float64)).sum(-1).T
    lse_full = np.zeros((h, n)); Dv_full = np.zeros((h, n))
    lse_full[:, rows] = lse_r; Dv_full[:, rows] = Dv_rows
    g = O.attn_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"], lse_full, Dv_full,
                   rows=rows, want_dT=False, want_dkdv=False)
    assert_close("dq[rows]", got["dq"][rows], g["dq"], "bf16")
    bound = 2.0 ** -8 * np.abs(x["dO"].astype(np.float64) * got["o"]).sum(axis=(0, 2)) + 1e-4
    assert np.all(np.abs(got["dT"].sum(1)) <= bound)
    dsum = got["dv"].sum(0)
    assert np.linalg.norm(dsum - x["dO"].astype(np.float64).sum(0)) <= 2e-2 * np.linalg.norm(dsum) + 1e-3


def test_back_to_back_calls_on_one_stream(gt):
    """Calls of three sizes with different splits (n = 3000 and 700: every tile's
    stream split; n = 10000: only the tasks past the last full wave split; all
    three with the balanced forward), enqueued back to back on one non-default
    stream with no host
    synchronisation between them, give what each gives alone (the launches of
    a call overlap one another; completion order must still hold across calls).
    The split sums add in fp32 in any order, so fp32 outputs agree to 1e-5
    relative and bf16 ones to one bf16 unit (a sum near a rounding boundary may
    round either way); a read of an unfinished result would be far off."""
    cases = []
    for n, d, seed in ((3000, 16, 80), (10000, 8, 81), (700, 16, 82)):
        x = gi.make_layer_tensors(n, 8, d, 26, "bf16", seed=seed)
        spd = torch.randint(0, 26, (n, gt.spd_ld(n)), dtype=torch.int8, device="cuda",
                            generator=torch.Generator(device="cuda").manual_seed(seed))
        args = [to_dev(x[a], "bf16") for a in ("q", "k", "v")] + [spd, torch.from_numpy(x["T"]).cuda()]
        cases.append((args, to_dev(x["dO"], "bf16")))
    alone = []
    for args, dO in cases:
        o, lse = gt.gt_bias_attn_fwd(*args)
        g = gt.gt_bias_attn_bwd(*args[:3], o, dO, lse, *args[3:])
        torch.cuda.synchronize()
        alone.append([t.clone() for t in (o, lse, *g)])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        outs = []
        for args, dO in cases:
            o, lse = gt.gt_bias_attn_fwd(*args)
            g = gt.gt_bias_attn_bwd(*args[:3], o, dO, lse, *args[3:])
            outs.append([o, lse, *g])
    s.synchronize()
    gt.gt_check_device_status()
    for ref, got in zip(alone, outs):
        for a, b in zip(ref, got):
            a64, b64 = a.double(), b.double()
            rtol = 2.0 ** -7 if a.dtype == torch.bfloat16 else 1e-5
            assert torch.allclose(a64, b64, rtol=rtol, atol=1e-6 * a64.abs().max().item()), \
                (a.dtype, (a64 - b64).abs().max().item())


def _config_spd(w):
    g = gi.config_graph(w)
    return O.spd(g.n, g.indptr, g.indices, w.D)


@pytest.mark.parametrize("cfg", [1, 2])
def test_config_full_parity(gt, cfg):
    w = gi.CONFIGS[cfg]
    spd = _config_spd(w)
    x = gi.config_layer_tensors(w)
    got = _run_gpu(gt, x, spd, w.dtype, kv_block=w.kv_block)
    ref = O.attn_fwd_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"])
    _compare_full(got, ref, w.dtype)


def _sampled_check(gt, w, spd, layer, rng, full_cols: bool):
    x = gi.config_layer_tensors(w, layer)
    got = _run_gpu(gt, x, spd, w.dtype, kv_block=w.kv_block)
    n = w.n
    rows = np.sort(np.concatenate([rng.choice(n, 96, replace=False), [0, n - 1]]))
    o_r, lse_r = O.attn_fwd(x["q"], x["k"], x["v"], spd, x["T"], rows=rows)
    assert_close("o[rows]", got["o"][rows], o_r, w.dtype)
    assert_close("lse[rows]", got["lse"][:, rows], lse_r, w.dtype)
    # row-local backward: D_i needs only o_i, so dq of sampled rows needs no full pass
    Dv_rows = (o_r * x["dO"][rows].astype(np.float64)).sum(-1).T      # [h][rows]
    lse_full = np.zeros((w.heads, n)); Dv_full = np.zeros((w.heads, n))
    lse_full[:, rows] = lse_r; Dv_full[:, rows] = Dv_rows
    g = O.attn_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"], lse_full, Dv_full,
                   rows=rows, want_dT=False, want_dkdv=False)
    assert_close("dq[rows]", got["dq"][rows], g["dq"], w.dtype)
    # properties at any size: every row of dS sums to 0, so sum_c dT[h][c] = 0;
    # rows of P sum to 1, so sum_j dv_j = sum_i dO_i
    # (with o rounded to bf16, sum_c dT[h][c] = sum_i <dO_i, o_i - o_i'> exactly, which
    # is bounded by half an ulp of o' per element)
    dT = got["dT"]
    ulp = 2.0 ** -8 if w.dtype == "bf16" else 2.0 ** -22
    bound = ulp * np.abs(x["dO"].astype(np.float64) * got["o"]).sum(axis=(0, 2)) + 1e-4
    assert np.all(np.abs(dT.sum(1)) <= bound), (dT.sum(1), bound)
    dsum = got["dv"].sum(0)
    assert np.linalg.norm(dsum - x["dO"].astype(np.float64).sum(0)) <= 2e-2 * np.linalg.norm(dsum) + 1e-3
    if full_cols:
        o_all, lse_all = O.attn_fwd(x["q"], x["k"], x["v"], spd, x["T"])
        Dv_all = O.bwd_delta(o_all, x["dO"])
        cols = np.sort(np.concatenate([rng.choice(n, 96, replace=False), [0, n - 1]]))
        g = O.attn_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"], lse_all, Dv_all,
                       cols=cols, want_dq=False, want_dT=True)
        assert_close("dk[cols]", got["dk"][cols], g["dk"], w.dtype)
        assert_close("dv[cols]", got["dv"][cols], g["dv"], w.dtype)
        assert_close("dT", got["dT"], g["dT"], w.dtype)
        assert_close("o", got["o"], o_all, w.dtype)


@pytest.mark.slow
def test_config3_sixteen_layers(gt):
    w = gi.CONFIGS[3]
    spd = _config_spd(w)
    rng = np.random.default_rng(33)
    for layer in range(w.layers):
        _sampled_check(gt, w, spd, layer, rng, full_cols=layer in (0, w.layers - 1))


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [4, 5])
def test_config_large_sampled_and_full_dT(gt, cfg):
    w = gi.CONFIGS[cfg]
    spd = _config_spd(w)
    _sampled_check(gt, w, spd, 0, np.random.default_rng(40 + cfg), full_cols=True)
