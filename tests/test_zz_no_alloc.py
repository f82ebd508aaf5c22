"""gt_bias_attn_bwd_noalloc, the backward pass for callers that cannot allocate.

Callers such as a host framework that owns all device memory, or a real-time host
that forbids allocation after start-up, cannot hand the library a workspace.
The no-allocation variant keeps its scratch in an array compiled into the
library.  This test calls it through the C ABI (ctypes, raw pointers), twice in
a row on the same inputs, and checks both results against the regular
gt_bias_attn_bwd within the tolerances of the other parity tests.  The file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gt_inputs as gi
from oracle import oracle as O
from tests.helpers import assert_close, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gt():
    import graph_transformer_attention_gb300 as m
    from graph_transformer_attention_gb300 import build
    build.build()
    lib = m.load_library()
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.gt_bias_attn_bwd_noalloc.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, i64, P, i32,
                                             f32, P, P, P, P, P]
    lib.gt_bias_attn_bwd_noalloc.restype = ctypes.c_int
    return m


def _noalloc(gt, q, k, v, o, dO, lse, spd, T, scale):
    lib = gt.load_library()
    n, h, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dT = torch.empty_like(T)
    dt = gt.GT_BF16 if q.dtype == torch.bfloat16 else gt.GT_F32
    rc = lib.gt_bias_attn_bwd_noalloc(
        dt, n, h, d, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(),
        lse.data_ptr(), spd.data_ptr(), spd.stride(0), T.data_ptr(), T.shape[1], scale,
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dT.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0, gt.gt_status_string(rc)
    gt.gt_check_device_status()
    return dict(dq=host(dq), dk=host(dk), dv=host(dv), dT=host(dT))


@pytest.mark.parametrize("dtype,n,d", [("f32", 300, 8), ("bf16", 700, 16), ("bf16", 513, 8), ("bf16", 4000, 16)])
def test_noalloc_matches_regular_backward_twice(gt, dtype, n, d):
    """(bf16, 4000, 16): the regular call splits the backward's streams over 4
    CTAs per tile and sums in fp32; the built-in scratch is too small for those
    sums, so the no-allocation call runs unsplit, with the two backward kernels
    side by side on the library's second stream: both must agree."""
    h, D = 8, 12
    g = gi.barabasi_albert(n, 2, seed=n)
    spd_np = O.spd(n, g.indptr, g.indices, D)
    ld = (n + 15) // 16 * 16
    buf = np.zeros((n, ld), np.int8)
    buf[:, :n] = spd_np
    spd = torch.from_numpy(buf).cuda()
    x = gi.make_layer_tensors(n, h, d, D + 2, dtype, seed=n + d)
    q, k, v, dO = (to_dev(x[a], dtype) for a in ("q", "k", "v", "dO"))
    T = torch.from_numpy(x["T"]).cuda()
    scale = 1.0 / np.sqrt(d)
    o, lse = gt.gt_bias_attn_fwd(q, k, v, spd, T)
    ref = gt.gt_bias_attn_bwd(q, k, v, o, dO, lse, spd, T)
    gt.gt_check_device_status()
    ref = dict(zip(("dq", "dk", "dv", "dT"), (host(t) for t in ref)))
    for _ in range(2):
        got = _noalloc(gt, q, k, v, o, dO, lse, spd, T, scale)
        for name in ("dq", "dk", "dv", "dT"):
            assert_close(name, got[name], ref[name], dtype)


def test_noalloc_rejects_oversized_problem(gt):
    lib = gt.load_library()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check comes first
    n = 1 << 22                        # n * h far beyond the built-in scratch
    rc = lib.gt_bias_attn_bwd_noalloc(gt.GT_BF16, n, 8, 8, fake, fake, fake, fake, fake, fake,
                                      fake, n, fake, 18, 0.35, fake, fake, fake, fake, None)
    assert rc == -5
