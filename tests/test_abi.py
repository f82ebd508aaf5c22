"""The C ABI of libgt on the host (no GPU needed, no kernel launched).

Checks that the library builds and loads, that it exports every function that
include/gt_attn.h declares, and that argument checks reject bad calls with the
documented status codes before touching the device.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gt_attn.h")


@pytest.fixture(scope="module")
def lib():
    from graph_transformer_attention_gb300 import build
    build.build()
    import graph_transformer_attention_gb300 as gt
    return gt.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gt_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("gt_spd_build", "gt_bias_attn_fwd", "gt_bias_attn_bwd"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libgt.so does not export {name}"


def test_status_strings(lib):
    import graph_transformer_attention_gb300 as gt
    for code in (0, -1, -2, -3, -4, -5):
        s = gt.gt_status_string(code)
        assert s and s != "unknown status"
    assert gt.gt_status_string(42) == "unknown status"


def test_invalid_arguments_rejected_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)      # never dereferenced: every call below fails its host checks
    # gt_spd_build: NULL indptr, bad n, bad D, bad ld, misaligned output
    assert lib.gt_spd_build(None, fake, 4, 2, 2, fake, 16, fake, 1 << 20, None) == -1
    assert lib.gt_spd_build(fake, fake, 0, 2, 2, fake, 16, fake, 1 << 20, None) == -1
    assert lib.gt_spd_build(fake, fake, 4, 2, 0, fake, 16, fake, 1 << 20, None) == -1
    assert lib.gt_spd_build(fake, fake, 4, 2, 127, fake, 16, fake, 1 << 20, None) == -1
    assert lib.gt_spd_build(fake, fake, 4, 2, 3, fake, 8, fake, 1 << 20, None) == -1
    assert lib.gt_spd_build(fake, fake, 20, 2, 3, fake, 24, fake, 1 << 20, None) == -1
    assert lib.gt_spd_build(fake, fake, 4, 2, 3, P(0x1001), 16, fake, 1 << 20, None) == -1
    # GT layer: unsupported widths, NULL weights
    assert lib.gt_layer_fwd(100, 4, 8, 64, fake, fake, fake, 112, fake, 8, fake, fake, fake, fake, fake, fake,
                            fake, 1 << 20, None) == -2
    assert lib.gt_layer_fwd(100, 8, 8, 64, fake, None, fake, 112, fake, 8, fake, fake, fake, fake, fake, fake,
                            fake, 1 << 20, None) == -1
    assert lib.gt_layer_workspace_size(100, 8, 16, 64) == 0 and lib.gt_layer_workspace_size(100, 8, 8, 64) > 0
    # GT layer: node-row arrays must be 16-byte aligned (whole tiles move by bulk copies)
    class Twelve(ctypes.Structure):
        _fields_ = [(f"p{i}", P) for i in range(12)]
    wts = Twelve(*([fake] * 12))
    grads = Twelve(*([fake] * 12))
    odd = P(0x1004)
    assert lib.gt_layer_fwd(100, 8, 8, 64, odd, ctypes.byref(wts), fake, 112, fake, 8, fake, fake, fake, fake,
                            fake, fake, fake, 1 << 20, None) == -1
    assert lib.gt_layer_fwd(100, 8, 8, 64, fake, ctypes.byref(wts), fake, 112, fake, 8, fake, fake, fake, fake,
                            fake, odd, fake, 1 << 20, None) == -1
    assert lib.gt_layer_bwd(100, 8, 8, 64, fake, ctypes.byref(wts), fake, 112, fake, 8, fake, fake, fake, fake,
                            fake, odd, fake, ctypes.byref(grads), fake, fake, 1 << 20, None) == -1
    # bounded-wait self-test: limits out of range
    assert lib.gt_selftest_wait_timeout(ctypes.c_int64(10), None) == -1
    assert lib.gt_selftest_wait_timeout(ctypes.c_int64(2_000_000_000), None) == -1
    # unknown search algorithm
    assert lib.gt_spd_build_algo(9, fake, fake, 4, 2, 3, fake, 16, fake, 1 << 20, None) == -1
    assert lib.gt_spd_build_algo(-1, fake, fake, 4, 2, 3, fake, 16, fake, 1 << 20, None) == -1
    # forward: bad dtype, NULL q, misaligned q, bad ld, nb too large, bad kv_block
    args = lambda **kw: [kw.get("dt", 1), kw.get("n", 64), kw.get("h", 8), kw.get("d", 8),
                         kw.get("q", fake), fake, fake, fake, kw.get("ld", 64), fake,
                         kw.get("nb", 18), ctypes.c_float(0.35), kw.get("kvb", 0), fake, fake,
                         fake, 1 << 30, None]
    assert lib.gt_bias_attn_fwd(*args(dt=7)) == -1
    assert lib.gt_bias_attn_fwd(*args(q=None)) == -1
    assert lib.gt_bias_attn_fwd(*args(q=P(0x1008))) == -1
    assert lib.gt_bias_attn_fwd(*args(ld=63)) == -1
    assert lib.gt_bias_attn_fwd(*args(ld=48)) == -1
    assert lib.gt_bias_attn_fwd(*args(n=0)) == -1
    assert lib.gt_bias_attn_fwd(*args(nb=129)) == -2
    assert lib.gt_bias_attn_fwd(*args(d=65)) == -2
    assert lib.gt_bias_attn_fwd(*args(kvb=100)) == -1
    assert lib.gt_bias_attn_fwd(*args(kvb=-128)) == -1
    # backward: NULL dT
    bargs = [1, 64, 8, 8, fake, fake, fake, fake, fake, fake, fake, 64, fake, 18,
             ctypes.c_float(0.35), fake, fake, fake, None, fake, 1 << 30, None]
    assert lib.gt_bias_attn_bwd(*bargs) == -1
    # workspace too small
    bargs[18] = fake
    bargs[20] = 0
    assert lib.gt_bias_attn_bwd(*bargs) == -5


def test_workspace_sizes(lib):
    import graph_transformer_attention_gb300 as gt
    a = gt.gt_bias_attn_workspace_size(1, 4096, 8, 8, 0)
    b = gt.gt_bias_attn_workspace_size(1, 32768, 8, 8, 4096)
    assert a > 0 and b > a
    assert gt.gt_bias_attn_workspace_size(9, 4096, 8, 8, 0) == 0
    assert gt.gt_spd_workspace_size(0, 0, 16) == 0
    assert gt.gt_spd_workspace_size(512, 4000, 16) > 0
    # the global-memory search takes any n; an unknown algorithm takes none
    assert gt.gt_spd_workspace_size(512, 4000, 16, algo=gt.GT_SPD_GLOBAL64) > 0
    assert gt.gt_spd_workspace_size(512, 4000, 16, algo=9) == 0


def test_spd_ld():
    import graph_transformer_attention_gb300 as gt
    assert [gt.spd_ld(n) for n in (1, 16, 17, 6800)] == [16, 16, 32, 6800]


def test_kernel_stats_table_on_host(lib):
    import graph_transformer_attention_gb300 as gt
    count = ctypes.c_int32(-7)
    assert lib.gt_kernel_stats_read(None, -1, ctypes.byref(count)) == -1
    assert lib.gt_kernel_stats_read(None, 2, ctypes.byref(count)) == -1
    assert lib.gt_kernel_stats_read(None, 0, None) == -1
    # nothing launched since the reset: an empty table, no CUDA call needed
    gt.gt_kernel_stats_reset(False)
    assert gt.gt_kernel_stats() == {}


def test_partial_and_merge_reject_bad_ranges(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    f32p = ctypes.c_float
    # kv_begin not a multiple of 128, empty range, range past n, NULL outputs
    for kb, ke in ((64, 300), (128, 128), (0, 301), (-128, 10)):
        assert lib.gt_bias_attn_fwd_partial(1, 300, 8, 16, fake, fake, fake, fake, 304, fake, 18,
                                            f32p(0.25), kb, ke, fake, fake, None) == -1
    assert lib.gt_bias_attn_fwd_partial(1, 300, 8, 16, fake, fake, fake, fake, 304, fake, 18,
                                        f32p(0.25), 0, 300, None, fake, None) == -1
    assert lib.gt_bias_attn_merge(1, 300, 8, 16, 0, fake, fake, fake, fake, None) == -1
    assert lib.gt_bias_attn_merge(1, 300, 8, 128, 2, fake, fake, fake, fake, None) == -2
    assert lib.gt_bias_attn_merge(1, 300, 8, 16, 2, None, fake, fake, fake, None) == -1
