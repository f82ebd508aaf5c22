"""Failure detection on the GPU without a fault: a bounded wait that nothing
ends gives up, the host reads GT_ERR_TIMEOUT, and the context stays usable."""
import time

import numpy as np
import pytest

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


def test_bounded_wait_gives_up_and_reports_timeout(gt):
    gt.gt_check_device_status()                    # start from a clean status word
    t0 = time.perf_counter()
    gt.gt_selftest_wait_timeout(50_000_000)        # 50 ms
    with pytest.raises(gt.GtError) as e:
        gt.gt_check_device_status()
    assert e.value.status == -4                    # GT_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.045       # it waited its limit, no less
    # the check cleared the word, and the context still computes correctly
    gt.gt_check_device_status()
    g = gi.barabasi_albert(300, 2, seed=3)
    ip, ix = graph_to_dev(g)
    got = gt.gt_spd_build(ip, ix, g.n, 9)[:, :g.n].cpu().numpy()
    gt.gt_check_device_status()
    assert np.array_equal(got, O.spd(g.n, g.indptr, g.indices, 9))


def test_selftest_rejects_limits_out_of_range(gt):
    for bad in (0, 999_999, 1_000_000_001):
        with pytest.raises(gt.GtError):
            gt.gt_selftest_wait_timeout(bad)
