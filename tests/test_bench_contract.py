"""The benchmark's output contract on CPU: the roofline arithmetic of its JSON
line (algorithmic work per launch over the launch's time, against the stated
peak), the work it credits per step, and the reference arm's line, which runs
the fp64 oracle only and so needs no GPU."""
import json
import os
import subprocess
import sys

import pytest

import bench
import gt_inputs as gi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_credited_work_per_step():
    w = gi.CONFIGS[4]                       # N = 16384, H = 8, d = 16, one layer
    assert bench.attn_flops(w) == 14.0 * 16384 ** 2 * 8 * 16
    assert bench.exps(w) == 2.0 * 16384 ** 2 * 8
    w3 = gi.CONFIGS[3]                      # 16 layers of N = 6800, d = 8
    assert bench.attn_flops(w3) == 16 * 14.0 * 6800 ** 2 * 8 * 8


def test_exp_kernel_roofline_is_work_over_time_over_peak():
    w = gi.CONFIGS[4]
    peak = 152 * 32.0 * 2.07e9              # ex2 results per second
    r = bench.kernel_roofline("fwd_tc", w, 1.25, peak, 6693.5e9)
    work = 16384.0 ** 2 * 8                 # one exp per (query, key, head) per launch
    assert r["bound"] == "exp" and r["unit"] == "Texp/s"
    assert r["work_per_launch"] == work
    assert r["achieved"] == pytest.approx(work / 1.25e-3 / 1e12, abs=1e-4)
    assert r["peak"] == pytest.approx(peak / 1e12, abs=1e-3)
    assert r["frac"] == pytest.approx(work / 1.25e-3 / peak, abs=1e-4)
    assert r["traffic"] == bench.DRAM_BYTES[("fwd_tc", "ba64x256")]
    # a workload without a capture reports no traffic rather than another's
    assert bench.kernel_roofline("fwd_tc", gi.CONFIGS[2], 1.0, peak, 6693.5e9)["traffic"] is None
    # a kernel with several launches per layer: the layer's exps over its launches,
    # and the mean DRAM bytes of its launches (the dk/dv full wave, 179.953 MB, and
    # split tail, 132.676 MB, captured separately)
    r2 = bench.kernel_roofline("bwd_dkdv", w, 0.5, peak, 6693.5e9, launches_per_layer=2.0)
    assert r2["work_per_launch"] == work / 2
    assert r2["traffic"] == pytest.approx((179.953e6 + 132.676e6) / 2, rel=1e-5)
    assert r2["frac"] == pytest.approx(work / 2 / 0.5e-3 / peak, abs=1e-4)


def test_hbm_kernel_roofline_counts_the_bucket_bytes():
    w = gi.CONFIGS[4]
    r = bench.kernel_roofline("spd_bfs", w, 0.1, 1.0, 6693.5e9)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(16384.0 ** 2 / 1e-4 / 1e9, abs=0.01)   # GB/s, two decimals
    assert r["frac"] == pytest.approx(16384.0 ** 2 / 1e-4 / 6693.5e9, abs=1e-4)


def test_reference_arm_line():
    """`bench.py --impl reference` times the oracle; its line carries the same
    metric and unit as the GPU arm, a cpu_baseline describing the run, and an
    e2e with no host-device copies."""
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "1", "--steps", "1",
                          "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 1 and line["value"] > 0
    assert line["config"]["workload"].startswith("er512")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and isinstance(cb["sample"], str)
    assert cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
