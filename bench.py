"""Benchmark: biased-attention fwd+bwd TFLOP/s and fraction of roofline on one GB300.

One step = one pass of the whole hot path on one synthetic graph:
SPD build (gt_spd_build) + forward (gt_bias_attn_fwd) + backward
(gt_bias_attn_bwd) for every layer, inputs resident in HBM.  Default workload
(--config 4): N = 16384 nodes, a disjoint union of 64 Barabasi-Albert graphs
(m = 3, 256 nodes each), H = 8 heads, head dim 16, bf16, clip D = 24.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gt|reference]
                    [--config 1..5]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload (the path needs no exchange between GPUs); value = work of all
ranks / max time over ranks.  `--impl reference` times the fp64 CPU oracle on
a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gt_inputs as gi  # noqa: E402

METRIC = "biased-attention fwd+bwd TFLOP/s and % of roofline on 1 GB300"

# Exp throughput of one GB300 SM: 32 ex2.approx.f32 results per clock (measured
# on this GPU with a throughput loop of independent ex2 chains, 16 warps per SM
# on all 152 SMs: 31.8 per clock per SM; packed f16x2/bf16x2 ex2 give the same 32
# results per clock).  MEASURED_PEAKS.json has no exp entry, so this figure is
# the denominator of the exp-unit roofline, at the maximum SM clock.
EX2_PER_CLK_SM = 32.0
SMS = 152
EXP_PEAK_SOURCE = ("152 SMs x 32 ex2.approx.f32 results/clk/SM (this library's throughput probe on a GB300: "
                   "31.8/clk/SM) x max SM clock from MEASURED_PEAKS.json")


def attn_flops(w: gi.Workload) -> float:
    """Algorithmic flops of one fwd+bwd over all layers: 14 N^2 H d per layer
    (4 N^2 H d forward: QK^T and PV; 10 N^2 H d backward: QK^T again, dO V^T,
    P^T dO, dS^T Q, dS K)."""
    return 14.0 * w.n * w.n * w.heads * w.head_dim * w.layers


def exps(w: gi.Workload) -> float:
    """exp evaluations of one fwd+bwd: N^2 H forward plus N^2 H to recompute P."""
    return 2.0 * w.n * w.n * w.heads * w.layers


def algo_bytes(w: gi.Workload) -> float:
    """HBM bytes of one fwd+bwd per the path's algorithm: the N^2 SPD bytes read
    twice per layer plus the [N][H][d] tensors (fwd: q k v o; bwd: q k v o dO dq
    dk dv) and the fp32 lse/D vectors."""
    e = 4 if w.dtype == "f32" else 2
    nhd = w.n * w.heads * w.head_dim * e
    return w.layers * (2.0 * w.n * w.n + 12 * nhd + 4 * w.n * w.heads * 4)


def workload_config(w: gi.Workload) -> dict:
    return {"workload": f"{w.name}: N={w.n} {w.graph_kind} graph, H={w.heads}, d={w.head_dim}, "
                        f"D={w.D}, layers={w.layers}, kv_block={w.kv_block}",
            "n": w.n, "heads": w.heads, "head_dim": w.head_dim, "D": w.D, "layers": w.layers,
            "kv_block": w.kv_block, "graph": w.graph_kind,
            "l2": "inputs larger than L2: the int8 SPD matrix (N^2 bytes) is re-read every step"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            for ln in open(self.path):
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks not sampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        smax = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# -------------------------------------------------------------- GPU arm

def measured_peaks() -> dict:
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


# Exp-bound kernels: one exp per (query, key, head) per launch.
EXP_KERNELS = ("fwd_tc", "bwd_dq", "bwd_dkdv", "fwd_simt", "bwd_rows_simt", "bwd_cols_simt")

# DRAM bytes (read + write) per launch of a kernel at a workload, from ncu
# captures of the kernel as it stands (dram__bytes_read.sum + dram__bytes_write.sum);
# the capture summaries live under profiles/.  For a kernel launched more than once
# per layer (bwd_dkdv: the full wave, 179.953 MB, and the split tail, 132.676 MB)
# the entry is the mean over the layer's launches, like the work per launch.  A
# kernel changed since its capture has no entry (its traffic is reported as null).
DRAM_BYTES = {("fwd_tc", "ba64x256"): 295.499e6, ("bwd_dq", "ba64x256"): 318.958e6,
              ("bwd_dkdv", "ba64x256"): 156.315e6, ("spd_bfs", "ba64x256"): 214.420e6}


def kernel_roofline(name: str, w: gi.Workload, ms: float, exp_peak: float, hbm_peak: float,
                    launches_per_layer: float = 1.0) -> dict:
    """Roofline of one kernel: algorithmic work per launch / measured launch time.

    An exp-bound kernel evaluates one exp per (query, key, head) of a layer; when
    it takes several launches per layer (the dk/dv kernel's full waves and split
    tail) the work per launch is the layer's N^2 H over its launches, and `ms` the
    mean launch time, so work / time is the layer's exps over the kernel's time."""
    t = ms * 1e-3
    traffic = DRAM_BYTES.get((name, w.name))
    if name in EXP_KERNELS:
        work = float(w.n) * w.n * w.heads / launches_per_layer     # exps per launch
        return {"kernel": name, "bound": "exp", "achieved": round(work / t / 1e12, 4),
                "peak": round(exp_peak / 1e12, 3), "unit": "Texp/s",
                "frac": round(work / t / exp_peak, 4), "traffic": traffic,
                "work_per_launch": work, "ms_per_launch": round(ms, 4),
                "launches_per_layer": launches_per_layer, "peak_source": EXP_PEAK_SOURCE}
    # anything else is taken as bound by HBM on its output (the N^2 bucket bytes)
    work = float(w.n) * w.n
    return {"kernel": name, "bound": "hbm", "achieved": round(work / t / 1e9, 2),
            "peak": round(hbm_peak / 1e9, 1), "unit": "GB/s", "frac": round(work / t / hbm_peak, 4),
            "traffic": traffic, "work_per_launch": work, "ms_per_launch": round(ms, 4),
            "peak_source": "MEASURED_PEAKS.json hbm_gbs"}


def max_over_ranks(values, world: int, device) -> list:
    """Each rank's times -> their maximum over the ranks (the job lasts as long as
    its slowest replica); a no-op on one rank."""
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_tflops(flops_per_step: float, steps: int, ms: float, world: int) -> float:
    """Replicas only: every rank runs the whole workload, so the job's work is
    world x the per-rank work, over the slowest rank's time."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def run_gpu(args, w: gi.Workload, rank: int, world: int) -> dict | None:
    import torch
    import graph_transformer_attention_gb300 as gt
    from graph_transformer_attention_gb300 import build as gtb

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(gt.library_path()):
        gtb.build()
    if world > 1:
        torch.distributed.barrier()
    gt.load_library()
    stream = torch.cuda.current_stream()

    g = gi.config_graph(w)
    layers = [gi.config_layer_tensors(w, li) for li in range(w.layers)]
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dt_code = gt.GT_BF16 if w.dtype == "bf16" else gt.GT_F32

    # pinned host copies for the end-to-end measurement
    h_ip = torch.from_numpy(g.indptr).pin_memory()
    h_ix = torch.from_numpy(g.indices).pin_memory()
    h_layers = [{k: torch.from_numpy(x[k]).to(tdt if k != "T" else torch.float32).pin_memory()
                 for k in ("q", "k", "v", "dO", "T")} for x in layers]
    d_ip, d_ix = h_ip.to(dev), h_ix.to(dev)
    d_layers = [{k: t.to(dev) for k, t in hl.items()} for hl in h_layers]
    n, H, d = w.n, w.heads, w.head_dim
    spd = torch.empty((n, gt.spd_ld(n)), dtype=torch.int8, device=dev)
    ws_spd = torch.empty(gt.gt_spd_workspace_size(n, g.nnz, w.D), dtype=torch.uint8, device=dev)
    ws_attn = torch.empty(max(256, gt.gt_bias_attn_workspace_size(dt_code, n, H, d, w.kv_block)),
                          dtype=torch.uint8, device=dev)
    outs = [dict(o=torch.empty((n, H, d), dtype=tdt, device=dev),
                 lse=torch.empty((H, n), dtype=torch.float32, device=dev),
                 dq=torch.empty((n, H, d), dtype=tdt, device=dev),
                 dk=torch.empty((n, H, d), dtype=tdt, device=dev),
                 dv=torch.empty((n, H, d), dtype=tdt, device=dev),
                 dT=torch.empty((H, w.nb), dtype=torch.float32, device=dev))
            for _ in range(w.layers)]
    h_outs = [{k: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k, t in oo.items()
               if k in ("o", "dq", "dk", "dv", "dT")} for oo in outs]

    # a second set of device inputs and outputs: the end-to-end steps alternate
    # between the two, so that one step's copies overlap its neighbour's compute
    sets = [dict(ip=d_ip, ix=d_ix, layers=d_layers, outs=outs),
            dict(ip=torch.empty_like(d_ip), ix=torch.empty_like(d_ix),
                 layers=[{k: torch.empty_like(t) for k, t in dl.items()} for dl in d_layers],
                 outs=[{k: torch.empty_like(t) for k, t in oo.items()} for oo in outs])]

    def step(ev=None, S=None):
        # ev: [spd0, spd1, fwd0, fwd1, bwd0, bwd1] events around the parts of layer 0
        S = S or sets[0]
        if ev:
            ev[0].record(stream)
        gt.gt_spd_build(S["ip"], S["ix"], n, w.D, out=spd, workspace=ws_spd)
        if ev:
            ev[1].record(stream)
        for li in range(w.layers):
            x, oo = S["layers"][li], S["outs"][li]
            if ev and li == 0:
                ev[2].record(stream)
            gt.gt_bias_attn_fwd(x["q"], x["k"], x["v"], spd, x["T"], kv_block=w.kv_block,
                                out=oo["o"], lse=oo["lse"], workspace=ws_attn)
            if ev and li == 0:
                ev[3].record(stream)
                ev[4].record(stream)
            gt.gt_bias_attn_bwd(x["q"], x["k"], x["v"], oo["o"], x["dO"], oo["lse"], spd, x["T"],
                                dq=oo["dq"], dk=oo["dk"], dv=oo["dv"], dT=oo["dT"],
                                workspace=ws_attn)
            if ev and li == 0:
                ev[5].record(stream)

    # end-to-end steps: every step copies its inputs in from pinned host memory and
    # its results out; step k's inputs go in on one copy stream while step k - 1
    # computes, and its results go out on another while step k + 1 computes
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(k_steps):
        for kk in range(k_steps):
            si = kk % 2
            S = sets[si]
            with torch.cuda.stream(h2d_s):
                if kk >= 2:
                    h2d_s.wait_event(ev_done[si])          # step kk - 2 has finished reading set si
                S["ip"].copy_(h_ip, non_blocking=True)
                S["ix"].copy_(h_ix, non_blocking=True)
                for li in range(w.layers):
                    for k in S["layers"][li]:
                        S["layers"][li][k].copy_(h_layers[li][k], non_blocking=True)
                ev_in[si].record(h2d_s)
            stream.wait_event(ev_in[si])
            if kk >= 2:
                stream.wait_event(ev_out[si])              # step kk - 2's results are out
            step(S=S)
            ev_done[si].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[si])
                for li in range(w.layers):
                    for k, t in h_outs[li].items():
                        t.copy_(S["outs"][li][k], non_blocking=True)
                ev_out[si].record(d2h_s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    gt.gt_check_device_status()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # device-timed region: K steps, per-part events on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gt.gt_kernel_stats_reset(False)          # count the library's launches in the timed region
    with ClockSampler(dev.index) as clk:
        barrier()
        t0.record(stream)
        for s in range(args.steps):
            step(evs[s])
        t1.record(stream)
        barrier()
    ms_total = t0.elapsed_time(t1)
    clocks = clk.summary()
    gt.gt_check_device_status()
    launches = sum(c for c, _ in gt.gt_kernel_stats().values())
    part_ms = {"spd": float(np.mean([e[0].elapsed_time(e[1]) for e in evs])),
               "fwd": float(np.mean([e[2].elapsed_time(e[3]) for e in evs])),
               "bwd": float(np.mean([e[4].elapsed_time(e[5]) for e in evs]))}

    # per-kernel device time: a few more steps with every launch bracketed by
    # CUDA events on its stream (kept out of the timed region above)
    n_kt = min(args.steps, 3)
    gt.gt_kernel_stats_reset(True)
    for _ in range(n_kt):
        step()
    torch.cuda.synchronize()
    kstats = gt.gt_kernel_stats()
    gt.gt_kernel_stats_reset(False)
    kernels = {name: {"launches_per_step": c / n_kt, "ms_per_launch": ms / c}
               for name, (c, ms) in kstats.items()}

    # end-to-end through the public API, host buffers in and out (host clock
    # around the K steps: every step's copies in and out are inside)
    e2e_run(2)
    barrier()
    e0 = time.perf_counter()
    e2e_run(args.steps)
    barrier()
    e2e_ms = (time.perf_counter() - e0) * 1e3

    # the same, one step at a time with nothing overlapped: inputs in, the step,
    # results out, synchronised (the latency of one step through the API)
    lat = []
    S0 = sets[0]
    for _ in range(args.steps):
        barrier()
        l0 = time.perf_counter()
        S0["ip"].copy_(h_ip, non_blocking=True)
        S0["ix"].copy_(h_ix, non_blocking=True)
        for li in range(w.layers):
            for k in S0["layers"][li]:
                S0["layers"][li][k].copy_(h_layers[li][k], non_blocking=True)
        step(S=S0)
        for li in range(w.layers):
            for k, t in h_outs[li].items():
                t.copy_(S0["outs"][li][k], non_blocking=True)
        torch.cuda.synchronize()
        lat.append((time.perf_counter() - l0) * 1e3)

    h2d = h_ip.numel() * 8 + h_ix.numel() * 4 + sum(t.numel() * t.element_size()
                                                    for hl in h_layers for t in hl.values())
    d2h = sum(t.numel() * t.element_size() for ho in h_outs for t in ho.values())

    ms_total, e2e_ms = max_over_ranks([ms_total, e2e_ms], world, dev)
    if rank != 0:
        return None

    ms_step = ms_total / args.steps
    flops = attn_flops(w)
    value = whole_job_tflops(flops, args.steps, ms_total, world)
    e2e_value = whole_job_tflops(flops, args.steps, e2e_ms, world)
    peaks = measured_peaks()
    clk_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    exp_peak = SMS * EX2_PER_CLK_SM * clk_mhz * 1e6           # exps / s
    tensor_peak = float(peaks.get("bf16_tflops_sustained", 1700.0)) * 1e12
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0)) * 1e9
    # dominant kernel: largest device time per step
    dom = max(kernels, key=lambda k: kernels[k]["launches_per_step"] * kernels[k]["ms_per_launch"])
    roof = kernel_roofline(dom, w, kernels[dom]["ms_per_launch"], exp_peak, hbm_peak,
                           launches_per_layer=kernels[dom]["launches_per_step"] / w.layers)
    # whole-path roofline: the slowest of tensor pipe, HBM and exp unit
    t_attn = (part_ms["fwd"] + part_ms["bwd"]) * w.layers * 1e-3
    t_roof = max(flops / tensor_peak, algo_bytes(w) / hbm_peak, exps(w) / exp_peak)
    return {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded random graph and N(0,1) tensors)",
        "config": workload_config(w),
        "parts_ms": {k: round(v, 4) for k, v in part_ms.items()},
        "node_pairs_per_s": {"spd": round(n * n / (part_ms["spd"] * 1e-3), 1),
                             "attn_fwd_bwd": round(n * n * w.layers / t_attn, 1)},
        "roofline": roof,
        "kernels_ms": {k: {"launches_per_step": round(v["launches_per_step"], 3),
                           "ms_per_launch": round(v["ms_per_launch"], 4)} for k, v in kernels.items()},
        "path_roofline": {"t_roof_ms": round(t_roof * 1e3, 4), "t_attn_ms": round(t_attn * 1e3, 4),
                          "frac": round(t_roof / t_attn, 4) if t_attn > 0 else None,
                          "bound": "exp unit (MUFU)"},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "pipelined": "step k's copies overlap steps k - 1 and k + 1 (two buffer sets)",
                "latency_ms_per_step": round(float(np.median(lat)), 4),
                "latency_note": "one step alone: copies in, SPD build, fwd, bwd, copies out, synchronised "
                                "(median of the timed steps, host clock)"},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "memory": memory_line(w, dev),
        "cpu_baseline": None,
        "configs": extra_configs(args, w, dev, world, exp_peak, tensor_peak, hbm_peak),
    }


def extra_configs(args, w: gi.Workload, dev, world: int, exp_peak: float, tensor_peak: float,
                  hbm_peak: float) -> dict | None:
    """Every other workload timed the same way after the headline (one GPU only;
    --no-extra-configs skips them)."""
    if world > 1 or args.no_extra_configs:
        return None
    out = {}
    for ci, wc in sorted(gi.CONFIGS.items()):
        if wc.name == w.name:
            continue
        steps = 3 if wc.layers > 1 or wc.n >= 32768 else 10
        out[wc.name] = measure_config(wc, dev, steps, 2, exp_peak, tensor_peak, hbm_peak)
    return out


def measure_config(w: gi.Workload, dev, steps: int, warmup: int, exp_peak: float, tensor_peak: float,
                   hbm_peak: float) -> dict:
    """Device time of one step (SPD build + fwd + bwd of every layer, inputs
    resident) of another workload, with per-part CUDA events on the stream."""
    import torch
    import graph_transformer_attention_gb300 as gt
    stream = torch.cuda.current_stream()
    g = gi.config_graph(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ip, ix = torch.from_numpy(g.indptr).to(dev), torch.from_numpy(g.indices).to(dev)
    layers = []
    for li in range(w.layers):
        x = gi.config_layer_tensors(w, li)
        layers.append({k: torch.from_numpy(x[k]).to(dev).to(tdt if k != "T" else torch.float32)
                       for k in ("q", "k", "v", "dO", "T")})
    n, H, d = w.n, w.heads, w.head_dim
    code = gt.GT_BF16 if w.dtype == "bf16" else gt.GT_F32
    spd = torch.empty((n, gt.spd_ld(n)), dtype=torch.int8, device=dev)
    ws_spd = torch.empty(gt.gt_spd_workspace_size(n, g.nnz, w.D), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(256, gt.gt_bias_attn_workspace_size(code, n, H, d, w.kv_block)), dtype=torch.uint8,
                     device=dev)
    outs = [dict(o=torch.empty((n, H, d), dtype=tdt, device=dev), lse=torch.empty((H, n), device=dev),
                 dq=torch.empty((n, H, d), dtype=tdt, device=dev), dk=torch.empty((n, H, d), dtype=tdt, device=dev),
                 dv=torch.empty((n, H, d), dtype=tdt, device=dev), dT=torch.empty((H, w.nb), device=dev))
            for _ in range(w.layers)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]

    def step(e=None):
        if e:
            e[0].record(stream)
        gt.gt_spd_build(ip, ix, n, w.D, out=spd, workspace=ws_spd)
        if e:
            e[1].record(stream)
        for li, x in enumerate(layers):
            oo = outs[li]
            gt.gt_bias_attn_fwd(x["q"], x["k"], x["v"], spd, x["T"], kv_block=w.kv_block, out=oo["o"],
                                lse=oo["lse"], workspace=ws)
            if e and li == 0:
                e[2].record(stream)
            gt.gt_bias_attn_bwd(x["q"], x["k"], x["v"], oo["o"], x["dO"], oo["lse"], spd, x["T"], dq=oo["dq"],
                                dk=oo["dk"], dv=oo["dv"], dT=oo["dT"], workspace=ws)
        if e:
            e[3].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for sidx in range(steps):
        step(ev[sidx])
    t1.record(stream)
    torch.cuda.synchronize()
    gt.gt_check_device_status()
    ms_step = t0.elapsed_time(t1) / steps
    spd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    attn_ms = float(np.mean([e[1].elapsed_time(e[3]) for e in ev]))
    flops = attn_flops(w)
    t_roof = max(flops / tensor_peak, algo_bytes(w) / hbm_peak, exps(w) / exp_peak)
    return {"workload": workload_config(w)["workload"], "ms_per_step": round(ms_step, 4),
            "tflops": round(flops / (ms_step * 1e-3) / 1e12, 3), "spd_ms": round(spd_ms, 4),
            "attn_fwd_bwd_ms": round(attn_ms, 4),
            "path_frac": round(t_roof / (attn_ms * 1e-3), 4) if attn_ms > 0 else None,
            "path_bound": "exp unit" if w.dtype == "bf16" else "exp unit (fp32 CUDA-core path: not its bound)",
            "steps": steps, "warmup": warmup}


def memory_line(w: gi.Workload, dev) -> dict:
    """Model bytes of one layer's forward + backward, blockwise (this library) and
    materialised (N x N per head), and the process's measured peak."""
    import torch
    from graph_transformer_attention_gb300 import memory as M
    blk = M.blockwise_layer_bytes(w.n, w.heads, w.head_dim, w.nb, w.dtype, w.kv_block)
    mat = M.materialised_layer_bytes(w.n, w.heads, w.head_dim, w.dtype)
    return {"model_blockwise_layer_bytes": int(blk["peak"]),
            "model_materialised_layer_bytes_min": int(mat["peak_min"]),
            "process_peak_allocated_bytes": int(torch.cuda.max_memory_allocated(dev))}


# ------------------------------------------------- the GT layer stack (Fig. 8)

LAYER_METRIC = "GT layer stack (pre-LN, QKV/O projections, GELU FFN, biased attention) fwd+bwd TFLOP/s on 1 GB300"
LAYER_DENSE_FLOPS_PER_ROW = 3 * 2 * 64 * (3 * 64 + 64 + 64 + 64)   # fwd + bwd (dx and dW) of the four matmuls


def run_layer(args, w: gi.Workload, rank: int, world: int) -> dict | None:
    """One step = SPD build + every layer's forward and backward (gt_layer_fwd /
    gt_layer_bwd), layers independent (each with its own seeded weights, x, dy)."""
    import torch
    import graph_transformer_attention_gb300 as gt
    from graph_transformer_attention_gb300 import build as gtb

    if w.heads != 8 or w.head_dim != 8 or w.dtype != "bf16":
        raise SystemExit(f"--model gt-layer needs a bf16 workload with 8 heads of width 8 (not {w.name})")
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(gt.library_path()):
        gtb.build()
    if world > 1:
        torch.distributed.barrier()
    gt.load_library()
    stream = torch.cuda.current_stream()
    g = gi.config_graph(w)
    n = w.n
    d_ip, d_ix = torch.from_numpy(g.indptr).to(dev), torch.from_numpy(g.indices).to(dev)
    spd = torch.empty((n, gt.spd_ld(n)), dtype=torch.int8, device=dev)
    ws_spd = torch.empty(gt.gt_spd_workspace_size(n, g.nnz, w.D), dtype=torch.uint8, device=dev)
    ws = torch.empty(gt.gt_layer_workspace_size(n), dtype=torch.uint8, device=dev)
    layers = []
    for li in range(w.layers):
        p = gi.make_gt_layer_params(64, 64, w.nb, 8, seed=w.tensor_seed(li))
        io = gi.make_gt_layer_io(n, 64, seed=w.tensor_seed(li) + 50)
        layers.append(dict(params={k: torch.from_numpy(v).to(dev) for k, v in p.items() if k != "T"},
                           T=torch.from_numpy(p["T"]).to(dev), x=torch.from_numpy(io["x"]).to(dev),
                           dy=torch.from_numpy(io["dy"]).to(dev)))

    def step():
        gt.gt_spd_build(d_ip, d_ix, n, w.D, out=spd, workspace=ws_spd)
        for L in layers:
            y, saved = gt.gt_layer_fwd(L["x"], L["params"], spd, L["T"], workspace=ws)
            gt.gt_layer_bwd(L["x"], L["params"], spd, L["T"], saved, L["dy"], workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    gt.gt_check_device_status()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gt.gt_kernel_stats_reset(False)
    with ClockSampler(dev.index) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    ms_total = t0.elapsed_time(t1)
    gt.gt_check_device_status()
    launches = sum(c for c, _ in gt.gt_kernel_stats().values())
    gt.gt_kernel_stats_reset(True)
    for _ in range(min(args.steps, 3)):
        step()
    torch.cuda.synchronize()
    kst = gt.gt_kernel_stats()
    gt.gt_kernel_stats_reset(False)
    nk = min(args.steps, 3)
    kernels = {k: {"launches_per_step": c / nk, "ms_per_launch": t / c} for k, (c, t) in kst.items() if c}
    (ms_total,) = max_over_ranks([ms_total], world, dev)
    if rank != 0:
        return None
    flops = w.layers * (14.0 * n * n * 8 * 8 + LAYER_DENSE_FLOPS_PER_ROW * n)
    around = ("layer_ln_qkv", "layer_out_ffn", "layer_ffn_bwd", "layer_qkv_bwd", "layer_grad_sum")
    per_step = {k: v["launches_per_step"] * v["ms_per_launch"] for k, v in kernels.items()}
    return {
        "metric": LAYER_METRIC, "value": round(whole_job_tflops(flops, args.steps, ms_total, world), 3),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 attention; tf32 projections and bf16 weight-gradient products around it, fp32 accumulation",
        "data": "synthetic (seeded random graph, weights, x and dy)",
        "config": {**workload_config(w), "model": "GT encoder layer, 8 heads, hidden 64, FFN 64"},
        "kernels_ms": {k: {"launches_per_step": round(v["launches_per_step"], 3),
                           "ms_per_launch": round(v["ms_per_launch"], 4)} for k, v in kernels.items()},
        "around_attention_ms_per_step": round(sum(per_step.get(k, 0.0) for k in around), 4),
        "around_attention_ms_per_layer": round(sum(per_step.get(k, 0.0) for k in around) / w.layers, 4),
        "gpu_launches": int(launches), "clocks": clk.summary(),
    }


# --------------------------------------------------------- CPU oracle arm

def oracle_sample(w: gi.Workload, rows_per_step: int, seed: int = 0):
    """Time the fp64 oracle on a bounded sample: forward, dq and dT over
    `rows_per_step` rows plus dk, dv over as many columns, on the full graph
    (the SPD matrix is built once, outside the timing).  Returns (seconds,
    flops credited = 14 R N H d, threads)."""
    from oracle import oracle as O
    g = gi.config_graph(w)
    spd = O.spd(g.n, g.indptr, g.indices, w.D)
    x = gi.config_layer_tensors(w, 0)
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.n, rows_per_step, replace=False)).astype(np.int32)
    nt = O.default_threads()
    t0 = time.perf_counter()
    o_r, lse_r = O.attn_fwd(x["q"], x["k"], x["v"], spd, x["T"], rows=rows, nthreads=nt)
    Dv_rows = (o_r * x["dO"][rows].astype(np.float64)).sum(-1).T
    lse_full = np.zeros((w.heads, w.n)); Dv_full = np.zeros((w.heads, w.n))
    lse_full[:, rows] = lse_r; Dv_full[:, rows] = Dv_rows
    O.attn_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"], lse_full, Dv_full, rows=rows,
               want_dkdv=False, nthreads=nt)
    # dk/dv for R columns: the oracle's cost does not depend on the values, so the
    # lse/D of unsampled rows are left as placeholders and the results discarded
    O.attn_bwd(x["q"], x["k"], x["v"], x["dO"], spd, x["T"], lse_full, Dv_full,
               cols=rows, want_dq=False, want_dT=False, nthreads=nt)
    dt = time.perf_counter() - t0
    flops = 14.0 * rows_per_step * w.n * w.heads * w.head_dim
    return dt, flops, nt


def run_reference(args, w: gi.Workload) -> dict:
    rows = int(args.oracle_rows) or max(8, w.n // 8)
    dts, fl, nt = [], 0.0, 1
    for s in range(args.warmup + args.steps):
        dt, fl, nt = oracle_sample(w, rows, seed=s)
        if s >= args.warmup:
            dts.append(dt)
    tot = sum(dts)
    value = fl * len(dts) / tot / 1e12
    sample = (f"{rows} of {w.n} rows: forward, dq and dT over those rows plus dk, dv over {rows} "
              f"columns, of layer 0 on the full graph; flops credited 14*R*N*H*d")
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / len(dts) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded random graph and N(0,1) tensors)",
        "config": workload_config(w), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gt", "reference"], default="gt")
    ap.add_argument("--config", type=int, default=4, choices=sorted(gi.CONFIGS))
    ap.add_argument("--oracle-rows", type=int, default=0,
                    help="rows (and columns) the CPU oracle processes per sample "
                         "(default: N/2 for the baseline line, N/8 per reference step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time only the chosen workload (by default the others follow it, in 'configs')")
    ap.add_argument("--model", choices=["attention", "gt-layer"], default="attention",
                    help="attention: the biased-attention path (default); gt-layer: the whole encoder "
                         "layer around it (default workload then ba6800x16)")
    args = ap.parse_args(argv)
    if args.model == "gt-layer" and "--config" not in (argv if argv is not None else sys.argv):
        args.config = 3
    w = gi.CONFIGS[args.config]
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    if args.model == "gt-layer":
        line = run_layer(args, w, rank, world)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
        return 0
    line = run_gpu(args, w, rank, world)
    if rank == 0 and line is not None:
        if world == 1 and not args.no_cpu_baseline:
            rows = args.oracle_rows or max(8, w.n // 2)
            dt, fl, nt = oracle_sample(w, rows)
            line["cpu_baseline"] = {
                "value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
                "sample": f"{rows} of {w.n} rows (fwd, dq, dT) and as many columns (dk, dv) of "
                          f"layer 0; flops credited 14*R*N*H*d; {dt:.1f} s wall"}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
