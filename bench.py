#!/usr/bin/env python
"""Benchmark of the layout-folding hot path on GB300.

Headline line (one JSON line on rank 0): TFLOP/s of ``gemm_nt`` on the NT
projection workload -- X bf16[384,2,13824] viewed [768,13824], W
bf16[5120,13824] in its stored layout, out bf16[384,2,5120] -- one step = one
``gemm_nt`` call on inputs resident in HBM, with L2 flushed (a 256 MiB write,
then a 256 MiB read) between steps and each step timed with CUDA events on the
launching stream.  The line also carries ``roofline`` (the headline kernel
against the measured bf16 peak, with its DRAM traffic from the committed ncu
capture), ``e2e`` (the same call with host buffers and the copies inside the
timed region), ``clocks`` and ``cpu_baseline``.  Under "paths": the K=1 product
(the page's [64,4096] and 2 GiB out), the RoPE segment and the fp8 dual-layout
cast (bandwidth-bound legs, run first), the fused GEMM + cross-entropy with
gradient (4096x32768x4096, one pass), the loss-only large-vocabulary case
(8192x128256x4096) with the unfused comparison, the large-vocabulary gradient
(two passes), the other operand layouts, batched and strided views, and the
skinny swapped-operand GEMM.  Under "paths.library": the same workloads computed
by PyTorch's own GPU operators (cuBLAS matmuls, eager elementwise kernels),
timed the same way, with the ratio of their time to this library's.

``--impl reference`` times the CPU oracle (fp64, plain loops) on a bounded
sample of the same workload, on this machine's host cores.

Multi-GPU: the path has no exchange step, so N ranks run N independent
replicas (weak scaling, no data-path collective); value = all ranks' FLOPs /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TFLOP/s and % of dense-BF16 peak for gemm_nt and gemm_nt_xent; K=1 GB/s"
L2_FLUSH_BYTES = 256 << 20
LAUNCH_SHADOW_CYCLES = 200_000   # ~0.1 ms of device-side delay before each timed step
# the files the headline kernel's device code is compiled from (host-only declarations excluded)
KERNEL_SOURCES = ["layout_folding_gb300/csrc/gemm_nt_pair.cu", "layout_folding_gb300/csrc/lf_gemm_common.cuh",
                  "layout_folding_gb300/csrc/lf_ptx.cuh", "layout_folding_gb300/csrc/lf_kernel_params.h"]
# source files whose hash a recorded DRAM figure is tied to, per kernel
TRAFFIC_SOURCES = {
    "k_gemm_nt_pair<EPI_STORE>": KERNEL_SOURCES,
    "k_fp8_cast_dual_v16": ["layout_folding_gb300/csrc/fp8_cast.cu"],
    "k_rope_cos_sin_v8": ["layout_folding_gb300/csrc/rope.cu"],
}
HEADLINE_KERNEL = "k_gemm_nt_pair<EPI_STORE>"   # CTA-pair tiles, stream-K split (chosen automatically here)


# ---------------------------------------------------------------- helpers

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def reduce_over_ranks(value: float, op: str) -> float:
    """max or sum of a float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("kernel_hash") != kernel_hash(TRAFFIC_SOURCES.get(kernel)):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="lf_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = max((num(r[2]) for r in rows if num(r[2]) is not None), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [v for v in sm if smax and v >= 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ our arm

class Timer:
    """Per-step CUDA events on the launching stream, L2 flushed between steps."""

    def __init__(self, torch, stream):
        self.torch = torch
        self.stream = stream
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.clean_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.clean_out = torch.empty((), dtype=torch.float32, device="cuda")

    def run(self, fn, steps, warmup, flush=True, counter=None):
        """Returns per-step ms; if `counter` is given, also the number of
        library launches inside the timed steps."""
        torch = self.torch
        # warm-up steps are the timed steps without events: the flush buffers'
        # first use (page mapping) then falls outside the timed region
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                if flush:
                    self.flush_buf.fill_(1.0)
                    torch.sum(self.clean_buf, dim=0, out=self.clean_out)
                torch.cuda._sleep(LAUNCH_SHADOW_CYCLES)
                fn()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        c0 = counter() if counter else 0
        evs = []
        with torch.cuda.stream(self.stream):
            for _ in range(steps):
                if flush:
                    # evict L2 by writing a buffer larger than it, then read a
                    # second one so the write-backs of the first happen here,
                    # not inside the timed call
                    self.flush_buf.fill_(1.0)
                    torch.sum(self.clean_buf, dim=0, out=self.clean_out)
                # keep the device busy while the host issues the timed call, so
                # the start event is not followed by an idle gap (host launch
                # latency is not kernel time; the e2e figure carries it)
                torch.cuda._sleep(LAUNCH_SHADOW_CYCLES)
                s = torch.cuda.Event(enable_timing=True)
                e = torch.cuda.Event(enable_timing=True)
                s.record(self.stream)
                fn()
                e.record(self.stream)
                evs.append((s, e))
        torch.cuda.synchronize()
        launches = (counter() - c0) if counter else None
        barrier()
        torch.cuda.synchronize()
        times = [s.elapsed_time(e) for s, e in evs]   # ms per step
        return (times, launches) if counter else times


def headline_config(wl, world):
    """The headline workload's `config`, identical in both arms' lines."""
    return {"workload": "nt_projection", "path": "gemm_nt", "M": wl.M, "N": wl.N, "K": wl.K,
            "x_shape": list(wl.x_shape), "accumulate": "fp32", "out": "bf16",
            "l2": "GPU arm: flushed between steps outside the timed events (a 256 MiB write, then a 256 MiB "
                  "read that retires the write's dirty lines; L2 is 129 MB); CPU arm: not applicable",
            "parallelism": "replicas" if world > 1 else "single"}


def run_ours(args, rank, world, local_rank):
    import torch

    import layout_folding_gb300 as lf
    from layout_folding_gb300 import synthetic

    torch.cuda.set_device(local_rank)
    lf.lib()
    if args.no_cooperative:
        lf.set_cooperative(False)
    lf.set_tile_schedule({"auto": -1, "fixed": 0, "claimed": 1}[args.tile_schedule])
    peaks = load_peaks()
    stream = torch.cuda.Stream()
    timer = Timer(torch, stream)

    # ---------------- headline: gemm_nt, NT projection
    wl = synthetic.WORKLOADS["nt_projection"]
    inp = synthetic.make_workload("nt_projection")
    x_h, w_h = inp["x"].pin_memory(), inp["w"].pin_memory()
    x, w = x_h.to("cuda"), w_h.to("cuda")
    out = torch.empty(384, 2, wl.N, dtype=torch.bfloat16, device="cuda")
    flops = 2.0 * wl.M * wl.N * wl.K

    def step():
        lf.gemm_nt(x, w, out, stream=stream)

    with ClockSampler(local_rank) as clk:
        times, launches = timer.run(step, args.steps, args.warmup, counter=lf.launch_count)
    lf.check_device_error(stream)
    total_ms = reduce_over_ranks(sum(times), "max")
    ms_per_step = total_ms / args.steps
    value = reduce_over_ranks(flops * args.steps, "sum") / (total_ms * 1e-3) / 1e12
    kernel_ms = statistics.mean(times)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    traffic = recorded_traffic(HEADLINE_KERNEL, "nt_projection")

    # ---------------- e2e: host buffers in, result out, through the same C-ABI call
    out_h = torch.empty(out.shape, dtype=torch.bfloat16, pin_memory=True)
    xs = torch.empty_like(x)
    ws_ = torch.empty_like(w)

    def e2e_step():
        xs.copy_(x_h, non_blocking=True)
        ws_.copy_(w_h, non_blocking=True)
        lf.gemm_nt(xs, ws_, out, stream=stream)
        out_h.copy_(out, non_blocking=True)

    def e2e_in_stream():
        with torch.cuda.stream(stream):
            e2e_step()
    e2e_times = timer.run(e2e_in_stream, max(3, args.steps // 2), 2, flush=False)
    e2e_ms = reduce_over_ranks(sum(e2e_times), "max") / len(e2e_times)
    e2e_value = reduce_over_ranks(flops, "sum") / (e2e_ms * 1e-3) / 1e12
    del xs, ws_

    paths = {}
    if not args.headline_only:
        paths = secondary_paths(args, torch, lf, synthetic, timer, stream, peaks)
        lib = paths.get("library")
        if lib:
            # time of PyTorch's operators / time of this library's, per workload
            ours = {"gemm_nt_projection": kernel_ms, "gemm_skinny_m64": paths.get("skinny_m64", {}).get("ms"),
                    "xent_grad": paths.get("xent_grad", {}).get("ms"),
                    "k1_scaled": paths.get("k1_scaled", {}).get("ms"),
                    "rope_scaled": paths.get("rope_scaled", {}).get("ms"),
                    "fp8_cast_scaled": paths.get("fp8_cast_scaled", {}).get("ms")}
            for k, v in lib.items():
                if isinstance(v, dict) and ours.get(k):
                    v["speedup_of_this_library"] = round(v["ms"] / ours[k], 3)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_gemm(inp["x"].reshape(wl.M, wl.K), inp["w"], wl, budget_s=args.cpu_budget)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)*0.02 bf16; no dataset)",
        "config": headline_config(wl, world),
        "timing": "CUDA events around each call on the launching stream; a 0.1 ms device delay "
                  "precedes each start event so host launch latency is not counted",
        "cooperative_launches": not args.no_cooperative,
        "tile_schedule": args.tile_schedule,
        "pct_of_peak": round(100.0 * achieved / peak, 1),
        "roofline": {"bound": "tensor", "kernel": HEADLINE_KERNEL, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": "bf16 burst (%s)" % peaks["source"], "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": (wl.M * wl.K + wl.N * wl.K + wl.M * wl.N) * 2},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": (x.numel() + w.numel()) * 2, "d2h_bytes_per_step": out.numel() * 2,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "paths": paths,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def grad_form(want_grad, launches_per_call):
    """The cross-entropy form a call took, from its launch count: loss only
    (partials + combine), one pass, exp pass + rescale, or recompute."""
    if not want_grad:
        return "loss_only"
    return {1: "one_pass", 2: "exp_rescale", 3: "recompute"}.get(int(round(launches_per_call)), "unknown")


def xent_fractions(flops, executed, ms, peaks):
    """Fractions of the bf16 peak for a cross-entropy leg.  Each call is timed
    alone between L2 flushes (milliseconds, not a seconds-long loop), so the
    burst peak is the denominator; the sustained one is reported beside it."""
    burst, sustained = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    alg, exe = flops / ms / 1e9, executed / ms / 1e9
    return {"pct_of_burst_algorithmic": round(100 * alg / burst, 1),
            "pct_of_burst_executed": round(100 * exe / burst, 1),
            "pct_of_sustained_algorithmic": round(100 * alg / sustained, 1),
            "pct_of_sustained_executed": round(100 * exe / sustained, 1),
            "peak_burst": burst, "peak_sustained": sustained, "peak_source": peaks["source"]}


def secondary_paths(args, torch, lf, synthetic, timer, stream, peaks):
    res = {}
    steps = max(3, min(args.steps, 10))
    want = {p.strip() for p in args.paths.split(",") if p.strip()}
    # The tiny oracle-sized case (X [64,128], W [256,128]): parity is its
    # point; its latency is reported here (median of the timed calls).
    if "tiny" in want:
        inp = synthetic.make_workload("tiny")
        x, w, lab = inp["x"].to("cuda"), inp["w"].to("cuda"), inp["labels"].to("cuda")
        out = torch.empty(64, 256, dtype=torch.bfloat16, device="cuda")
        loss = torch.empty(64, dtype=torch.float32, device="cuda")
        grad = torch.empty(64, 256, dtype=torch.bfloat16, device="cuda")
        t_nt = timer.run(lambda: lf.gemm_nt(x, w, out, stream=stream), max(steps, 10), 3)
        t_xg, n_xg = timer.run(lambda: lf.gemm_nt_xent(x, w, lab, loss=loss, grad=grad, stream=stream),
                               max(steps, 10), 3, counter=lf.launch_count)
        t_xl = timer.run(lambda: lf.gemm_nt_xent(x, w, lab, loss=loss, stream=stream), max(steps, 10), 3)
        lf.check_device_error(stream)
        res["tiny"] = {"M": 64, "N": 256, "K": 128, "gemm_nt_us": round(1e3 * statistics.median(t_nt), 2),
                       "gemm_nt_xent_grad_us": round(1e3 * statistics.median(t_xg), 2),
                       "gemm_nt_xent_loss_us": round(1e3 * statistics.median(t_xl), 2),
                       "xent_grad_launches": n_xg / max(steps, 10),
                       "what": "latency of one call (median, L2 flushed before each); launch-bound"}
        del x, w, lab, out, loss, grad
    # The bandwidth-bound legs run first: in one process, after the
    # cross-entropy legs' multi-GB allocations had been freed, the 2 GiB K=1
    # write measured 431 us against 360 us run first or in a fresh process
    # (an allocation effect, not a thermal one: a fresh process right after a
    # cross-entropy run measured 360 us too).
    # K=1: the page's [64,1]x[1,4096] (latency regime) and a scaled column count for bandwidth
    a, b = synthetic.k1_operands(64, 4096)
    for label, N in ((("k1_rope", 4096), ("k1_scaled", 1 << 23)) if "k1" in want else ()):
        bb = torch.arange(N, dtype=torch.float32).reshape(1, N) if N != 4096 else b
        ad, bd = a.to("cuda"), bb.to("cuda")
        out = torch.empty(64, N, dtype=torch.float32, device="cuda")

        def step():
            lf.matmul_k1(ad, bd, out, stream=stream)
        times = timer.run(step, max(steps, 10), 3)
        ms = statistics.median(times)
        nbytes = (64 + N + 64 * N) * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[label] = {"M": 64, "N": N, "ms": round(ms, 5), "GB/s": round(gbs, 1),
                      "pct_of_hbm": round(100 * gbs / peaks["hbm_gbs"], 1), "bytes": nbytes}
        del ad, bd, out
    torch.cuda.empty_cache()
    # RoPE segment (K=1 matmul + permute + cat + cos/sin -> bf16): the page's 4096
    # positions, and 2^20 positions (32 sequences of 32768) for bandwidth
    for label, (S, maxp) in ((("rope_page", (4096, 0)), ("rope_scaled", (1 << 20, 32768))) if "rope" in want else ()):
        inv, pos = synthetic.rope_operands(64, S, max_position=maxp)
        inv, pos = inv.to("cuda"), pos.to("cuda")
        co = torch.empty(S, 128, dtype=torch.bfloat16, device="cuda")
        so = torch.empty(S, 128, dtype=torch.bfloat16, device="cuda")

        def step():
            lf.rope_cos_sin(inv, pos, cos_out=co, sin_out=so, stream=stream)
        times = timer.run(step, max(steps, 10), 3)
        ms = statistics.median(times)
        nbytes = 64 * 2 + S * 8 + 2 * S * 128 * 2
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[label] = {"H": 64, "S": S, "ms": round(ms, 5), "GB/s": round(gbs, 1),
                      "pct_of_hbm": round(100 * gbs / peaks["hbm_gbs"], 1), "bytes": nbytes,
                      "angles_per_s": round(S * 64 / (ms * 1e-3), 1),
                      "traffic": recorded_traffic("k_rope_cos_sin_v8", label)}
        del inv, pos, co, so
    # fused fp8 cast, both layouts: the page's 4096 x 4096 and a scaled case larger than L2
    scale = torch.tensor([10.0], dtype=torch.float32, device="cuda")
    for label, (M, K) in ((("fp8_cast_page", (4096, 4096)), ("fp8_cast_scaled", (16384, 16384))) if "fp8" in want
                          else ()):
        x = synthetic.bf16_normal((M, K), 1.0, 15).to("cuda")
        out = torch.empty(M, K, dtype=torch.float8_e4m3fn, device="cuda")
        out_t = torch.empty(K, M, dtype=torch.float8_e4m3fn, device="cuda").t()

        def step():
            lf.fp8_cast_dual(x, scale, out=out, out_t=out_t, stream=stream)
        times = timer.run(step, max(steps, 10), 3)
        ms = statistics.median(times)
        nbytes = M * K * (2 + 1 + 1)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[label] = {"M": M, "K": K, "scale": 10.0, "ms": round(ms, 5), "GB/s": round(gbs, 1),
                      "pct_of_hbm": round(100 * gbs / peaks["hbm_gbs"], 1), "bytes": nbytes,
                      "traffic": recorded_traffic("k_fp8_cast_dual_v16", label)}
        del x, out, out_t
    torch.cuda.empty_cache()
    # "xent" selects all three cross-entropy legs; "xent_grad", "xent_loss" and
    # "xent_grad_large_vocab" one each
    xent_legs = [(name, g) for name, g, tag in (("xent_grad", True, "xent_grad"), ("xent_loss", False, "xent_loss"),
                                                 ("xent_loss", True, "xent_grad_large_vocab"))
                 if "xent" in want or tag in want]
    for name, want_grad in xent_legs:
        wl = synthetic.WORKLOADS[name]
        inp = synthetic.make_workload(name)
        x, w, lab = inp["x"].to("cuda"), inp["w"].to("cuda"), inp["labels"].to("cuda")
        loss = torch.empty(wl.M, dtype=torch.float32, device="cuda")
        grad = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda") if want_grad else None

        def step():
            lf.gemm_nt_xent(x, w, lab, loss=loss, grad=grad, stream=stream)
        times, launches = timer.run(step, steps, 3, counter=lf.launch_count)
        lf.check_device_error(stream)
        ms = statistics.mean(times)
        flops = 2.0 * wl.M * wl.N * wl.K
        form = grad_form(want_grad, launches / steps)
        # the recompute form runs the GEMM twice; the one-pass kernel and the
        # exp pass + rescale run it once
        executed = flops * (2 if form == "recompute" else 1)
        key = name if not (want_grad and name == "xent_loss") else "xent_grad_large_vocab"
        res[key] = {"M": wl.M, "N": wl.N, "K": wl.K, "grad": want_grad, "ms": round(ms, 4),
                    "tflops_algorithmic": round(flops / ms / 1e9, 1),
                    "tflops_executed": round(executed / ms / 1e9, 1),
                    **xent_fractions(flops, executed, ms, peaks),
                    "launches_per_step": launches / steps, "grad_form": form}
        if want_grad:
            # the other gradient forms on the same workload, for comparison
            for label, path in (("one_pass", 1), ("exp_rescale", 2)):
                lf.set_xent_grad_path(path)
                try:
                    t_alt, n_alt = timer.run(step, steps, 3, counter=lf.launch_count)
                    lf.check_device_error(stream)
                finally:
                    lf.set_xent_grad_path(0)
                ms_alt = statistics.mean(t_alt)
                f_alt = grad_form(True, n_alt / steps)
                res[key]["form_" + label] = {"ms": round(ms_alt, 4), "grad_form": f_alt,
                                             "tflops_algorithmic": round(flops / ms_alt / 1e9, 1),
                                             "pct_of_burst_algorithmic":
                                                 round(100 * flops / ms_alt / 1e9 / peaks["bf16_tflops"], 1)}
        if not want_grad and name == "xent_loss":
            # The unfused comparison of the loss-only fusion ("the IO saving"): this
            # library's GEMM writing the bf16 logits to HBM, then PyTorch's
            # cross-entropy reading them back.  A measured comparison, not a target.
            logits = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
            lab64 = lab.long()

            def unfused():
                lf.gemm_nt(x, w, logits, stream=stream)
                with torch.cuda.stream(stream):
                    torch.nn.functional.cross_entropy(logits, lab64, reduction="none")
            times = timer.run(unfused, steps, 3)
            ms_u = statistics.mean(times)
            res["xent_loss_unfused"] = {"M": wl.M, "N": wl.N, "K": wl.K, "ms": round(ms_u, 4),
                                        "what": "gemm_nt to bf16 logits + torch cross_entropy(reduction='none')",
                                        "logits_bytes": wl.M * wl.N * 2,
                                        "fused_speedup": round(ms_u / ms, 3)}
            del logits, lab64
        if want_grad and name == "xent_grad":
            # the same gradient with the weight stored [K, N] (read N-major in
            # place, e.g. a tied embedding used transposed)
            w_kn = w.t().contiguous()

            def step_kn():
                lf.gemm_nt_xent(x, w_kn, lab, loss=loss, grad=grad, stream=stream, w_mn=True)
            times, launches = timer.run(step_kn, steps, 3, counter=lf.launch_count)
            lf.check_device_error(stream)
            ms = statistics.mean(times)
            form_kn = grad_form(True, launches / steps)
            executed = flops * (2 if form_kn == "recompute" else 1)
            res["xent_grad_w_stored_kn"] = {"M": wl.M, "N": wl.N, "K": wl.K, "grad": True, "w_stored": "[K,N]",
                                            "ms": round(ms, 4),
                                            "tflops_algorithmic": round(flops / ms / 1e9, 1),
                                            "tflops_executed": round(executed / ms / 1e9, 1),
                                            **xent_fractions(flops, executed, ms, peaks),
                                            "launches_per_step": launches / steps,
                                            "grad_form": form_kn}
            del w_kn
        del x, w, lab, loss, grad, inp
        torch.cuda.empty_cache()
    # other operand layouts at the headline shape: W stored [K,N] (the trace's
    # transposed copy, read as is), X stored [K,M], both
    if "layouts" in want:
        wl = synthetic.WORKLOADS["nt_projection"]
        inp = synthetic.make_workload("nt_projection")
        x = inp["x"].reshape(wl.M, wl.K)
        w = inp["w"]
        flops = 2.0 * wl.M * wl.N * wl.K
        out = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
        for label, x_mn, w_mn in (("layout_nn", False, True), ("layout_tn", True, False), ("layout_tt", True, True)):
            xs = (x.t().contiguous() if x_mn else x).to("cuda")
            ws = (w.t().contiguous() if w_mn else w).to("cuda")

            def step():
                lf.gemm_layout(xs, ws, x_mn=x_mn, w_mn=w_mn, out=out, stream=stream)
            times = timer.run(step, max(steps, 10), 3)
            ms = statistics.median(times)
            res[label] = {"M": wl.M, "N": wl.N, "K": wl.K, "x_stored": "[K,M]" if x_mn else "[M,K]",
                          "w_stored": "[K,N]" if w_mn else "[N,K]", "ms": round(ms, 5),
                          "tflops": round(flops / ms / 1e9, 1),
                          "pct_of_peak": round(100 * flops / ms / 1e9 / peaks["bf16_tflops"], 1),
                          "peak_kind": "bf16 burst (%s)" % peaks["source"]}
            del xs, ws
        # batched strided views: the same FLOPs as 4 batches of N/4 columns (one
        # shared X, W sliced by a batch stride), and X read through a view with
        # padded rows (row pitch 16384 instead of 13824)
        xd, wd = x.to("cuda"), w.to("cuda")
        B, Nb = 4, wl.N // 4
        outb = torch.empty(B, wl.M, Nb, dtype=torch.bfloat16, device="cuda")
        xpad = torch.zeros(wl.M, 16384, dtype=torch.bfloat16, device="cuda")
        xpad[:, :wl.K] = xd
        cases = (("batched_4x", lambda: lf.gemm_batched(xd, False, wl.K, 0, wd, False, wl.K, Nb * wl.K, outb, Nb,
                                                         wl.M * Nb, B, wl.M, Nb, wl.K, stream=stream),
                  "4 batches of [768 x 1280], X shared (stride 0), W batch stride 1280*13824"),
                 ("strided_x", lambda: lf.bmm(xpad[:, :wl.K], wd.t(), out=out, stream=stream),
                  "X a [768, 13824] view of [768, 16384] rows"))
        for label, fn, what in cases:
            times = timer.run(fn, max(steps, 10), 3)
            ms = statistics.median(times)
            res[label] = {"M": wl.M, "N": wl.N, "K": wl.K, "what": what, "ms": round(ms, 5),
                          "tflops": round(flops / ms / 1e9, 1),
                          "pct_of_peak": round(100 * flops / ms / 1e9 / peaks["bf16_tflops"], 1),
                          "peak_kind": "bf16 burst (%s)" % peaks["source"]}
        # skinny X (decode-like): 64 rows against the same W; HBM-bound on the
        # 141.6 MB weight stream, computed with the operands swapped
        xs64 = xd[:64].contiguous()
        outs = torch.empty(64, wl.N, dtype=torch.bfloat16, device="cuda")
        times = timer.run(lambda: lf.gemm_nt(xs64, wd, outs, stream=stream), max(steps, 10), 3)
        ms = statistics.median(times)
        wbytes = wl.N * wl.K * 2
        res["skinny_m64"] = {"M": 64, "N": wl.N, "K": wl.K, "ms": round(ms, 5),
                             "tflops": round(2.0 * 64 * wl.N * wl.K / ms / 1e9, 1),
                             "w_stream_GB/s": round(wbytes / ms / 1e6, 1),
                             "pct_of_hbm": round(100 * wbytes / ms / 1e6 / peaks["hbm_gbs"], 1),
                             "what": "W bytes / time against the HBM copy peak (swapped operands)"}
        del xd, wd, outb, xpad, xs64, outs
        del out, inp
        torch.cuda.empty_cache()
    if "library" in want:
        try:
            res["library"] = library_paths(torch, synthetic, timer, stream, peaks, steps)
        except Exception as e:  # context only: it never costs the bench line
            res["library"] = {"error": "%s: %s" % (type(e).__name__, e)}
    torch.cuda.empty_cache()
    return res


def library_paths(torch, synthetic, timer, stream, peaks, steps):
    """The same workloads computed by PyTorch's own GPU operators (cuBLAS for
    the matmuls, eager elementwise and reduction kernels for the rest), timed
    the same way: context for the kernels above, not part of this library."""
    res = {}
    F = torch.nn.functional

    def timed(fn):
        def in_stream():
            with torch.cuda.stream(stream):
                fn()
        return statistics.median(timer.run(in_stream, max(steps, 10), 3))

    # the headline GEMM and its skinny (64-row) form through torch.mm
    wl = synthetic.WORKLOADS["nt_projection"]
    inp = synthetic.make_workload("nt_projection")
    x = inp["x"].reshape(wl.M, wl.K).to("cuda")
    w = inp["w"].to("cuda")
    out = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
    ms = timed(lambda: torch.mm(x, w.t(), out=out))
    flops = 2.0 * wl.M * wl.N * wl.K
    res["gemm_nt_projection"] = {"M": wl.M, "N": wl.N, "K": wl.K, "what": "torch.mm(x, w.t()) (cuBLAS)",
                                 "ms": round(ms, 5), "tflops": round(flops / ms / 1e9, 1),
                                 "pct_of_peak": round(100 * flops / ms / 1e9 / peaks["bf16_tflops"], 1)}
    x64 = x[:64].contiguous()
    out64 = torch.empty(64, wl.N, dtype=torch.bfloat16, device="cuda")
    ms = timed(lambda: torch.mm(x64, w.t(), out=out64))
    wbytes = wl.N * wl.K * 2
    res["gemm_skinny_m64"] = {"M": 64, "N": wl.N, "K": wl.K, "what": "torch.mm(x[:64], w.t()) (cuBLAS)",
                              "ms": round(ms, 5), "w_stream_GB/s": round(wbytes / ms / 1e6, 1),
                              "pct_of_hbm": round(100 * wbytes / ms / 1e6 / peaks["hbm_gbs"], 1)}
    del x, w, out, x64, out64, inp
    torch.cuda.empty_cache()

    # cross-entropy loss and logit gradient, unfused: cuBLAS logits in bf16,
    # then log-sum-exp, the label logit and softmax minus the one-hot label
    wl = synthetic.WORKLOADS["xent_grad"]
    inp = synthetic.make_workload("xent_grad")
    x, w = inp["x"].to("cuda"), inp["w"].to("cuda")
    lab = inp["labels"].to("cuda").long()
    logits = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
    rows = torch.arange(wl.M, device="cuda")

    def xent_grad():
        torch.mm(x, w.t(), out=logits)
        z = logits.float()
        lse = torch.logsumexp(z, dim=1)
        loss = lse - z[rows, lab]
        g = torch.exp(z - lse[:, None])
        g[rows, lab] -= 1.0
        return loss, g.to(torch.bfloat16)
    ms = timed(xent_grad)
    flops = 2.0 * wl.M * wl.N * wl.K
    res["xent_grad"] = {"M": wl.M, "N": wl.N, "K": wl.K,
                        "what": "torch.mm to bf16 logits, logsumexp, exp(z - lse) minus one-hot, cast to bf16",
                        "ms": round(ms, 4), "tflops_algorithmic": round(flops / ms / 1e9, 1)}
    del x, w, lab, logits, rows, inp
    torch.cuda.empty_cache()

    # the K=1 product through torch.mm, at the bandwidth size
    a = torch.randn(64, 1, device="cuda")
    b = torch.arange(1 << 23, dtype=torch.float32, device="cuda").reshape(1, -1)
    o = torch.empty(64, 1 << 23, dtype=torch.float32, device="cuda")
    ms = timed(lambda: torch.mm(a, b, out=o))
    nbytes = (64 + (1 << 23) + 64 * (1 << 23)) * 4
    res["k1_scaled"] = {"M": 64, "N": 1 << 23, "what": "torch.mm([64,1], [1,N]) fp32", "ms": round(ms, 5),
                        "GB/s": round(nbytes / ms / 1e6, 1),
                        "pct_of_hbm": round(100 * nbytes / ms / 1e6 / peaks["hbm_gbs"], 1)}
    del a, b, o
    torch.cuda.empty_cache()

    # RoPE cos/sin in eager PyTorch: outer product, concatenation, cos, sin, casts
    inv, pos = synthetic.rope_operands(64, 1 << 20, max_position=32768)
    inv, pos = inv.to("cuda"), pos.to("cuda")

    def rope():
        f = pos.float()[:, None] * inv[None, :]
        emb = torch.cat((f, f), dim=-1)
        return emb.cos().to(torch.bfloat16), emb.sin().to(torch.bfloat16)
    ms = timed(rope)
    S = 1 << 20
    nbytes = 64 * 2 + S * 8 + 2 * S * 128 * 2
    res["rope_scaled"] = {"H": 64, "S": S, "what": "eager outer product, cat, cos, sin, bf16 casts",
                          "ms": round(ms, 5), "GB/s_algorithmic": round(nbytes / ms / 1e6, 1)}
    del inv, pos
    torch.cuda.empty_cache()

    # the fp8 cast in both layouts, eager: scale, clamp, cast, then a transposed copy
    xs = synthetic.bf16_normal((16384, 16384), 1.0, 15).to("cuda")
    scale = torch.tensor([10.0], dtype=torch.float32, device="cuda")

    def fp8():
        q = (xs.float() * scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        return q, q.t().contiguous()
    ms = timed(fp8)
    nbytes = 16384 * 16384 * 4
    res["fp8_cast_scaled"] = {"M": 16384, "K": 16384, "what": "eager scale, clamp, cast, transposed copy",
                              "ms": round(ms, 5), "GB/s_algorithmic": round(nbytes / ms / 1e6, 1)}
    del xs, scale
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------- CPU oracle legs

def cpu_baseline_gemm(x, w, wl, budget_s=15.0):
    """Time the oracle (as it stands) on a bounded sample of rows of the workload:
    a probe of 2 rows per thread sizes the sample to about `budget_s` seconds."""
    import numpy as np

    import oracle
    xb = oracle._bits(x)
    wb = oracle._bits(w)
    threads = oracle.num_threads()
    probe = np.arange(min(wl.M, 2 * threads), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.gemm_nt_rows(xb, wb, probe)
    t_probe = max(time.perf_counter() - t0, 1e-3)
    nrows = int(max(probe.size, min(wl.M, probe.size * budget_s / t_probe)))
    nrows -= nrows % threads if nrows > threads else 0
    rows = np.arange(nrows, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.gemm_nt_rows(xb, wb, rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * nrows * wl.N * wl.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "%d of %d rows of X (all %d columns of W, K=%d), fp64 plain loops" % (nrows, wl.M, wl.N, wl.K)}


def run_reference(args, rank, world):
    from layout_folding_gb300 import synthetic
    wl = synthetic.WORKLOADS["nt_projection"]
    inp = synthetic.make_workload("nt_projection")
    import numpy as np

    import oracle
    xb = oracle._bits(inp["x"].reshape(wl.M, wl.K))
    wb = oracle._bits(inp["w"])
    # size one step to about (6 * budget / (warmup + steps)) seconds, from a
    # probe of 2 rows per thread
    threads = oracle.num_threads()
    probe = np.arange(min(wl.M, 2 * threads), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.gemm_nt_rows(xb, wb, probe)
    per_row = max(time.perf_counter() - t0, 1e-3) / probe.size
    per_step_s = args.cpu_budget * 6 / max(1, args.steps + args.warmup)
    nrows = int(max(1, min(wl.M, per_step_s / per_row)))
    times = []
    for i in range(args.warmup + args.steps):
        rows = (np.arange(nrows, dtype=np.int64) + i * nrows) % wl.M
        t0 = time.perf_counter()
        oracle.gemm_nt_rows(xb, wb, rows)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    flops = 2.0 * nrows * wl.N * wl.K
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = "%d of %d rows of X per step (all %d columns of W, K=%d), fp64 plain loops" % (nrows, wl.M, wl.N, wl.K)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1)*0.02 bf16; no dataset)",
        "config": headline_config(wl, world),
        "timing": "wall clock around each step's oracle call on the host cores",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true", help="skip every secondary path")
    ap.add_argument("--paths", default="tiny,xent,k1,layouts,rope,fp8,library",
                    help="secondary paths to time after the headline (comma list of tiny, xent, k1, layouts, rope, "
                         "fp8, library; xent_grad, xent_loss, xent_grad_large_vocab select one cross-entropy leg)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cooperative", action="store_true",
                    help="launch the stream-K and one-pass kernels without the cooperative attribute (for ncu, "
                         "which cannot replay cooperative cluster launches); same kernels")
    ap.add_argument("--tile-schedule", choices=["auto", "fixed", "claimed"], default="auto",
                    help="whole tiles on CTA pairs: the automatic choice (fixed), the fixed assignment or tiles "
                         "claimed at run time (for comparisons; results are identical)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
