#!/usr/bin/env python3
"""Benchmark of the fine-grained FP8 hot path on one B300.

One step = the whole path over one batch of the dense-projection workload
(A = 4096 x 7168 BF16 activations, W = 18432 x 7168 BF16 weights):
  1. fp8_quant_act_1x128       A -> E4M3 codes + FP32 scales per 1x128 tile
  2. fp8_quant_weight_128x128  W -> E4M3 codes + FP32 scales per 128x128 block
  3. fp8_blockscaled_gemm      C = A W^T, per-128-K promotion into FP32, BF16 output
The metric is block-scaled FP8 GEMM throughput in TFLOP/s (2*M*N*K per step divided by the
step time, quantizers included); per-kernel GB/s and TFLOP/s against the rooflines ride along.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the step (the path needs no
exchange between GPUs); the reported time is the maximum over ranks and `value` counts the work
of all ranks. `--impl reference` times the CPU oracle (plain C, the correctness reference) on a
bounded sample of the same workload on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_fine_grained_23_b300 import workloads as WL  # noqa: E402

METRIC = "block-scaled FP8 GEMM TFLOPS (% FP8 peak); quantizer GB/s (% HBM), 1 B300"
SHAPE = WL.DENSE
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
FP8_OVER_BF16 = 2.0      # nominal dense ratio on B300: 4.5 / 2.25 PFLOP/s
ACT_BYTES_PER_ELEM = 2 + 1 + 4 / 128      # BF16 read, code write, one FP32 scale per 128
W_BYTES_PER_ELEM = 2 + 1 + 4 / (128 * 128)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        out = {k: float(p[k]) for k in FALLBACK_PEAKS}
        mhz = (p.get("clocks_under_load") or {}).get("sm_mhz_median")
        out["sustained_sm_mhz"] = float(mhz) if mhz is not None else None
        return out, "measured"
    except (OSError, KeyError, ValueError, TypeError):
        return dict(FALLBACK_PEAKS, sustained_sm_mhz=None), "fallback"


def choose_fp8_peak(peaks, clk):
    """FP8 denominators for the GEMM timed inside the step: (peak, burst peak, note).

    The measured BF16 figures come as a burst (a GEMM alone at full clock) and as a sustained
    loop under the 1.1 kW power cap, at the power-capped median SM clock recorded with them. The
    step's GEMM is compared with the sustained figure only when the clocks sampled during the
    timed region show that same state (power cap active, median SM clock no higher than 10%
    above the sustained measurement's); otherwise (a short timed region at full clock, or no
    clock record) the burst figure is the denominator."""
    burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    sustained = peaks["bf16_tflops_sustained"] * FP8_OVER_BF16
    cap_mhz = peaks.get("sustained_sm_mhz")
    capped = (clk is not None and "sw_power_cap" in (clk.get("reasons") or [])
              and cap_mhz is not None and clk.get("sm_mhz") is not None
              and clk["sm_mhz"] <= 1.1 * cap_mhz)
    if capped:
        return sustained, burst, (f"2 x bf16 sustained {peaks['bf16_tflops_sustained']} TFLOP/s "
                                  f"(power-capped, measured at a {cap_mhz:.0f} MHz median; this "
                                  f"run's median {clk['sm_mhz']:.0f} MHz under sw_power_cap)")
    seen = "no clock record" if clk is None else \
        f"median SM clock {clk.get('sm_mhz')} MHz, reasons {clk.get('reasons')}"
    return burst, burst, (f"2 x bf16 burst {peaks['bf16_tflops']} TFLOP/s (nominal fp8/bf16 "
                          f"ratio 4.5/2.25); the timed region's clocks ({seen}) are not the "
                          "power-capped state of the sustained figure")


def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def reduce_max(values, device=None):
    """Element-wise maximum of `values` over all ranks (the slowest rank sets the time)."""
    t = torch.tensor(values, dtype=torch.float64)
    dist = torch.distributed
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if dist.get_backend() == "nccl":
            t = t.to(device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


# --------------------------------------------------------------------------------------
# Clock sampling during the timed region
# --------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # the extras' sampler also records the memory clock and the HBM temperature
    MEMORY_FIELDS = ",clocks.mem,temperature.memory"

    def __init__(self, device_index: int, memory: bool = False):
        self.proc = None
        self.path = None
        self.memory = memory
        self.n_fields = 10 if memory else 8
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.ident = str(device_index)

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident,
                 f"--query-gpu={self.FIELDS + (self.MEMORY_FIELDS if self.memory else '')}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == self.n_fields:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[0]) for r in rows]
        mx = [num(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
               "power_w_max": max(num(r[2]) for r in rows), "samples": len(rows),
               "reasons": reasons}
        if self.memory:
            out["mem_mhz_min"] = min(num(r[8]) for r in rows)
            out["hbm_temp_c_max"] = max(num(r[9]) for r in rows)
        # a field the GPU does not report ("N/A") becomes null, never NaN, in the JSON line
        return {k: (None if isinstance(v, float) and v != v else v) for k, v in out.items()}


# --------------------------------------------------------------------------------------
# Our path
# --------------------------------------------------------------------------------------

def traffic_from_profile():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was taken on the
    current kernel source (matching SHA-256); otherwise None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "gemm_dense_4096x18432x7168.txt")
    src = os.path.join(ROOT, "fp8_fine_grained_23_b300", "csrc", "gemm.cu")
    try:
        kv = {}
        for line in open(path):
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if kv.get("gemm_cu_sha256") != sha:
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def run_ours(args, rank, world, local_rank):
    from fp8_fine_grained_23_b300 import build as B
    if rank == 0 or not os.path.exists(B.LIB_PATH):
        B.build()
    if world > 1:
        torch.distributed.barrier()
    from fp8_fine_grained_23_b300 import fp8bs as F

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    M, N, K = SHAPE.M, SHAPE.N, SHAPE.K
    a, w = WL.gemm_inputs(SHAPE, dev)
    aq = torch.empty(M, K, dtype=torch.uint8, device=dev)
    a_s = torch.empty(K // 128, M, dtype=torch.float32, device=dev)
    wq = torch.empty(N, K, dtype=torch.uint8, device=dev)
    w_s = torch.empty((N + 127) // 128, K // 128, dtype=torch.float32, device=dev)
    c = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    # The two quantizers are independent: the weight quantizer runs on a second stream beside the
    # activation quantizer (both HBM-bound; overlapping them hides one's ramp-up and tail behind
    # the other), and the GEMM waits for both.
    stream_w = torch.cuda.Stream(dev)
    ev_go, ev_w = torch.cuda.Event(), torch.cuda.Event()

    def step(ev=None):
        ev_go.record(stream)                # the previous step's GEMM has been issued
        stream_w.wait_event(ev_go)
        if ev is not None:
            ev[0].record(stream)
            ev[4].record(stream_w)
        F.fp8_quant_act_1x128(a, aq, a_s, stream=sh)
        F.fp8_quant_weight_128x128(w, wq, w_s, stream=stream_w.cuda_stream)
        if ev is not None:
            ev[1].record(stream)
            ev[5].record(stream_w)
        ev_w.record(stream_w)
        stream.wait_event(ev_w)
        if ev is not None:
            ev[2].record(stream)
        F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out=c, stream=sh)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if F.fp8bs_last_error(sh) != F.FP8BS_OK:
        raise RuntimeError("a kernel reported a pipeline timeout during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)                        # let the sampler take its first readings
    t0.record(stream)
    for i in range(args.steps):
        step(events[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if F.fp8bs_last_error(sh) != F.FP8BS_OK:
        raise RuntimeError("a kernel reported a pipeline timeout in the timed region")

    ms = t0.elapsed_time(t1) / args.steps
    # per kernel: activation quantizer (stream), weight quantizer (second stream, concurrent),
    # GEMM (stream, after both)
    k_ms = [statistics.mean(e[0].elapsed_time(e[1]) for e in events),
            statistics.mean(e[4].elapsed_time(e[5]) for e in events),
            statistics.mean(e[2].elapsed_time(e[3]) for e in events)]
    ms, qa_ms, qw_ms, g_ms = reduce_max([ms] + k_ms, dev)

    # End to end through the C ABI from pinned host buffers, every step: H2D of that step's A and
    # W, the three calls, D2H of C. The steps are pipelined over three streams (copies in,
    # compute, copies out) with two device buffer sets, so step i+1's inputs cross PCIe while
    # step i computes and its result crosses back (PCIe is full duplex); every copy of every
    # step is inside the timed region.
    a_h = a.cpu().pin_memory()
    w_h = w.cpu().pin_memory()
    c_h = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    bufs = [(a, w, aq, a_s, wq, w_s, c),
            tuple(torch.empty_like(t) for t in (a, w, aq, a_s, wq, w_s, c))]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_steps = max(3, min(10, args.steps))
    n_e2e = e2e_steps + 1                   # the first pass is a warm-up
    ev = [[torch.cuda.Event() for _ in range(3)] for _ in range(n_e2e)]   # in, computed, out
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(n_e2e):
        if i == 1:
            torch.cuda.synchronize(dev)
            s0.record(s_in)
        ab, wb, aqb, asb, wqb, wsb, cb = bufs[i % 2]
        if i >= 2:
            s_in.wait_event(ev[i - 2][1])   # step i-2 has finished reading this buffer set
        with torch.cuda.stream(s_in):
            ab.copy_(a_h, non_blocking=True)
            wb.copy_(w_h, non_blocking=True)
        ev[i][0].record(s_in)
        stream.wait_event(ev[i][0])
        if i >= 2:
            stream.wait_event(ev[i - 2][2])   # step i-2's result has left this buffer set
        F.fp8_quant_act_1x128(ab, aqb, asb, stream=sh)
        F.fp8_quant_weight_128x128(wb, wqb, wsb, stream=sh)
        F.fp8_blockscaled_gemm(aqb, asb, wqb, wsb, out=cb, stream=sh)
        ev[i][1].record(stream)
        s_out.wait_event(ev[i][1])
        with torch.cuda.stream(s_out):
            c_h.copy_(cb, non_blocking=True)
        ev[i][2].record(s_out)
    s1.record(s_out)
    torch.cuda.synchronize(dev)
    if F.fp8bs_last_error(sh) != F.FP8BS_OK:
        raise RuntimeError("a kernel reported a pipeline timeout in the end-to-end run")
    e2e_ms = reduce_max([s0.elapsed_time(s1) / e2e_steps], dev)[0]
    e2e = {"value": round(gemm_flops(M, N, K) * world / (e2e_ms * 1e-3) / 1e12, 2),
           "unit": "TFLOP/s",
           "h2d_bytes_per_step": a.numel() * 2 + w.numel() * 2,
           "d2h_bytes_per_step": c.numel() * 2,
           "ms_per_step": round(e2e_ms, 4),
           "pipelined": "copies in / compute / copies out on three streams, two buffer sets"}

    peaks, peak_src = load_peaks()
    fp8_peak, fp8_peak_burst, peak_note = choose_fp8_peak(peaks, clk)
    g_tflops = gemm_flops(M, N, K) / (g_ms * 1e-3) / 1e12
    qa_gbs = M * K * ACT_BYTES_PER_ELEM / (qa_ms * 1e-3) / 1e9
    qw_gbs = N * K * W_BYTES_PER_ELEM / (qw_ms * 1e-3) / 1e9
    traffic = traffic_from_profile()
    value = gemm_flops(M, N, K) * world / (ms * 1e-3) / 1e12

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic (seeded N(0,1) activations with 0.1% x100 outliers, N(0,0.02) weights)",
        "config": {"workload": SHAPE.name, "M": M, "N": N, "K": K, "out": "bf16",
                   "step": "quant_act_1x128 and quant_weight_128x128 (concurrent), then blockscaled_gemm",
                   "l2": "inputs larger than L2 (A+W BF16 = %.0f MB > 126 MB)"
                         % ((M + N) * K * 2 / 1e6),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"kernel": "fp8_blockscaled_gemm", "bound": "tensor",
                     "achieved": round(g_tflops, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(g_tflops / fp8_peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{peak_src}: {peak_note}",
                     "frac_of_burst_peak": round(g_tflops / fp8_peak_burst, 4),
                     "burst_peak": round(fp8_peak_burst, 1)},
        "kernels": {
            "quant_act_1x128": {"ms": round(qa_ms, 5), "GB/s": round(qa_gbs, 1),
                                "frac_hbm": round(qa_gbs / peaks["hbm_gbs"], 4)},
            "quant_weight_128x128": {"ms": round(qw_ms, 5), "GB/s": round(qw_gbs, 1),
                                     "frac_hbm": round(qw_gbs / peaks["hbm_gbs"], 4)},
            "blockscaled_gemm": {"ms": round(g_ms, 5), "TFLOP/s": round(g_tflops, 1),
                                 "frac_fp8_peak": round(g_tflops / fp8_peak, 4)},
            "hbm_peak_gbs": peaks["hbm_gbs"], "peak_source": peak_src,
        },
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
    }
    if not args.no_extras:
        del a, w, aq, a_s, wq, w_s, c, a_h, w_h, c_h
        torch.cuda.empty_cache()
        line["workloads"] = run_extras(F, dev, peaks, fp8_peak_burst)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget_s)
    return line


# --------------------------------------------------------------------------------------
# The other workloads, each kernel timed alone (L2 flushed between iterations)
# --------------------------------------------------------------------------------------

def _timed(fn, dev, iters=10, warm=3):
    """Mean device time (ms) of fn(). Before every run L2 is flushed by reading a 256 MB buffer
    (written once up front): reading evicts the cache without leaving dirty lines whose
    write-back would then compete with the kernel being timed. One untimed call runs and
    finishes first; then a spin kernel queued ahead keeps the GPU busy while the host enqueues
    every iteration, so that no host launch gap can fall between an iteration's start event and
    its kernel."""
    flush = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)   # 256 MB
    stream = torch.cuda.current_stream(dev)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(warm + iters)]
    # one call on its own first: a kernel's first launch in the process (module loading, launch
    # attributes) costs milliseconds of host time, which must not fall between timed events
    fn()
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(250_000 * (warm + iters))   # ~0.12 ms of GPU clock cycles per iteration
    for e0, e1 in events:
        sink = flush.sum()   # noqa: F841  (read-only flush)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return statistics.mean(a.elapsed_time(b) for a, b in events[warm:])


def run_backward(F, dev, hbm, fp8_peak):
    """Backward pass of the dense projection (M=4096 tokens, N=18432, K=7168): the four
    quantizations a training step needs (dY and X in 128x1 tiles for the weight gradient, dY in
    1x128 tiles and W as W^T codes for the data gradient) and the two GEMMs, each timed alone."""
    shape = WL.DENSE
    x, w, dy = WL.backward_inputs(shape, dev)
    M, N, K = shape.M, shape.N, shape.K
    res = {"workload": f"dense_bwd_{M}x{N}x{K}"}

    def quant(name, fn, elems, bytes_per_elem):
        ms = _timed(fn, dev)
        gbs = elems * bytes_per_elem / (ms * 1e-3) / 1e9
        res[name] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / hbm, 4)}

    dyt_q = torch.empty(N, M, dtype=torch.uint8, device=dev)
    dyt_s = torch.empty(M // 128, N, dtype=torch.float32, device=dev)
    xt_q = torch.empty(K, M, dtype=torch.uint8, device=dev)
    xt_s = torch.empty(M // 128, K, dtype=torch.float32, device=dev)
    dy_q = torch.empty(M, N, dtype=torch.uint8, device=dev)
    dy_s = torch.empty(N // 128, M, dtype=torch.float32, device=dev)
    wt_q = torch.empty(K, N, dtype=torch.uint8, device=dev)
    wt_s = torch.empty(K // 128, N // 128, dtype=torch.float32, device=dev)
    quant("quant_128x1_dY", lambda: F.fp8_quant_act_128x1(dy, dyt_q, dyt_s), M * N, ACT_BYTES_PER_ELEM)
    quant("quant_128x1_X", lambda: F.fp8_quant_act_128x1(x, xt_q, xt_s), M * K, ACT_BYTES_PER_ELEM)
    quant("quant_1x128_dY", lambda: F.fp8_quant_act_1x128(dy, dy_q, dy_s), M * N, ACT_BYTES_PER_ELEM)
    quant("quant_weight_t_W", lambda: F.fp8_quant_weight_128x128_t(w, wt_q, wt_s), N * K,
          W_BYTES_PER_ELEM)
    dw = torch.empty(N, K, dtype=torch.float32, device=dev)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    for name, fn in (
            ("wgrad_gemm_1d1d_f32", lambda: F.fp8_blockscaled_gemm_1d1d(dyt_q, dyt_s, xt_q, xt_s,
                                                                         out=dw)),
            ("dgrad_gemm_bf16", lambda: F.fp8_blockscaled_gemm(dy_q, dy_s, wt_q, wt_s, out=dx))):
        ms = _timed(fn, dev)
        tf = gemm_flops(M, N, K) / (ms * 1e-3) / 1e12
        res[name] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                     "frac_fp8_peak": round(tf / fp8_peak, 4)}
    res["gemm_shapes"] = {"wgrad_gemm_1d1d_f32": [N, K, M], "dgrad_gemm_bf16": [M, K, N]}
    return res


def section_only(rank, section, moe_experts):
    """One section of the other workloads alone (rank 0 only; no step, no baseline), e.g. to
    capture its kernels with ncu. moe_experts < 256 scales the MoE workload down to that many
    experts with the same rows per expert (tokens * experts / 256)."""
    if rank != 0:
        return None
    from fp8_fine_grained_23_b300 import fp8bs as F
    dev = torch.device("cuda", 0)
    peaks, _ = load_peaks()
    moe_shape = WL.MOE
    if moe_experts != WL.MOE.experts:
        moe_shape = dataclasses.replace(
            WL.MOE, name=f"moe_{WL.MOE.tokens * moe_experts // WL.MOE.experts}tok_{moe_experts}e_top8",
            experts=moe_experts, tokens=WL.MOE.tokens * moe_experts // WL.MOE.experts)
    return {"workloads": run_extras(F, dev, peaks, peaks["bf16_tflops"] * FP8_OVER_BF16,
                                    only=section, moe_shape=moe_shape)}


def run_sweep(F, dev, hbm, fp8_peak):
    # quantizer bandwidth sweep
    sweep = {}
    for M in WL.SWEEP_ACT_M:
        x = WL.sweep_activations(M, dev)
        q = torch.empty(M, WL.SWEEP_K, dtype=torch.uint8, device=dev)
        s = torch.empty(WL.SWEEP_K // 128, M, dtype=torch.float32, device=dev)
        ms = _timed(lambda: F.fp8_quant_act_1x128(x, q, s), dev)
        gbs = M * WL.SWEEP_K * ACT_BYTES_PER_ELEM / (ms * 1e-3) / 1e9
        sweep[f"act_{M}x{WL.SWEEP_K}"] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                                          "frac_hbm": round(gbs / hbm, 4)}
        del x, q, s
    wt = WL.sweep_weight(dev)
    q = torch.empty_like(wt, dtype=torch.uint8)
    s = torch.empty(WL.SWEEP_W_N // 128, WL.SWEEP_W_K // 128, dtype=torch.float32, device=dev)
    ms = _timed(lambda: F.fp8_quant_weight_128x128(wt, q, s), dev)
    gbs = wt.numel() * W_BYTES_PER_ELEM / (ms * 1e-3) / 1e9
    sweep[f"weight_{WL.SWEEP_W_N}x{WL.SWEEP_W_K}"] = {"us": round(ms * 1e3, 2),
                                                      "GB/s": round(gbs, 1),
                                                      "frac_hbm": round(gbs / hbm, 4)}
    del wt, q, s
    return sweep


def run_mla(F, dev, hbm, fp8_peak):
    # MLA projections
    mla = {}
    for shape in WL.MLA:
        a, w = WL.gemm_inputs(shape, dev)
        aq, a_s = F.fp8_quant_act_1x128(a)
        wq, w_s = F.fp8_quant_weight_128x128(w)
        c = torch.empty(a.shape[0], w.shape[0], dtype=torch.bfloat16, device=dev)
        ms = _timed(lambda: F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out=c), dev)
        tf = gemm_flops(a.shape[0], w.shape[0], a.shape[1]) / (ms * 1e-3) / 1e12
        mla[shape.name] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                           "frac_fp8_peak": round(tf / fp8_peak, 4), "N_run": w.shape[0]}
        del a, w, aq, a_s, wq, w_s, c
    return mla


def run_decode(F, dev, hbm, fp8_peak):
    # decode-size GEMMs (few rows of A): bound by streaming the weights once
    dec = {}
    for (N, K, seed) in ((WL.DENSE.N, WL.DENSE.K, WL.DENSE.seed), (1536, 7168, 2), (24576, 1536, 4)):
        g = WL.generator(seed, dev)
        wq, w_s = F.fp8_quant_weight_128x128(WL.weights(N, K, g, dev))
        for M in (1, 16, 64):
            aq, a_s = F.fp8_quant_act_1x128(WL.activations(M, K, g, dev))
            c = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            ms = _timed(lambda: F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out=c), dev)
            byts = wq.numel() + w_s.numel() * 4 + aq.numel() + a_s.numel() * 4 + c.numel() * 2
            gbs = byts / (ms * 1e-3) / 1e9
            dec[f"{M}x{N}x{K}"] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                                   "frac_hbm": round(gbs / hbm, 4)}
        del wq, w_s, aq, a_s, c
    return dec


def run_moe(F, dev, hbm, fp8_peak, shape=WL.MOE):
    # MoE grouped GEMMs: gate+up and down alone (BF16 out), the gate+up GEMM with the fused
    # SwiGLU + 1x128 re-quantization, and the expert FFN chain (fused gate+up, then down on h)
    moe = {}
    off, token_of_row = WL.moe_routing(shape)
    R = int(off[-1])
    offs = torch.from_numpy(off).to(dev)
    E = shape.experts
    ops = {}
    for which in ("gate_up", "down"):
        if which == "gate_up":
            N, K = shape.n_gate_up, shape.hidden
            a = WL.moe_tokens(shape, dev)[torch.from_numpy(token_of_row).to(dev)]
        else:
            N, K = shape.hidden, shape.k_down
            a = WL.moe_down_input(shape, R, dev)
        wts = WL.moe_expert_weights(shape, N, K, which, dev)
        aq, a_s = F.fp8_quant_act_1x128(a)
        wq, w_s = F.fp8_quant_weight_128x128(wts.view(-1, K))
        del wts, a
        wq = wq.view(E, N, K)
        w_s = w_s.view(E, N // 128, K // 128)
        c = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
        ms = _timed(lambda: F.fp8_blockscaled_grouped_gemm(aq, a_s, wq, w_s, offs, out=c), dev)
        tf = gemm_flops(R, N, K) / (ms * 1e-3) / 1e12
        algo_bytes = wq.numel() + aq.numel() + c.numel() * 2 + a_s.numel() * 4 + w_s.numel() * 4
        gbs = algo_bytes / (ms * 1e-3) / 1e9
        moe[which] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                      "frac_fp8_peak": round(tf / fp8_peak, 4), "GB/s": round(gbs, 1),
                      "frac_hbm": round(gbs / hbm, 4), "R": R, "N": N, "K": K,
                      "experts": E}
        ops[which] = (aq, a_s, wq, w_s)
        del c
        torch.cuda.empty_cache()
    aq, a_s, wq, w_s = ops["gate_up"]
    N2, I = shape.n_gate_up, shape.n_gate_up // 2
    hq = torch.empty(R, I, dtype=torch.uint8, device=dev)
    hs = torch.empty(I // 128, R, dtype=torch.float32, device=dev)
    fused = lambda: F.fp8_blockscaled_grouped_gemm_swiglu_quant(aq, a_s, wq, w_s, offs, hq, hs)
    ms = _timed(fused, dev)
    algo_bytes = wq.numel() + aq.numel() + a_s.numel() * 4 + w_s.numel() * 4 + hq.numel() + \
        hs.numel() * 4
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    moe["gate_up_swiglu_quant"] = {
        "us": round(ms * 1e3, 1), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
        "TFLOP/s": round(gemm_flops(R, N2, shape.hidden) / (ms * 1e-3) / 1e12, 1),
        "out": "E4M3 h [R][N2/2] + 1x128 scales (gate/up weight rows interleaved per 128)"}
    dq, ds_, dwq, dws = ops["down"]
    y = torch.empty(R, shape.hidden, dtype=torch.bfloat16, device=dev)

    def chain():
        fused()
        F.fp8_blockscaled_grouped_gemm(hq, hs, dwq, dws, offs, out=y)
    ms = _timed(chain, dev)
    chain_bytes = algo_bytes + dwq.numel() + dws.numel() * 4 + y.numel() * 2
    gbs = chain_bytes / (ms * 1e-3) / 1e9
    moe["ffn_chain_fused"] = {
        "us": round(ms * 1e3, 1), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
        "TFLOP/s": round((gemm_flops(R, N2, shape.hidden) + gemm_flops(R, shape.hidden, I)) /
                         (ms * 1e-3) / 1e12, 1),
        "steps": "gate/up GEMM + SwiGLU + 1x128 re-quantization, then the down GEMM on h"}
    del ops, aq, a_s, wq, w_s, dq, ds_, dwq, dws, hq, hs, y
    torch.cuda.empty_cache()
    # token-side dispatch: permute the quantized tokens into expert order; combine the expert
    # outputs back per token with the routing weights
    T, Kh = shape.tokens, shape.hidden
    xq, xs = F.fp8_quant_act_1x128(WL.moe_tokens(shape, dev))
    tok = torch.from_numpy(token_of_row.astype(np.int32)).to(dev)
    qp = torch.empty(R, Kh, dtype=torch.uint8, device=dev)
    sp = torch.empty(Kh // 128, R, dtype=torch.float32, device=dev)
    ms = _timed(lambda: F.fp8_moe_permute(xq, xs, tok, qp, sp), dev)
    pbytes = 2 * R * Kh + 2 * sp.numel() * 4 + tok.numel() * 4
    moe["permute"] = {"us": round(ms * 1e3, 2), "GB/s": round(pbytes / (ms * 1e-3) / 1e9, 1),
                      "frac_hbm": round(pbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                      "rows": R, "K": Kh}
    rows = torch.from_numpy(WL.moe_row_of_token(token_of_row, T, shape.topk)).to(dev)
    gw = torch.from_numpy(WL.moe_gate_weights(shape)).to(dev)
    yv = WL.activations(R, Kh, WL.generator(shape.seed + 3, dev), dev)   # expert outputs
    outv = torch.empty(T, Kh, dtype=torch.bfloat16, device=dev)
    ms = _timed(lambda: F.fp8_moe_combine(yv, rows, gw, outv), dev)
    cbytes = 2 * R * Kh + 2 * T * Kh + rows.numel() * 8
    moe["combine"] = {"us": round(ms * 1e3, 2), "GB/s": round(cbytes / (ms * 1e-3) / 1e9, 1),
                      "frac_hbm": round(cbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                      "tokens": T, "topk": shape.topk, "N": Kh}
    del xq, xs, tok, qp, sp, rows, gw, yv, outv
    torch.cuda.empty_cache()
    return moe


def run_ue8m0(F, dev, hbm):
    """Power-of-two (UE8M0) tile scales against the pages' amax/448 scales on the dense
    workload: quantizer speed, and the GEMM's relative error on a 256 x 1024 block of C against
    the FP64 product of the BF16 inputs (computed here with PyTorch; a measurement, not parity)."""
    a, w = WL.gemm_inputs(WL.DENSE, dev)
    M, K = a.shape
    N = w.shape[0]
    res = {"workload": WL.DENSE.name}
    ref = a[:256].double() @ w[:1024].double().t()
    for mode, qa_fn, qw_fn in (("fp32_scales", F.fp8_quant_act_1x128, F.fp8_quant_weight_128x128),
                               ("ue8m0_scales", F.fp8_quant_act_1x128_ue8m0,
                                F.fp8_quant_weight_128x128_ue8m0)):
        q = torch.empty(M, K, dtype=torch.uint8, device=dev)
        s = torch.empty(K // 128, M, dtype=torch.float32, device=dev)
        ms_a = _timed(lambda: qa_fn(a, q, s), dev)
        qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
        sw = torch.empty(N // 128, K // 128, dtype=torch.float32, device=dev)
        ms_w = _timed(lambda: qw_fn(w, qw, sw), dev)
        c = F.fp8_blockscaled_gemm(q[:256].contiguous(), s[:, :256].contiguous(), qw[:1024],
                                   sw[:8], out_dtype=torch.float32)
        err = float(torch.linalg.norm(c.double() - ref) / torch.linalg.norm(ref))
        res[mode] = {"quant_act_us": round(ms_a * 1e3, 2),
                     "quant_act_frac_hbm": round(M * K * ACT_BYTES_PER_ELEM / (ms_a * 1e-3) / 1e9 / hbm, 4),
                     "quant_weight_us": round(ms_w * 1e3, 2),
                     "gemm_rel_err_vs_fp64": float(f"{err:.4g}")}
    return res


def run_requant(F, dev, hbm, fp8_peak):
    """The dense GEMM writing its output re-quantized to E4M3 with 1x128 scales (the next GEMM's
    A operand) against the same GEMM writing BF16, each alone."""
    a, w = WL.gemm_inputs(WL.DENSE, dev)
    M, N, K = WL.DENSE.M, WL.DENSE.N, WL.DENSE.K
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    c = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    cq = torch.empty(M, N, dtype=torch.uint8, device=dev)
    cs = torch.empty(N // 128, M, dtype=torch.float32, device=dev)
    res = {"workload": WL.DENSE.name}
    for name, fn in (("bf16_out", lambda: F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out=c)),
                     ("e4m3_1x128_out", lambda: F.fp8_blockscaled_gemm_quant(aq, a_s, wq, w_s,
                                                                             cq, cs))):
        ms = _timed(fn, dev)
        tf = gemm_flops(M, N, K) / (ms * 1e-3) / 1e12
        res[name] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                     "frac_fp8_peak": round(tf / fp8_peak, 4)}
    return res


def run_library_reference(F, dev, hbm, fp8_peak):
    """A library FP8 GEMM on the dense shape as the external comparison point: cuBLASLt through
    torch._scaled_mm with one scale per tensor (no per-block scales, so no promotion work; an
    upper bound for the block-scaled kernel on the same codes). The block-scaled library form
    (1x128 x 128x128 scales) is tried too and its answer recorded."""
    a, w = WL.gemm_inputs(WL.DENSE, dev)
    M, N, K = WL.DENSE.M, WL.DENSE.N, WL.DENSE.K
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    a8, w8t = aq.view(torch.float8_e4m3fn), wq.view(torch.float8_e4m3fn).t()
    one = torch.ones((), dtype=torch.float32, device=dev)
    c = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    res = {"workload": WL.DENSE.name, "library": f"cuBLASLt (torch {torch.__version__})"}
    runs = (("ours_block_scaled", lambda: F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out=c)),
            ("cublaslt_per_tensor_fp8",
             lambda: torch._scaled_mm(a8, w8t, one, one, out_dtype=torch.bfloat16)))
    for name, fn in runs:
        ms = _timed(fn, dev)
        tf = gemm_flops(M, N, K) / (ms * 1e-3) / 1e12
        res[name] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                     "frac_fp8_peak": round(tf / fp8_peak, 4)}
    res["ours_over_library"] = round(res["cublaslt_per_tensor_fp8"]["us"] /
                                     res["ours_block_scaled"]["us"], 4)
    try:
        from torch.nn.functional import ScalingType, scaled_mm
        scaled_mm(a8, w8t, a_s.t(), ScalingType.BlockWise1x128, w_s.t(),
                  ScalingType.BlockWise128x128, output_dtype=torch.bfloat16)
        res["library_block_scaled"] = "ran (not timed)"
    except Exception as e:   # not offered on this GPU: record the library's own answer
        res["library_block_scaled"] = f"unavailable: {type(e).__name__}: {str(e)[:160]}"
    return res


SECTIONS = {"quantizer_sweep": run_sweep, "mla_gemm": run_mla, "decode_gemm": run_decode,
            "moe_grouped_gemm": run_moe, "library_reference": run_library_reference,
            "backward": lambda F, dev, hbm, fp8_peak: run_backward(F, dev, hbm, fp8_peak),
            "ue8m0_variant": lambda F, dev, hbm, fp8_peak: run_ue8m0(F, dev, hbm),
            "dense_requant": run_requant}


def run_extras(F, dev, peaks, fp8_peak, only=None, moe_shape=WL.MOE):
    """The other configurations, each kernel timed alone; `only` runs one section."""
    out = {"timing": "each kernel alone, L2 flushed (256 MB read) before every iteration, "
                     "mean of 10 after 3 warm-up, all enqueued behind a GPU spin so that no host "
                     "launch gap is timed; SM and memory clocks sampled during each section"}
    hbm = peaks["hbm_gbs"]
    for name, fn in SECTIONS.items():
        if only is not None and name != only:
            continue
        sampler = ClockSampler(dev.index if dev.index is not None else 0, memory=True)
        sampler.start()
        if name == "moe_grouped_gemm":
            out[name] = run_moe(F, dev, hbm, fp8_peak, moe_shape)
            if moe_shape is not WL.MOE:
                out[name]["reduced_workload"] = moe_shape.name
        else:
            out[name] = fn(F, dev, hbm, fp8_peak)
        out[name]["clocks"] = sampler.stop()
    if F.fp8bs_last_error() != F.FP8BS_OK:
        raise RuntimeError("a kernel reported a pipeline timeout in the extra workloads")
    return out


# --------------------------------------------------------------------------------------
# The oracle on the host cores (CPU baseline and the reference arm)
# --------------------------------------------------------------------------------------

def _oracle_sample(rows: int, a_bits, w_bits, threads: int):
    """The oracle's version of one step restricted to `rows` activation rows: quantize those
    rows and all of W, then the GEMM of those rows against every weight row. Returns seconds."""
    from oracle import oracle as O
    M, K = a_bits.shape
    N = w_bits.shape[0]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        acuts = np.linspace(0, rows, threads + 1).astype(int)
        aparts = list(ex.map(lambda i: O.quant_act_1x128(a_bits[acuts[i]:acuts[i + 1]]),
                             range(threads)))
        nb = (N + 127) // 128
        wcuts = (np.linspace(0, nb, threads + 1).astype(int) * 128).clip(max=N)
        wparts = list(ex.map(lambda i: O.quant_weight_128x128(w_bits[wcuts[i]:wcuts[i + 1]]),
                             range(threads)))
        qa = np.concatenate([p[0] for p in aparts])
        sa = np.concatenate([p[1] for p in aparts], axis=1)
        qw = np.concatenate([p[0] for p in wparts])
        sw = np.concatenate([p[1] for p in wparts], axis=0)
        mm, nn = np.meshgrid(np.arange(rows), np.arange(N), indexing="ij")
        pm, pn = mm.ravel(), nn.ravel()
        pcuts = np.linspace(0, pm.size, threads + 1).astype(int)
        list(ex.map(lambda i: O.gemm_points(qa, sa, qw, sw, pm[pcuts[i]:pcuts[i + 1]],
                                            pn[pcuts[i]:pcuts[i + 1]]), range(threads)))
    return time.perf_counter() - t0


def _host_inputs():
    a, w = WL.gemm_inputs(SHAPE, "cpu")
    from oracle import oracle as O
    O.build()
    return (a.view(torch.int16).numpy().view(np.uint16),
            w.view(torch.int16).numpy().view(np.uint16))


def _threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _calibrate_rows(a_bits, w_bits, threads, budget_s):
    """Rows of the oracle sample that take about budget_s seconds: two probes give the fixed
    cost (quantizing W) and the cost per activation row. The probes differ by at least 16 rows,
    so that the per-row cost stands out of the run-to-run noise of the fixed cost."""
    r1 = max(threads, 4)
    t1 = _oracle_sample(r1, a_bits, w_bits, threads)
    r2 = r1 + max(2 * threads, 16)
    t2 = _oracle_sample(r2, a_bits, w_bits, threads)
    per_row = max((t2 - t1) / (r2 - r1), 1e-6)
    fixed = max(t1 - r1 * per_row, 0.0)
    rows = int((budget_s - fixed) / per_row)
    return max(1, min(SHAPE.M, rows))


def cpu_baseline(budget_s: float = 20.0, single_core_budget_s: float = 8.0):
    """The oracle on all host cores (the reported baseline) and, beside it, on one core."""
    a_bits, w_bits = _host_inputs()
    threads = _threads()
    N, K = SHAPE.N, SHAPE.K
    rows = _calibrate_rows(a_bits, w_bits, threads, budget_s)
    t = _oracle_sample(rows, a_bits, w_bits, threads)
    value = gemm_flops(rows, N, K) / t / 1e12
    rows1 = _calibrate_rows(a_bits, w_bits, 1, single_core_budget_s)
    t1 = _oracle_sample(rows1, a_bits, w_bits, 1)
    return {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "seconds": round(t, 3),
            "sample": f"oracle step on {rows} of {SHAPE.M} activation rows: quantize those rows "
                      f"and all of W ({N}x{K}), then the FP64 block-scaled GEMM of the "
                      f"{rows}x{N}x{K} slab; value = 2*{rows}*{N}*{K} / wall time",
            "single_core": {"value": gemm_flops(rows1, N, K) / t1 / 1e12, "rows": rows1,
                            "seconds": round(t1, 3)}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    a_bits, w_bits = _host_inputs()
    threads = _threads()
    N, K = SHAPE.N, SHAPE.K
    per_step = max(0.5, args.ref_budget_s / max(1, args.steps + args.warmup))
    rows = _calibrate_rows(a_bits, w_bits, threads, per_step)
    for _ in range(args.warmup):
        _oracle_sample(rows, a_bits, w_bits, threads)
    times = [_oracle_sample(rows, a_bits, w_bits, threads) for _ in range(args.steps)]
    sec = sum(times) / len(times)
    value = gemm_flops(rows, N, K) / sec / 1e12
    sample = (f"each step: the oracle's quantize + FP64 block-scaled GEMM on {rows} of "
              f"{SHAPE.M} activation rows against all of W ({N}x{K}); "
              f"value = 2*{rows}*{N}*{K} / step time")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded dense workload, generated on the host)",
        "config": {"workload": SHAPE.name, "M": SHAPE.M, "N": N, "K": K, "out": "f64",
                   "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _free_port():
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def launch_ranks(n, impl):
    """`--gpus N` without an external launcher: start N copies of this command, one per GPU, with
    the rendezvous variables torchrun would set (127.0.0.1, a free port), and wait for all of
    them. Each rank runs an independent replica; rank 0 prints the line. Returns the worst exit
    code."""
    if impl == "ours" and torch.cuda.device_count() < n:
        print(f"bench.py: --gpus {n} needs {n} visible GPUs, found {torch.cuda.device_count()}",
              file=sys.stderr)
        return 2
    port = str(_free_port())
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=port)
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *sys.argv[1:]],
                                      env=env))
    codes = [p.wait() for p in procs]
    return max(codes, key=abs)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing on the host cores")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="--impl reference: host seconds for all warm-up and timed steps")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the quantizer sweep, MLA, MoE and backward workloads")
    ap.add_argument("--backward-only", action="store_true",
                    help="same as --only backward")
    ap.add_argument("--only", choices=sorted(SECTIONS),
                    help="time one section of the other workloads alone (one JSON object), "
                         "e.g. for ncu")
    ap.add_argument("--moe-experts", type=int, default=WL.MOE.experts,
                    help="with --only moe_grouped_gemm: scale the MoE workload down to this "
                         "many experts, same rows per expert (small ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank, world, local_rank = dist_env()
    if world == 1 and args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args.gpus, args.impl))
    if world > 1:
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend)
    try:
        if args.backward_only or args.only:
            section = args.only or "backward"
            line = section_only(rank, section, args.moe_experts) if args.impl == "ours" else None
        elif args.impl == "reference":
            line = run_reference(args, rank, world)
        else:
            line = run_ours(args, rank, world, local_rank)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
