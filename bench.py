#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on GB300.

One step = one forward (fa_fwd) and one backward (fa_bwd) over the workload
B=2, H=16, N=4096, d=128, causal, scale 1/sqrt(d), bf16 N(0,1) inputs (seed 0):
the one workload that runs every step of the path.  Throughput is algorithmic
TFLOPS: 4*B*H*N^2*d per forward and 10*B*H*N^2*d per backward (the five GEMMs
S, dP, dV, dK, dQ), both halved for the causal mask.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own copy of the
workload on its own GPU (weak scaling, no data-path collective); the timed region
is bracketed by a barrier and a synchronize, and the slowest rank's time counts.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle on the host cores instead (a
bounded row sample of the same workload per step).

The line ends with `targets`: the five configurations the parity and throughput
target is stated on (C1-C5), each with TFLOPS, its fraction of the measured bf16
GEMM peak and of the clock-derived tensor peak, and the max-abs error of a seeded
sample against the float64 oracle (checked in the cpu_baseline leg, the one leg
that runs the oracle), plus whether the forward at N = 16384, d = 128 reaches 60%
of the measured peak.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS (causal & non-causal) and % of GB300 dense BF16 peak"
UNIT = "TFLOPS"
WORKLOAD = dict(B=2, H=16, N=4096, d=128, causal=True)
WORKLOAD_NAME = "exact SDPA fwd+bwd, B=2 H=16 N=4096 d=128, causal, bf16 in, fp32 dQ/dK/dV"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}

# Forward/backward workloads reported beside the step (context, outside the timed region).
FWD_WORKLOADS = [
    ("B8_H16_N2048_d64_noncausal", 8, 16, 2048, 64, False, "normal"),
    ("B8_H16_N2048_d64_causal", 8, 16, 2048, 64, True, "normal"),
    ("B1_H16_N16384_d128_causal", 1, 16, 16384, 128, True, "normal"),
    ("B4_H8_N8192_d256_noncausal_boosted", 4, 8, 8192, 256, False, "boosted"),
    ("B2_H16_N4096_d128_causal", 2, 16, 4096, 128, True, "normal"),
    ("B4_H16_N4096_d96_causal", 4, 16, 4096, 96, True, "normal"),
    # fewer two-tile items than SMs: the one-tile mode
    ("B1_H8_N2048_d128_causal", 1, 8, 2048, 128, True, "normal"),
    ("B1_H2_N16384_d128_causal", 1, 2, 16384, 128, True, "normal"),
    # one head: the key ranges are cut over CTAs and merged
    ("B1_H1_N16384_d128_causal", 1, 1, 16384, 128, True, "normal"),
]
BWD_WORKLOADS = [
    ("B2_H16_N4096_d128_causal", 2, 16, 4096, 128, True),
    # fewer key-block CTAs than SMs: two CTAs per key block
    ("B1_H4_N4096_d128_causal", 1, 4, 4096, 128, True),
    ("B2_H16_N4096_d128_noncausal", 2, 16, 4096, 128, False),
    ("B8_H16_N2048_d64_causal", 8, 16, 2048, 64, True),
    ("B4_H16_N4096_d96_causal", 4, 16, 4096, 96, True),
]

# Split-KV decode against a long cache: bound by HBM.  One query row per sequence
# (CUDA-core kernel), and several rows per key/value head (four new tokens, or four
# query heads sharing a key/value head: tensor-core kernel).  (name, B, H, Hkv, Nq, Nk, d)
DEC_WORKLOADS = [
    ("B8_H32_Nq1_Nk32768_d128", 8, 32, 32, 1, 32768, 128),
    ("B1_H32_Nq1_Nk32768_d128", 1, 32, 32, 1, 32768, 128),
    ("B8_H32_Nq1_Nk32768_d64", 8, 32, 32, 1, 32768, 64),
    ("B4_H16_Nq1_Nk32768_d256", 4, 16, 16, 1, 32768, 256),
    ("B8_H32_Nq1_Nk32768_d96", 8, 32, 32, 1, 32768, 96),
    ("B8_H32_Nq4_Nk32768_d128", 8, 32, 32, 4, 32768, 128),
    ("B8_H32_Hkv8_Nq1_Nk32768_d128", 8, 32, 8, 1, 32768, 128),
]


# Paged decode: the same B8 H32 Nk32768 d128 cache in 16-token pages scattered at random.
PAGED_WORKLOADS = [
    ("B8_H32_Nq1_Nk32768_d128_page16", 8, 32, 1, 32768, 128, 16),
    ("B8_H32_Nq1_Nk32768_d128_page64", 8, 32, 1, 32768, 128, 64),
]


def decode_bytes(B, H, Nq, Nk, d, Hkv=None):
    """Algorithmic HBM bytes of one decode call: read K, V (bf16, Hkv heads) and q,
    write o (bf16) and L (fp32); the partial results stay in L2."""
    Hkv = H if Hkv is None else Hkv
    return 2 * B * Hkv * Nk * d * 2 + 2 * B * H * Nq * d * 2 + B * H * Nq * 4


def fwd_flops(B, H, N, d, causal):
    return 4.0 * B * H * N * N * d * (0.5 if causal else 1.0)


def bwd_flops(B, H, N, d, causal):
    return 10.0 * B * H * N * N * d * (0.5 if causal else 1.0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]), "hbm_gbs": float(p["hbm_gbs"]),
                "source": "measured (MEASURED_PEAKS.json, burst bf16 GEMM)"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback (no MEASURED_PEAKS.json)")


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if the kernel sources
    have not changed since it was captured; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel_key]
        if rec["source_digest"] != source_digest(rec["sources"]):
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


REJECTED_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks):
    """True when the sampled clocks disqualify a timed region: a hardware or thermal
    slowdown was active, or the median SM clock sat below 85% of its maximum with no
    reason reported."""
    reasons = set(clocks.get("reasons") or [])
    if reasons & set(REJECTED_REASONS):
        return True
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and smax and sm < 0.85 * smax and not (reasons - {"nvidia-smi unavailable"}))


# ------------------------------------------------------------------ ranks

def max_over_ranks(x, world, device):
    """The largest of every rank's value (the slowest rank sets the job's time)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step, world, step_ms):
    """Whole-job throughput: every rank ran its own copy of the step (weak scaling)."""
    return flops_per_rank_step * world / (step_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id is not None:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def run_forward_only(args):
    """`--only-forward B H N d causal [boosted]`: one forward shape, W untimed and K
    timed calls (CUDA events, L2 flushed before each), one JSON line.  A small,
    self-contained command for a profiler to capture a single forward launch."""
    import torch

    import exact_attention_26_gb300 as fa
    from exact_attention_26_gb300.inputs import boosted_qkv, normal_qkv

    vals = args.only_forward
    B, H, N, d, causal = (int(x) for x in vals[:5])
    gen = boosted_qkv if len(vals) > 5 and vals[5] == "boosted" else normal_qkv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load()
    q, k, v = (t.to(dev) for t in gen(B, H, N, d, seed=0))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ms = _time_call(torch, dev, lambda: fa.forward(q, k, v, causal=bool(causal), out=o, lse=lse),
                    flush, iters=args.steps, warm=args.warmup)
    status = fa.fa_device_status(None)
    if status != 0:
        raise RuntimeError(f"device status {fa.fa_status_string(status)}")
    tf = fwd_flops(B, H, N, d, bool(causal)) / (ms * 1e-3) / 1e12
    return {"only_forward": {"B": B, "H": H, "N": N, "d": d, "causal": bool(causal),
                             "inputs": gen.__name__}, "ms": round(ms, 5), "tflops": round(tf, 2)}


def run_backward_only(args):
    """`--only-backward B H N d causal`: one backward shape (fa_bwd on the output of one
    forward), W untimed and K timed calls (CUDA events, L2 flushed before each), one
    JSON line.  A small, self-contained command for a profiler to capture the
    backward's launches."""
    import torch

    import exact_attention_26_gb300 as fa
    from exact_attention_26_gb300.inputs import normal_qkv

    B, H, N, d, causal = (int(x) for x in args.only_backward)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load()
    q, k, v, do = (t.to(dev) for t in normal_qkv(B, H, N, d, seed=0, with_do=True))
    o, lse = fa.forward(q, k, v, causal=bool(causal))
    g = [torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(3)]
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ms = _time_call(torch, dev, lambda: fa.backward(q, k, v, o, lse, do, causal=bool(causal),
                                                    dq=g[0], dk=g[1], dv=g[2], workspace=ws),
                    flush, iters=args.steps, warm=args.warmup)
    status = fa.fa_device_status(None)
    if status != 0:
        raise RuntimeError(f"device status {fa.fa_status_string(status)}")
    tf = bwd_flops(B, H, N, d, bool(causal)) / (ms * 1e-3) / 1e12
    return {"only_backward": {"B": B, "H": H, "N": N, "d": d, "causal": bool(causal)},
            "ms": round(ms, 5), "tflops": round(tf, 2)}


def run_decode_only(args):
    """`--only-decode B H Hkv Nq Nk d`: one decode shape (automatic key ranges), W
    untimed and K timed calls (CUDA events, L2 flushed before each), one JSON line.  A
    small, self-contained command for a profiler to capture the decode's launches."""
    import torch

    import exact_attention_26_gb300 as fa
    from exact_attention_26_gb300.inputs import decode_qkv

    B, H, Hkv, Nq, Nk, d = (int(x) for x in args.only_decode)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fa.load()
    _, k, v = decode_qkv(B, Hkv, 1, Nk, d, seed=0, device=dev)
    q = torch.randn((B, H, Nq, d), generator=torch.Generator(device=dev).manual_seed(1),
                    device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, fa.fa_decode_workspace_bytes(B, H, Hkv, Nq, Nk, d, 0)),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ms = _time_call(torch, dev, lambda: fa.decode(q, k, v, out=o, lse=lse, workspace=ws), flush,
                    iters=args.steps, warm=args.warmup)
    status = fa.fa_device_status(None)
    if status != 0:
        raise RuntimeError(f"device status {fa.fa_status_string(status)}")
    gbs = decode_bytes(B, H, Nq, Nk, d, Hkv) / (ms * 1e-3) / 1e9
    return {"only_decode": {"B": B, "H": H, "Hkv": Hkv, "Nq": Nq, "Nk": Nk, "d": d},
            "kernel": "tcgen05" if fa.fa_decode_uses_tensor_cores(H, Hkv, Nq, d, 0) == 1 else "cuda-core",
            "splits": fa.fa_decode_num_splits(B, H, Hkv, Nq, Nk, d, 0),
            "ms": round(ms, 5), "GB/s": round(gbs, 1)}


def run_config():
    """The workload's description, the same for both arms of the benchmark."""
    B, H, N, d, causal = (WORKLOAD[k] for k in ("B", "H", "N", "d", "causal"))
    return {"workload": WORKLOAD_NAME, "B": B, "H": H, "N": N, "d": d, "causal": causal,
            "scale": 1.0 / math.sqrt(d),
            "inputs": "bf16(N(0,1)) q,k,v,dO from one torch CPU generator, seed 0",
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, outside "
                  "the per-step CUDA events)",
            "per_rank": "each rank runs its own copy (independent batches)"}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import exact_attention_26_gb300 as fa
    from exact_attention_26_gb300.inputs import boosted_qkv, normal_qkv

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    fa.load()
    B, H, N, d, causal = (WORKLOAD[k] for k in ("B", "H", "N", "d", "causal"))
    q_h, k_h, v_h, do_h = normal_qkv(B, H, N, d, seed=0, with_do=True)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        fa.forward(q, k, v, causal=causal, out=o, lse=lse)

    def bwd():
        fa.backward(q, k, v, o, lse, do, causal=causal, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        fwd()
        bwd()
    torch.cuda.synchronize(dev)
    status = fa.fa_device_status(None)
    if status != 0:
        raise RuntimeError(f"device status {fa.fa_status_string(status)} after warm-up")

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    def timed_region():
        sampler = ClockSampler(gpu_id)
        sampler.start()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        # Two extra flushes give the host a head start, so that it has enqueued the first
        # step's calls before the GPU reaches that step's first event (the host then
        # stays ahead: a step is ~0.5 ms of GPU work and far less host work).
        flush.zero_()
        flush.zero_()
        for it in range(args.steps):
            flush.zero_()  # L2 flush, outside the per-step events
            evs[it][0].record(stream)
            fwd()
            evs[it][1].record(stream)
            bwd()
            evs[it][2].record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        wall1 = time.perf_counter()
        clocks = sampler.stop()
        status = fa.fa_device_status(None)
        if status != 0:
            raise RuntimeError(f"device status {fa.fa_status_string(status)} in the timed region")
        return evs, wall0, wall1, clocks

    evs, wall0, wall1, clocks = timed_region()
    # A region that saw a hardware or thermal slowdown, or SM clocks stuck well below
    # their maximum with no reason given (a clock lock), is timed once more; every
    # rank takes the same decision.
    first_clocks = None
    if max_over_ranks(1.0 if clocks_rejected(clocks) else 0.0, world, dev) > 0:
        first_clocks = clocks
        evs, wall0, wall1, clocks = timed_region()

    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms_local = sum(fwd_ms) / len(fwd_ms) + sum(bwd_ms) / len(bwd_ms)
    step_ms = max_over_ranks(step_ms_local, world, dev)
    flops_step = fwd_flops(B, H, N, d, causal) + bwd_flops(B, H, N, d, causal)
    value = job_tflops(flops_step, world, step_ms)

    result = None
    if rank == 0:
        peaks = load_peaks()
        f_ms = statistics.mean(fwd_ms)
        b_ms = statistics.mean(bwd_ms)
        if b_ms >= f_ms:
            kern, kflops, kms = "fa_bwd (fa_bwd_pre_kernel<128> + fa_bwd_kernel<128, causal>)", \
                bwd_flops(B, H, N, d, causal), b_ms
            traffic = recorded_traffic("fa_bwd_d128_causal_b2h16n4096")
        else:
            kern, kflops, kms = "fa_fwd_kernel<128,causal>", fwd_flops(B, H, N, d, causal), f_ms
            traffic = recorded_traffic("fa_fwd_d128_causal_b2h16n4096")
        achieved = kflops / (kms * 1e-3) / 1e12
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": run_config(),
            "fwd_ms": round(f_ms, 5), "bwd_ms": round(b_ms, 5),
            "fwd_tflops": round(fwd_flops(B, H, N, d, causal) / (f_ms * 1e-3) / 1e12, 2),
            "bwd_tflops": round(bwd_flops(B, H, N, d, causal) / (b_ms * 1e-3) / 1e12, 2),
            # the same time under the 8 B H N^2 d convention, which leaves out the S and P
            # recompute (four of the five products instead of five)
            "bwd_tflops_excl_recompute": round(
                0.8 * bwd_flops(B, H, N, d, causal) / (b_ms * 1e-3) / 1e12, 2),
            "wall_ms_per_step_incl_flush": round((wall1 - wall0) * 1e3 / args.steps, 5),
            "roofline": {"bound": "tensor", "kernel": kern, "achieved": round(achieved, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "traffic": traffic, "peak_source": peaks["source"]},
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
        }
        if first_clocks is not None:
            result["remeasured"] = {"first_clocks": first_clocks,
                                    "why": "slowdown or low SM clock in the first timed region"}
    # End-to-end through the public API with host buffers: H2D of q, k, v, dO from
    # pinned memory, forward, backward, D2H of o, lse, dq, dk, dv, every step.
    e2e = run_e2e(args, fa, torch, dev, (q_h, k_h, v_h, do_h), causal, flops_step, world)
    e2e["ms"] = max_over_ranks(e2e["ms"], world, dev)
    if rank == 0:
        result["e2e"] = {"value": round(job_tflops(flops_step, world, e2e["ms"]), 2),
                         "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                         "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e["ms"], 5),
                         "pipelined": "HostPipeline: 2 steps in flight, H2D / kernels / D2H on "
                                      "separate streams",
                         "serial_ms_per_step": round(e2e["serial_ms"], 5),
                         "copy_only_ms_per_step": round(e2e["copy_ms"], 5),
                         "copy_note": "the step's H2D + D2H bytes on the two copy streams "
                                      "with no kernels: the host link's bound for e2e"}
        rates = unit_rates(fa, torch, dev, clocks)
        if rates is not None:
            result["unit_rates"] = rates
            pk_clk = rates.get("clock_derived_bf16_tflops")
            if pk_clk:
                result["roofline"]["peak_clock_derived"] = pk_clk
                result["roofline"]["frac_clock_derived"] = round(achieved / pk_clk, 4)
            ex2 = rates.get("ex2_per_sm_clk")
            if ex2:
                exps = B * H * N * N * (0.5 if causal else 1.0)  # one ex2 per score, fwd and bwd
                floor_ms = exps / (ex2 * rates["sms"] * rates["sm_mhz"] * 1e6) * 1e3
                result["ex2_floor_ms"] = {"fwd": round(floor_ms, 5), "bwd": round(floor_ms, 5)}
        if world == 1 and not args.no_extra:
            result["forward_workloads"] = sweep_forward(fa, torch, dev, flush, normal_qkv,
                                                        boosted_qkv, load_peaks(), rates)
            result["backward_workloads"] = sweep_backward(fa, torch, dev, flush, normal_qkv,
                                                          load_peaks())
            result["decode_workloads"] = sweep_decode(fa, torch, dev, flush, load_peaks())
            result["fp8_workloads"] = sweep_fp8(fa, torch, dev, flush, load_peaks())
            result["gqa_varlen_workloads"] = sweep_gqa_varlen(fa, torch, dev, flush, load_peaks())
        targets, jobs = None, []
        if world == 1 and not args.no_targets:
            targets, jobs = sweep_targets(fa, torch, dev, flush, load_peaks(), rates,
                                          (f_ms, b_ms), (q_h, k_h, v_h, do_h),
                                          (o, lse, dq, dk, dv))
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
            if targets is not None:
                parity_sample(targets, jobs)
        else:
            result["cpu_baseline"] = None
        if targets is not None:
            result["targets"] = targets  # last key: the shortest record of the line keeps it
    return result


# The configurations the target is stated on: (name, B, H, N, d, masks, inputs).
TARGET_CONFIGS = [
    ("C1_B1H1N128d64", 1, 1, 128, 64, (False, True), "normal"),
    ("C2_B8H16N2048d64", 8, 16, 2048, 64, (False, True), "normal"),
    ("C3_B1H16N16384d128", 1, 16, 16384, 128, (True,), "normal"),
    ("C4_B4H8N8192d256", 4, 8, 8192, 256, (False,), "boosted"),
]
TARGET_ROWS, TARGET_HEADS = 64, 2   # the oracle's seeded sample per configuration
FWD_TARGET = 0.60                   # forward fraction of the bf16 peak at N >= 8192, d = 128


def sweep_targets(fa, torch, dev, flush, peaks, rates, step_ms, step_inputs, step_outputs):
    """The target configurations C1-C5: forward (and, C5, backward) TFLOPS, their
    fraction of the measured bf16 GEMM peak and of the clock-derived peak, and the GPU
    results of a seeded sample of rows and heads for the oracle to check in the
    cpu_baseline leg (C5 reuses the timed step's inputs and outputs)."""
    from exact_attention_26_gb300.inputs import boosted_qkv, normal_qkv, sample_rows
    pk = peaks["bf16_tflops"]
    pk_clk = (rates or {}).get("clock_derived_bf16_tflops")

    def perf(flops, ms):
        tf = flops / (ms * 1e-3) / 1e12
        e = {"tflops": round(tf, 1), "frac": round(tf / pk, 3)}
        if pk_clk:
            e["frac_clk"] = round(tf / pk_clk, 3)
        return e

    out, jobs = {}, []
    for name, B, H, N, d, masks, kind in TARGET_CONFIGS:
        gen = boosted_qkv if kind == "boosted" else normal_qkv
        qh, kh, vh = gen(B, H, N, d, seed=0)
        q, k, v = (t.to(dev) for t in (qh, kh, vh))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        rows = sample_rows(N, TARGET_ROWS, seed=2)
        nh = min(TARGET_HEADS, B * H)
        entry = {}
        for causal in masks:
            ms = _time_call(torch, dev, lambda: fa.forward(q, k, v, causal=causal, out=o, lse=lse),
                            flush)
            e = perf(fwd_flops(B, H, N, d, causal), ms)
            torch.cuda.synchronize(dev)
            jobs.append({"entry": e, "gen": kind, "shape": (B, H, N, d), "causal": causal,
                         "rows": rows, "heads": nh,
                         "o": o.reshape(B * H, N, d)[:nh, rows].float().cpu(),
                         "lse": lse.reshape(B * H, N)[:nh, rows].cpu()})
            entry["causal" if causal else "noncausal"] = e
        out[name] = entry if len(masks) > 1 else entry[next(iter(entry))]
        del q, k, v, o, lse
    B, H, N, d, causal = (WORKLOAD[k] for k in ("B", "H", "N", "d", "causal"))
    o, lse, dq, dk, dv = step_outputs
    rows = sample_rows(N, TARGET_ROWS, seed=2)
    c5 = {"fwd": perf(fwd_flops(B, H, N, d, causal), step_ms[0]),
          "bwd": perf(bwd_flops(B, H, N, d, causal), step_ms[1])}
    jobs.append({"entry": c5, "gen": "step", "shape": (B, H, N, d), "causal": causal,
                 "rows": rows, "heads": 1, "inputs": step_inputs,
                 "o": o.reshape(B * H, N, d)[:1, rows].float().cpu(),
                 "lse": lse.reshape(B * H, N)[:1, rows].cpu(),
                 "grads": [t.reshape(B * H, N, d)[0].cpu() for t in (dq, dk, dv)]})
    out["C5_B2H16N4096d128_causal"] = c5
    c3 = out["C3_B1H16N16384d128"]["frac"]
    out["fwd_N16384_d128"] = {"frac": c3, "target": FWD_TARGET, "met": bool(c3 >= FWD_TARGET)}
    return out, jobs


def parity_sample(targets, jobs):
    """The oracle on each target's seeded sample (the rows and heads whose GPU results
    sweep_targets kept): max-abs error of O, L and, for the timed step, of dQ, dK, dV
    over its first head, and whether each is within the parity tolerance."""
    from exact_attention_26_gb300.inputs import boosted_qkv, normal_qkv, to_f64
    from oracle import default as oracle_default

    orc = oracle_default()
    ok = True
    for job in jobs:
        B, H, N, d = job["shape"]
        nh, rows = job["heads"], job["rows"].numpy()
        if job["gen"] == "step":
            q, k, v, do = job["inputs"]
        else:
            gen = boosted_qkv if job["gen"] == "boosted" else normal_qkv
            q, k, v = gen(B, H, N, d, seed=0)
        sel = [to_f64(t.reshape(1, B * H, N, d)[:, :nh]) for t in (q, k, v)]
        ro, rl = orc.fwd_rows(*sel, rows, causal=job["causal"])
        go, gl = job["o"].numpy()[None], job["lse"].numpy()[None]
        err_o = float(np.max(np.abs(go - ro)))
        err_l = float(np.max(np.abs(gl - rl)))
        ok &= bool(np.all(np.abs(go - ro) <= np.maximum(1e-2, 2.0 ** -7 * np.abs(ro))))
        ok &= err_l <= 1e-3
        errs = [err_o, err_l]
        if "grads" in job:
            dsel = to_f64(do.reshape(1, B * H, N, d)[:, :1])
            ref = orc.bwd(*[x[:, :1] for x in sel], dsel, causal=job["causal"])
            for g, r in zip(job["grads"], ref):
                e = float(np.max(np.abs(g.numpy() - r[0, 0])))
                errs.append(e)
                ok &= e <= 2e-2
        job["entry"]["err"] = [float(f"{e:.2e}") for e in errs]
    targets["parity"] = {"ok": bool(ok), "err": "max-abs [O, L] (+ [dQ, dK, dV] of head 0 "
                         "for C5) vs the float64 oracle", "tol": "O max(1e-2, 2^-7|O|), "
                         "L 1e-3, grads 2e-2"}


def run_e2e(args, fa, torch, dev, host_inputs, causal, flops_step, world):
    """The step through the public API with host buffers: every step copies q, k, v,
    dO from pinned host memory and o, lse, dq, dk, dv back.  `HostPipeline` keeps two
    steps in flight on separate copy and compute streams; the serial form (one
    stream, as a caller without it would write) is timed too, for reference."""
    from exact_attention_26_gb300.pipeline import HostPipeline
    pin = [t.pin_memory() for t in host_inputs]
    B, H, N, d = pin[0].shape
    outs_h = [torch.empty(pin[0].shape, dtype=torch.bfloat16).pin_memory(),
              torch.empty(pin[0].shape[:3], dtype=torch.float32).pin_memory()] + \
             [torch.empty(pin[0].shape, dtype=torch.float32).pin_memory() for _ in range(3)]
    n = max(3, min(args.steps, 30))

    pipe = HostPipeline(B, H, N, d, causal=causal, device=dev, depth=2)
    for _ in range(3):
        pipe.step(pin, outs_h)
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(pipe.s_h2d)
    for _ in range(n):
        pipe.step(pin, outs_h)
    b.record(pipe.s_d2h)
    b.synchronize()
    ms = a.elapsed_time(b) / n

    # serial reference: the same calls on one stream
    dq_, dk_, dv_ = (torch.empty(pin[0].shape, dtype=torch.float32, device=dev) for _ in range(3))
    dev_in = [torch.empty_like(t, device=dev) for t in pin]
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        for dst, src in zip(dev_in, pin):
            dst.copy_(src, non_blocking=True)
        q, k, v, do = dev_in
        o, lse = fa.forward(q, k, v, causal=causal)
        g = fa.backward(q, k, v, o, lse, do, causal=causal, dq=dq_, dk=dk_, dv=dv_, workspace=ws)
        for dst, src in zip(outs_h, (o, lse) + tuple(g)):
            dst.copy_(src, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    b.synchronize()
    serial_ms = a.elapsed_time(b) / n

    # the copy bound: the same per-step H2D and D2H on the pipeline's two copy
    # streams with no kernels (the host link's limit for this step's bytes)
    sl = pipe.slots[0]
    dev_out = [sl["o"], sl["lse"]] + sl["g"]
    a.record(pipe.s_h2d)
    pipe.s_d2h.wait_stream(pipe.s_h2d)
    for _ in range(n):
        with torch.cuda.stream(pipe.s_h2d):
            for dst, src in zip(sl["in"], pin):
                dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(pipe.s_d2h):
            for dst, src in zip(outs_h, dev_out):
                dst.copy_(src, non_blocking=True)
    pipe.s_h2d.wait_stream(pipe.s_d2h)
    b.record(pipe.s_h2d)
    b.synchronize()
    copy_ms = a.elapsed_time(b) / n
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    return {"ms": ms, "serial_ms": serial_ms, "copy_ms": copy_ms, "h2d": h2d, "d2h": d2h}


def _time_call(torch, dev, fn, flush, iters=20, warm=3):
    """Median device time of fn() between CUDA events, L2 flushed before each call.
    Every iteration is enqueued before any is waited for, so the host's per-call
    work (argument checks, tensor-map encoding) overlaps the previous flush and
    never leaves the GPU idle inside the events."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize(dev)
    evs = []
    flush.zero_()
    for _ in range(iters):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize(dev)
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def unit_rates(fa, torch, dev, clocks):
    """The library's unit-rate probes (dense bf16 MMA and MUFU ex2 per SM clock), run
    once outside the timed region, and the peaks they give at this GPU's SM count and
    clocks: the clock-derived tensor peak at the maximum SM clock, the ex2 rate at the
    median SM clock seen under load."""
    try:
        r = fa.probe_unit_rates(2048)
    except Exception as exc:  # reported, never fatal: the probes are context
        return {"error": str(exc)}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"sms": sms, "mma_bf16_flop_per_sm_clk_n256": round(r["mma_bf16_n256_flop_per_clk"], 1),
           "mma_bf16_flop_per_sm_clk_n64": round(r["mma_bf16_n64_flop_per_clk"], 1),
           "ex2_per_sm_clk": round(r["ex2_per_clk"], 2),
           "sm_max_mhz": clocks.get("sm_max_mhz"), "sm_mhz": clocks.get("sm_mhz")}
    if out["sm_max_mhz"]:
        out["clock_derived_bf16_tflops"] = round(
            r["mma_bf16_n256_flop_per_clk"] * sms * out["sm_max_mhz"] * 1e6 / 1e12, 1)
    if not out["sm_mhz"]:
        out["ex2_per_sm_clk"] = None
    return out


def sweep_forward(fa, torch, dev, flush, normal_qkv, boosted_qkv, peaks, rates=None):
    out = {}
    ex2 = (rates or {}).get("ex2_per_sm_clk")
    for name, B, H, N, d, causal, kind in FWD_WORKLOADS:
        gen = boosted_qkv if kind == "boosted" else normal_qkv
        q, k, v = (t.to(dev) for t in gen(B, H, N, d, seed=0))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        ms = _time_call(torch, dev, lambda: fa.forward(q, k, v, causal=causal, out=o, lse=lse),
                        flush)
        tf = fwd_flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 5), "tflops": round(tf, 2),
                     "frac_of_peak": round(tf / peaks["bf16_tflops"], 4)}
        if ex2:  # the exponential ceiling: one ex2 per score element
            exps = B * H * N * N * (0.5 if causal else 1.0)
            out[name]["ex2_floor_ms"] = round(
                exps / (ex2 * rates["sms"] * rates["sm_mhz"] * 1e6) * 1e3, 5)
        del q, k, v, o, lse
    return out


def sweep_backward(fa, torch, dev, flush, normal_qkv, peaks):
    out = {}
    for name, B, H, N, d, causal in BWD_WORKLOADS:
        q, k, v, do = (t.to(dev) for t in normal_qkv(B, H, N, d, seed=0, with_do=True))
        o, lse = fa.forward(q, k, v, causal=causal)
        g = [torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(3)]
        ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        ms = _time_call(torch, dev, lambda: fa.backward(q, k, v, o, lse, do, causal=causal,
                                                        dq=g[0], dk=g[1], dv=g[2], workspace=ws),
                        flush)
        tf = bwd_flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 5), "tflops": round(tf, 2),
                     "frac_of_peak": round(tf / peaks["bf16_tflops"], 4),
                     "tflops_excl_recompute": round(0.8 * tf, 2)}
        del q, k, v, do, o, lse, g, ws
    return out


def sweep_decode(fa, torch, dev, flush, peaks):
    """Decode calls (automatic key-range split) against the measured HBM read rate (a
    decode's traffic is almost all reads of the cache); the copy rate is kept beside it."""
    from exact_attention_26_gb300.inputs import decode_qkv
    out = {}
    read_peak = None
    for name, B, H, Hkv, Nq, Nk, d in DEC_WORKLOADS:
        _, k, v = decode_qkv(B, Hkv, 1, Nk, d, seed=0, device=dev)
        gq = torch.Generator(device=dev).manual_seed(1)
        q = torch.randn((B, H, Nq, d), generator=gq, device=dev).to(torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
        need = fa.fa_decode_workspace_bytes(B, H, Hkv, Nq, Nk, d, 0)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        if read_peak is None:
            read_peak = fa.probe_read_bandwidth(k, iters=5)
            out["read_peak"] = {"GB/s": round(read_peak, 1),
                                "how": "fa_probe_read_bandwidth: 16-byte non-allocating loads "
                                       "over the first cache's K (2.1 GB), 5 passes",
                                "copy_GB/s": peaks["hbm_gbs"]}
        ms = _time_call(torch, dev, lambda: fa.decode(q, k, v, out=o, lse=lse, workspace=ws), flush)
        gbs = decode_bytes(B, H, Nq, Nk, d, Hkv) / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 5), "GB/s": round(gbs, 1),
                     "splits": fa.fa_decode_num_splits(B, H, Hkv, Nq, Nk, d, 0),
                     "kernel": ("tcgen05" if fa.fa_decode_uses_tensor_cores(H, Hkv, Nq, d, 0) == 1
                                else "cuda-core"),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                                  "peak": round(read_peak, 1), "unit": "GB/s",
                                  "frac": round(gbs / read_peak, 4),
                                  "frac_of_copy_rate": round(gbs / peaks["hbm_gbs"], 4)}}
        del q, k, v, o, lse, ws
    from exact_attention_26_gb300.inputs import paged_cache
    for name, B, H, Nq, Nk, d, ps in PAGED_WORKLOADS:
        q, k, v = decode_qkv(B, H, Nq, Nk, d, seed=0, device=dev)
        kc, vc, bt = paged_cache(k, v, ps)
        del k, v
        lens = torch.full((B,), Nk, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
        need = fa.fa_decode_paged_workspace_bytes(B, H, H, Nq, d, ps, Nk // ps, 0)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        ms = _time_call(torch, dev, lambda: fa.decode_paged(q, kc, vc, bt, lens, out=o, lse=lse,
                                                            workspace=ws), flush)
        gbs = decode_bytes(B, H, Nq, Nk, d) / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 5), "GB/s": round(gbs, 1),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                                  "peak": round(read_peak, 1), "unit": "GB/s",
                                  "frac": round(gbs / read_peak, 4),
                                  "frac_of_copy_rate": round(gbs / peaks["hbm_gbs"], 4)}}
        del q, kc, vc, bt, o, lse, ws
    return out


# Grouped-query attention (query heads sharing key/value heads) and packed sequences
# of mixed lengths, forward and backward.
GQA_WORKLOADS = [
    ("B2_H32_Hkv8_N4096_d128_causal", 2, 32, 8, 4096, 128, True),
]
# 16 packed sequences, lengths drawn uniformly from [256, 8192] (torch generator seed 0,
# sorted), token-major, 16 query heads over 4 key/value heads, d = 128, causal.
VARLEN_WORKLOAD = ("T_mix16_256to8192_H16_Hkv4_d128_causal", 16, 256, 8192, 16, 4, 128, True)


def varlen_lengths(n, lo, hi, seed=0):
    import torch
    g = torch.Generator().manual_seed(seed)
    return sorted(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


def sweep_gqa_varlen(fa, torch, dev, flush, peaks):
    """GQA and packed variable-length calls; FLOPs count every query head's products
    (and, packed, each sequence's own N^2), the same convention as the fixed shapes."""
    from exact_attention_26_gb300.inputs import gqa_qkv, varlen_qkv
    out = {}
    pk = peaks["bf16_tflops"]

    def entry(ms_f, ms_b, ffl, bfl):
        tf, tb = ffl / (ms_f * 1e-3) / 1e12, bfl / (ms_b * 1e-3) / 1e12
        return {"fwd_ms": round(ms_f, 5), "fwd_tflops": round(tf, 2), "fwd_frac_of_peak": round(tf / pk, 4),
                "bwd_ms": round(ms_b, 5), "bwd_tflops": round(tb, 2), "bwd_frac_of_peak": round(tb / pk, 4)}

    for name, B, H, Hkv, N, d, causal in GQA_WORKLOADS:
        q, k, v, do = (t.to(dev) for t in gqa_qkv(B, H, Hkv, N, d, seed=0, with_do=True))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        g = [torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v)]
        ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        ms_f = _time_call(torch, dev, lambda: fa.forward(q, k, v, causal=causal, out=o, lse=lse), flush)
        ms_b = _time_call(torch, dev, lambda: fa.backward(q, k, v, o, lse, do, causal=causal, dq=g[0],
                                                          dk=g[1], dv=g[2], workspace=ws), flush)
        out[name] = entry(ms_f, ms_b, fwd_flops(B, H, N, d, causal), bwd_flops(B, H, N, d, causal))
        del q, k, v, do, o, lse, g, ws
    name, n, lo, hi, H, Hkv, d, causal = VARLEN_WORKLOAD
    lens = varlen_lengths(n, lo, hi)
    q, k, v, cu = varlen_qkv(lens, H, Hkv, d, seed=0)
    gen = torch.Generator().manual_seed(1)
    do = torch.randn(q.shape, generator=gen).to(torch.bfloat16)
    q, k, v, cu, do = (t.to(dev) for t in (q, k, v, cu, do))
    mx = max(lens)
    o, lse = fa.forward_varlen(q, k, v, cu, mx, causal=causal)
    g = [torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v)]
    ws = torch.empty(fa.fa_bwd_workspace_bytes(n, H, mx, d), dtype=torch.uint8, device=dev)
    ms_f = _time_call(torch, dev, lambda: fa.forward_varlen(q, k, v, cu, mx, causal=causal, out=o,
                                                            lse=lse), flush)
    ms_b = _time_call(torch, dev, lambda: fa.backward_varlen(q, k, v, o, lse, do, cu, mx, causal=causal,
                                                             dq=g[0], dk=g[1], dv=g[2], workspace=ws),
                      flush)
    ffl = sum(fwd_flops(1, H, L, d, causal) for L in lens)
    bfl = sum(bwd_flops(1, H, L, d, causal) for L in lens)
    out[name] = dict(entry(ms_f, ms_b, ffl, bfl), tokens=int(sum(lens)), max_seqlen=mx)
    return out


# Low-precision forward: e4m3 inputs (per-128-row scales of Q and K, per-head scale of
# V), both products on the tensor cores with 8-bit operands.
FP8_WORKLOADS = [
    ("B1_H16_N16384_d128_causal", 1, 16, 16384, 128, True),
    ("B2_H16_N4096_d128_causal", 2, 16, 4096, 128, True),
    ("B4_H8_N8192_d128_noncausal", 4, 8, 8192, 128, False),
]
# nominal dense e4m3 / bf16 tensor rates of the part (4.5 / 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0


def sweep_fp8(fa, torch, dev, flush, peaks):
    """fa_fwd_fp8 against the fp8 tensor peak (the measured bf16 GEMM rate times the
    nominal e4m3/bf16 ratio), and the quantiser against the HBM copy rate."""
    from exact_attention_26_gb300.inputs import normal_qkv
    out = {}
    peak8 = peaks["bf16_tflops"] * FP8_OVER_BF16
    for name, B, H, N, d, causal in FP8_WORKLOADS:
        q, k, v = (t.to(dev) for t in normal_qkv(B, H, N, d, seed=0))
        qc, qd = fa.quantize_fp8(q, 128)
        kc, kd = fa.quantize_fp8(k, 128)
        vc, vd = fa.quantize_fp8(v, 0, transpose=True)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        ms = _time_call(torch, dev, lambda: fa.forward_fp8(qc, kc, vc, qd, kd, vd, causal=causal,
                                                           out=o, lse=lse), flush)
        tf = fwd_flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        # quantiser: algorithmic bytes = read x (bf16) once + write the codes
        ws = torch.empty(max(fa.fa_quantize_fp8_workspace_bytes(B * H, N, d), 16),
                         dtype=torch.uint8, device=dev)
        qms = _time_call(torch, dev, lambda: fa.quantize_fp8(q, 128, workspace=ws), flush)
        gbs = (q.numel() * 3) / (qms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 5), "tflops": round(tf, 2),
                     "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak8,
                                  "unit": "TFLOP/s", "frac": round(tf / peak8, 4),
                                  "peak_source": "measured bf16 GEMM x nominal e4m3/bf16 ratio 2"},
                     "quantize_ms": round(qms, 5), "quantize_GB/s": round(gbs, 1),
                     "quantize_frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del q, k, v, qc, kc, vc, qd, kd, vd, o, lse, ws
    return out


# ------------------------------------------------------------------ oracle timing

_INPUTS = None


def _workload_heads(nheads):
    """The first `nheads` (batch, head) pairs of the workload's seeded inputs,
    upcast to float64 as [1, nheads, N, d] arrays (the bf16 tensors are cached)."""
    global _INPUTS
    from exact_attention_26_gb300.inputs import normal_qkv, to_f64
    if _INPUTS is None:
        B, H, N, d = (WORKLOAD[k] for k in ("B", "H", "N", "d"))
        _INPUTS = tuple(t.reshape(1, B * H, N, d)
                        for t in normal_qkv(B, H, N, d, seed=0, with_do=True))
    return tuple(to_f64(t[:, :nheads]) for t in _INPUTS)


def _oracle_sample(nrows, nheads=1, nthreads=None):
    """A bounded sample of the step on the CPU: forward and backward of `nrows`
    seeded query rows in each of the first `nheads` heads of the workload, on
    `nthreads` host threads (default: every core of the affinity mask).
    Returns (seconds, flops, rows, heads)."""
    from exact_attention_26_gb300.inputs import sample_rows
    from oracle import default as oracle_default

    orc = oracle_default()
    N, d, causal = WORKLOAD["N"], WORKLOAD["d"], WORKLOAD["causal"]
    q, k, v, do = _workload_heads(nheads)
    rows = sample_rows(N, nrows, seed=2).numpy()
    keys = (rows + 1) if causal else np.full(rows.shape, N)
    flops = float(nheads * ((4.0 + 10.0) * d * keys).sum())
    t0 = time.perf_counter()
    orc.fwd_rows(q, k, v, rows, causal=causal, nthreads=nthreads)
    orc.bwd_rows(q, k, v, do, rows, causal=causal, nthreads=nthreads)
    return time.perf_counter() - t0, flops, rows.size, nheads


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _sample_size(seconds):
    """(rows, heads) so that one sample takes about `seconds`: rows first, then heads."""
    max_heads = WORKLOAD["B"] * WORKLOAD["H"]
    N = WORKLOAD["N"]
    t, _, n, _ = _oracle_sample(min(512, N), 1)
    rows = int(max(8, min(N, seconds * n / max(t, 1e-9))))
    if rows < N:
        return rows, 1
    t_head, _, _, _ = _oracle_sample(N, 1)
    return N, int(max(1, min(max_heads, round(seconds / max(t_head, 1e-9)))))


def cpu_baseline(target_seconds):
    step_flops = fwd_flops(WORKLOAD["B"], WORKLOAD["H"], WORKLOAD["N"], WORKLOAD["d"],
                           WORKLOAD["causal"]) + bwd_flops(WORKLOAD["B"], WORKLOAD["H"],
                                                           WORKLOAD["N"], WORKLOAD["d"],
                                                           WORKLOAD["causal"])
    rows, heads = _sample_size(target_seconds)
    secs, flops, n, h = _oracle_sample(rows, heads)
    # the same oracle on one thread, on a sample about a quarter as long in time
    rows1 = max(16, min(WORKLOAD["N"], int(rows * heads / max(1, _cores()) / 4)))
    secs1, flops1, n1, _ = _oracle_sample(rows1, 1, nthreads=1)
    return {"value": round(flops / secs / 1e12, 6), "unit": UNIT, "cores": _cores(),
            "kind": "oracle",
            "sample": f"float64 oracle forward + backward of {n} seeded query rows in each of "
                      f"{h} heads of the workload ({secs:.1f} s on {_cores()} host threads; "
                      "same FLOP convention)",
            "single_core": {"value": round(flops1 / secs1 / 1e12, 6), "unit": UNIT, "cores": 1,
                            "sample": f"{n1} seeded query rows of one head ({secs1:.1f} s on "
                                      "one host thread)"},
            # the whole step at the sampled rate (extrapolated, not run)
            "extrapolated_full_step_s": round(step_flops / (flops / secs), 1)}


def run_reference(args):
    """The oracle as it stands, timed on the host cores: each step a bounded row
    sample of the workload sized so the whole run stays within a few minutes."""
    total_budget = 150.0
    rows, heads = _sample_size(total_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_sample(rows, heads)
    secs, flops = 0.0, 0.0
    n, h = rows, heads
    for _ in range(args.steps):
        s, f, n, h = _oracle_sample(rows, heads)
        secs += s
        flops += f
    value = flops / secs / 1e12
    sample = (f"float64 oracle forward + backward of {n} seeded query rows in each of {h} "
              f"heads per step, {_cores()} host threads")
    return {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-workload forward/backward sweep")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the C1-C5 target configurations and their oracle sample")
    ap.add_argument("--only-forward", nargs="+", metavar="B H N d causal [boosted]",
                    help="time one forward shape only (a small case for a profiler)")
    ap.add_argument("--only-backward", nargs=5, metavar=("B", "H", "N", "d", "causal"),
                    help="time one backward shape only (a small case for a profiler)")
    ap.add_argument("--only-decode", nargs=6, metavar=("B", "H", "Hkv", "Nq", "Nk", "d"),
                    help="time one decode shape only (a small case for a profiler)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.only_forward:
        if len(args.only_forward) not in (5, 6):
            ap.error("--only-forward takes B H N d causal [boosted]")
        print(json.dumps(run_forward_only(args)), flush=True)
        return

    if args.only_backward:
        print(json.dumps(run_backward_only(args)), flush=True)
        return
    if args.only_decode:
        print(json.dumps(run_decode_only(args)), flush=True)
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        result = run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
