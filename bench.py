#!/usr/bin/env python3
"""Benchmark: DeepSeekMoE layer forward at the V3 shape on B300.

One step = the whole hot path on one batch: routing (sigmoid affinities,
biased top-8, gates, loads), permutation with 1x128 FP8 quantisation, grouped
GEMM 1 (W1/W3) with the SwiGLU + FP8 epilogue, grouped GEMM 2 (W2), combine
h' = u + shared + sum g*FFN, and the bias update — 256 routed experts + 1
shared, d=7168, I=2048, T=8192 tokens, Zipf(1.1)-skewed expert popularity,
FP8 E4M3 expert weights resident in HBM with 128x128 scales.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Multi-GPU (torchrun): replicas, one per GPU,
no collective on the data path (weak scaling; value = all ranks' tokens / the
slowest rank's time). `--impl reference` times the FP64 CPU oracle on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer fwd tokens/s @V3 shape; FP8 grouped-GEMM % of B300 FP8 peak"
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor throughput (4.5 / 2.25 PFLOP/s)
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNELS_PER_STEP = 11        # split, gate GEMM, select | count, scan, rank, scatter | GEMM1 | GEMM2 | combine | bias


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def layer_flops(sh):
    R = sh.T * sh.K + sh.T
    g1 = 2.0 * R * (2 * sh.I) * sh.d
    g2 = 2.0 * R * sh.d * sh.I
    return g1, g2


# --------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------

def oracle_sample_timing(sh, layer_inputs, n_tokens: int, seed: int):
    """Times the FP64 oracle computing h' for n_tokens tokens of the workload:
    their routing against all 256 centroids, the 1x128 quantisation of their
    rows, the 128x128 quantisation of the weights of every expert they use,
    the SwiGLU FFNs and the combine. Weights are fetched to host memory
    before the clock starts. Returns (tokens/s, seconds, threads)."""
    import numpy as np
    import torch

    import oracle
    u, cent, bias, weight_fn = layer_inputs
    rng = np.random.Generator(np.random.PCG64(seed))
    toks = np.sort(rng.choice(sh.T, n_tokens, replace=False))
    r = oracle.route(u[torch.as_tensor(toks)], cent, bias, sh.K, sh.n_groups, sh.topk_groups)
    need = sorted(set(r.topk_idx.ravel().tolist()) | {sh.N})
    cache = {e: weight_fn(e) for e in need}
    t0 = time.perf_counter()
    oracle.layer_tokens(u, cent, bias, sh.K, lambda e: cache[e], toks, fp8=sh.fp8, n_groups=sh.n_groups,
                        topk_groups=sh.topk_groups)
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt, oracle.threads()


def host_layer_inputs(sh, device):
    import torch

    import synthetic as S
    u = S.tokens(sh, seed=0)
    cent = S.centroids(sh, zipf=True)
    bias = S.bias(sh)
    gen_dev = device if device is not None else "cpu"
    return u, cent, bias, (lambda e: tuple(w.cpu() for w in S.expert_weights(sh, e, device=gen_dev)))


def run_reference(args):
    """The FP64 oracle on the host cores, a bounded sample per step."""
    import torch

    import synthetic as S
    ws, rank, local = dist_env()
    if ws > 1 and rank != 0:
        return
    sh = S.LAYER_V3
    dev = f"cuda:{local}" if torch.cuda.is_available() else None
    inputs = host_layer_inputs(sh, dev)
    per_step = max(1, int(os.environ.get("REF_TOKENS_PER_STEP", "1")))
    for i in range(args.warmup):
        oracle_sample_timing(sh, inputs, per_step, seed=1000 + i)
    times, cores = [], 1
    for i in range(args.steps):
        _, dt, cores = oracle_sample_timing(sh, inputs, per_step, seed=i)
        times.append(dt)
    total = sum(times)
    value = per_step * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "v3-layer-fp8", "T": sh.T, "d": sh.d, "N": sh.N, "shared": 1, "K": sh.K,
                   "I": sh.I, "popularity": "zipf(1.1)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} token(s) of the T=8192 V3 FP8 layer per step: routing, FP8 "
                                   f"quantisation of the token and of its experts' weights, FFNs, combine"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------

def run_ours(args):
    import torch

    import mixture_experts_layer_90_b300 as moe
    import synthetic as S

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sh = S.LAYER_V3

    # ---- set-up (untimed): weights generated and quantised on the device ----
    cent = S.centroids(sh, zipf=True).to(dev)
    bias = S.bias(sh).to(dev)
    layer = moe.MoELayer.build(sh.d, sh.N, sh.K, sh.I, cent, bias,
                               lambda e: S.expert_weights(sh, e, device=dev), fp8=True, gamma=sh.gamma)
    u_bufs = [S.tokens(sh, seed=s, device=dev) for s in (0, 7)]     # alternate two token batches
    out = torch.empty_like(u_bufs[0])
    torch.cuda.synchronize()
    assert moe.device_status() == 0

    n_ev = len(moe.LAYER_STAGES) + 1
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    for i in range(args.warmup):
        layer.forward(u_bufs[i % 2], out)
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    with ClockSampler(local) as clocks:
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(args.steps):
            layer.forward(u_bufs[i % 2], out, stage_events=events[i])
        t1.record()
        barrier()
    status = moe.device_status()
    assert status == 0, f"device status {status}"
    elapsed_ms = t0.elapsed_time(t1)
    if ws > 1:
        tt = torch.tensor([elapsed_ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(tt.item())
    stage_ms = {name: statistics.mean(ev[j].elapsed_time(ev[j + 1]) for ev in events)
                for j, name in enumerate(moe.LAYER_STAGES)}

    # ---- end to end through the host-buffer C call ----
    u_host = [b.cpu().pin_memory() for b in u_bufs]
    out_host = torch.empty_like(u_host[0]).pin_memory()
    e_steps = max(1, min(args.steps, 50))
    for i in range(2):
        layer.forward_host(u_host[i % 2], out_host)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(e_steps):
        layer.forward_host(u_host[i % 2], out_host)
    e1.record()
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    if ws > 1:
        tt = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(tt.item())
    assert moe.device_status() == 0

    tokens = sh.T * args.steps * ws
    value = tokens / (elapsed_ms / 1000.0)
    g1, g2 = layer_flops(sh)
    pk, src = peaks()
    fp8_peak = pk["bf16_tflops_sustained"] * FP8_OVER_BF16
    t1s = stage_ms["gemm1_swiglu"] / 1000.0
    t2s = stage_ms["gemm2"] / 1000.0
    gemm1_tflops = g1 / t1s / 1e12
    gemm_pct = 100.0 * (g1 + g2) / (t1s + t2s) / 1e12 / fp8_peak
    traffic = None
    tp = os.path.join(ROOT, "profiles", "gemm1_traffic.json")
    if os.path.exists(tp):
        with open(tp) as f:
            traffic = json.load(f).get("bytes_per_launch")

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "v3-layer-fp8", "T": sh.T, "d": sh.d, "N": sh.N, "shared": 1, "K": sh.K,
                   "I": sh.I, "popularity": "zipf(1.1)", "global_batch": sh.T * ws, "parallelism": f"replicas{ws}",
                   "l2": "inputs larger than L2: 11.3 GB of FP8 expert weights streamed per step, two "
                         "alternating 117 MB token batches"},
        "fp8_gemm_pct_of_peak": gemm_pct,
        "stages_ms": stage_ms,
        "roofline": {"bound": "tensor", "kernel": "grouped_gemm_kernel<fp8, swiglu> (GEMM 1)",
                     "achieved": gemm1_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": gemm1_tflops / fp8_peak, "traffic": traffic,
                     "peak_source": f"{src} bf16 sustained x {FP8_OVER_BF16} (nominal FP8/BF16 ratio)",
                     "flop_per_launch": g1},
        "e2e": {"value": sh.T * e_steps * ws / (e2e_ms / 1000.0), "unit": "tokens/s",
                "h2d_bytes_per_step": sh.T * sh.d * 2, "d2h_bytes_per_step": sh.T * sh.d * 2},
        "clocks": clocks.summary(),
        "gpu_launches": KERNELS_PER_STEP * args.steps,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        inputs = (u_bufs[0].cpu(), cent.cpu(), bias.cpu(),
                  lambda e: tuple(w.cpu() for w in S.expert_weights(sh, e, device=dev)))
        n = max(1, int(os.environ.get("CPU_BASELINE_TOKENS", "4")))
        v, dt, cores = oracle_sample_timing(sh, inputs, n, seed=99)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{n} tokens of the same workload ({dt:.1f} s): routing, FP8 "
                                          f"quantisation of the tokens and of their experts' weights, FFNs, combine"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
