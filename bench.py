#!/usr/bin/env python3
"""Benchmark: DeepSeekMoE layer forward at the V3 shape on B300.

One step = the whole hot path on one batch: routing (sigmoid affinities,
biased top-8, gates, loads), permutation with 1x128 FP8 quantisation, grouped
GEMM 1 (W1/W3) with the SwiGLU + FP8 epilogue, grouped GEMM 2 (W2), combine
h' = u + shared + sum g*FFN, and the bias update — 256 routed experts + 1
shared, d=7168, I=2048, T=8192 tokens, Zipf(1.1)-skewed expert popularity,
FP8 E4M3 expert weights resident in HBM with 128x128 scales.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Besides the V3 layer (the headline metric), the
line carries under "configs" the other workloads of the benchmark, each timed
alone with L2 flushed before every launch and each with its own roofline and a
bounded CPU-oracle baseline: the tiny bf16 layer, route + dispatch at
T=16384, the dense FP8 block-scaled GEMM 4096x4096x7168, the two
group-limited decode batches (T=64, T=256) on the V3 layer's weights, and one
training step of the V3 layer (training forward, FP8 backward, SGD on fp32
masters with the FP8 weights quantised again).
Multi-GPU (torchrun): replicas, one per GPU, no collective on the data path
(weak scaling; value = all ranks' tokens / the slowest rank's time).
`--impl reference` times the FP64 CPU oracle on a bounded sample of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import itertools
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
KERNELS_PER_STEP = 10        # gate GEMM, select | count, scan, rank, scatter | GEMM1 | GEMM2 | combine | bias
ORACLE_TOKENS = 4            # V3-layer tokens per oracle sample (reference arm step and cpu_baseline)


def profiled_traffic(name):
    """DRAM bytes per launch of a kernel from its committed ncu summary
    (profiles/traffic.md, lines `name: bytes sha1`), or None when the kernel
    source changed since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    h = hashlib.sha1()
    for f in ("gemm.cu", "common.cuh"):   # the code only: // comments and blank lines do not count
        with open(os.path.join(ROOT, "mixture_experts_layer_90_b300", "csrc", f), encoding="utf-8") as fh:
            for ln in fh:
                code = ln.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    for ln in open(p):
        parts = ln.strip().strip("`").split()
        if len(parts) == 3 and parts[0] == name + ":" and parts[2] == h.hexdigest()[:12]:
            return float(parts[1])
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK, "fallback"


class NvmlPoller:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml, by ctypes; read-only queries) every ~2 ms in a thread, so
    that a timed region of a tenth of a second still gets dozens of samples.
    Inactive when the library cannot be loaded."""

    # nvmlClocksEventReason* bits
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
               ("sw_power_cap", 0x4))
    CLOCK_SM = 1

    def __init__(self, gpu_index: int):
        self.samples = []          # (sm_mhz, reason bits)
        self.on = False
        self.lib = None
        try:
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self._index(lib, gpu_index)),
                                                 ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(mx)) != 0:
                return
            self.max_mhz = float(mx.value)
            self.get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ctypes = ctypes
            self.lib = lib
        except (OSError, AttributeError):
            self.lib = None

    @staticmethod
    def _index(lib, gpu_index):
        # the NVML device with the CUDA device's UUID, else the same index
        try:
            import ctypes
            import torch
            want = str(torch.cuda.get_device_properties(gpu_index).uuid)
            n = ctypes.c_uint()
            lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
            for i in range(n.value):
                h = ctypes.c_void_p()
                buf = ctypes.create_string_buffer(96)
                if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(i), ctypes.byref(h)) == 0 and \
                        lib.nvmlDeviceGetUUID(h, buf, ctypes.c_uint(96)) == 0 and want and want in buf.value.decode():
                    return i
        except Exception:
            pass
        return gpu_index

    def start(self):
        if self.lib is None:
            return
        self.on = True
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def stop(self):
        if self.on:
            self.on = False
            self._t.join(timeout=2.0)

    def _run(self):
        ct = self.ctypes
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while self.on:
            if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(clk)) != 0 or \
                    self.get_reasons(self.h, ct.byref(rs)) != 0:
                return
            self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.002)

    def summary(self):
        if not self.samples:
            return None
        sm = [c for c, _ in self.samples]
        reasons = sorted(name for name, bit in self.REASONS if any(r & bit for _, r in self.samples))
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sm), "source": "NVML, every ~2 ms"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms, plus NVML
    polled every ~2 ms (NvmlPoller); summary() covers the samples taken between
    mark_start() and mark_stop() (the timed region), or all samples if no mark
    was set. The NVML samples are the record when there are any; the
    nvidia-smi summary is kept beside them."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.start, self.stop = 0, None
        self.nvml = NvmlPoller(gpu_index)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 10.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def mark_start(self):
        self.start = len(self.lines)
        self.nvml.start()

    def mark_stop(self):
        self.nvml.stop()
        time.sleep(0.05)          # let the sampler report the region's last interval
        self.stop = len(self.lines)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.nvml.stop()
        if self.stop is None:
            self.stop = len(self.lines)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.start:self.stop]:
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
        smi = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
               "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, every 20 ms"}
        fine = self.nvml.summary()
        if fine is None:
            return smi
        # a reason either source saw during the region counts
        fine["reasons"] = sorted(set(fine["reasons"]) | set(smi["reasons"]))
        fine["nvidia_smi"] = smi
        return fine


def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks (the slowest rank's time); x itself when
    torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


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
    per_step = max(1, int(os.environ.get("REF_TOKENS_PER_STEP", str(ORACLE_TOKENS))))
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

def fp8_peak_tflops(pk, region_s):
    """FP8 dense peak to divide by: 2 x the measured bf16 cuBLAS figure (the
    nominal FP8 / BF16 ratio), burst for a timed region under 2 s, sustained
    for a longer one."""
    if region_s < 2.0:
        return pk["bf16_tflops"] * FP8_OVER_BF16, "bf16 burst"
    return pk["bf16_tflops_sustained"] * FP8_OVER_BF16, "bf16 sustained"


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
        clocks.mark_start()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(args.steps):
            layer.forward(u_bufs[i % 2], out, stage_events=events[i])
        t1.record()
        barrier()
        clocks.mark_stop()
    status = moe.device_status()
    assert status == 0, f"device status {status}"
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), dev)
    stage_ms = {name: statistics.mean(ev[j].elapsed_time(ev[j + 1]) for ev in events)
                for j, name in enumerate(moe.LAYER_STAGES)}

    # ---- end to end through the pipelined host-buffer C call: every step copies its
    # batch in from pinned host memory and h' back out; consecutive steps overlap ----
    u_host = [b.cpu().pin_memory() for b in u_bufs]
    out_host = [torch.empty_like(u_host[0]).pin_memory() for _ in range(2)]
    e_steps = max(1, min(args.steps, 50))
    warm = [torch.cuda.Event() for _ in range(2)]
    for i in range(2):
        layer.forward_host_pipelined(u_host[i % 2], out_host[i % 2], slot=i % 2, done=warm[i])
    warm[1].synchronize()
    barrier()
    done = [torch.cuda.Event() for _ in range(e_steps)]
    w0 = time.perf_counter()           # host wall clock: the copies run on the library's own streams
    for i in range(e_steps):
        if i >= 2:
            done[i - 2].synchronize()  # step i-2's h' is in out_host[i % 2]: a user would read it here
        layer.forward_host_pipelined(u_host[i % 2], out_host[i % 2], slot=i % 2, done=done[i])
    done[e_steps - 1].synchronize()
    barrier()
    e2e_ms = max_over_ranks(1000.0 * (time.perf_counter() - w0), dev)
    assert moe.device_status() == 0

    tokens = sh.T * args.steps * ws
    value = tokens / (elapsed_ms / 1000.0)
    g1, g2 = layer_flops(sh)
    pk, src = peaks()
    fp8_peak, peak_kind = fp8_peak_tflops(pk, elapsed_ms / 1000.0)
    t1s = stage_ms["gemm1_swiglu"] / 1000.0
    t2s = stage_ms["gemm2"] / 1000.0
    gemm1_tflops = g1 / t1s / 1e12
    gemm_pct = 100.0 * (g1 + g2) / (t1s + t2s) / 1e12 / fp8_peak
    traffic = profiled_traffic("gemm1_swiglu")

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "v3-layer-fp8", "T": sh.T, "d": sh.d, "N": sh.N, "shared": 1, "K": sh.K,
                   "I": sh.I, "popularity": "zipf(1.1)", "global_batch": sh.T * ws, "parallelism": f"replicas{ws}",
                   "l2": "inputs larger than L2: 11.3 GB of FP8 expert weights streamed per step, two "
                         "alternating 117 MB token batches"},
        "fp8_gemm_pct_of_peak": gemm_pct,
        "gemm2_frac_of_fp8_peak": g2 / t2s / 1e12 / fp8_peak,
        "stages_ms": stage_ms,
        "roofline": {"bound": "tensor", "kernel": "grouped_gemm_kernel<fp8, swiglu> (GEMM 1)",
                     "achieved": gemm1_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": gemm1_tflops / fp8_peak, "traffic": traffic,
                     "peak_source": f"{src} {peak_kind} x {FP8_OVER_BF16} (nominal FP8/BF16 ratio); timed region "
                                    f"{elapsed_ms / 1000.0:.2f} s",
                     "flop_per_launch": g1},
        "e2e": {"value": sh.T * e_steps * ws / (e2e_ms / 1000.0), "unit": "tokens/s",
                "h2d_bytes_per_step": sh.T * sh.d * 2, "d2h_bytes_per_step": sh.T * sh.d * 2},
        "clocks": clocks.summary(),
        "gpu_launches": KERNELS_PER_STEP * args.steps,
    }
    cpu_rows = []
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        inputs = (u_bufs[0].cpu(), cent.cpu(), bias.cpu(),
                  lambda e: tuple(w.cpu() for w in S.expert_weights(sh, e, device=dev)))
        n = max(1, int(os.environ.get("CPU_BASELINE_TOKENS", str(ORACLE_TOKENS))))
        v, dt, cores = oracle_sample_timing(sh, inputs, n, seed=99)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{n} tokens of the same workload ({dt:.1f} s): routing, FP8 "
                                          f"quantisation of the tokens and of their experts' weights, FFNs, combine"}
    if rank == 0 and not args.no_configs:
        # the benchmark's other workloads, each alone, L2 flushed before every launch
        flush = L2Flush(dev)
        cb = ws == 1 and not args.no_cpu_baseline
        line["configs"] = {
            "tiny_bf16_layer": case_tiny(moe, S, dev, args, flush, cpu_baseline=cb),
            "route_dispatch_t16384": case_route(moe, S, dev, args, flush, cpu_baseline=cb),
            "fp8_gemm_4096x4096x7168": case_gemm(moe, S, dev, args, flush, cpu_baseline=cb),
        }
        for dsh in S.DECODE_V3:
            line["configs"][f"decode_t{dsh.T}"] = case_decode(moe, S, dev, args, flush, layer, dsh,
                                                              cpu_baseline=cb)
        line["configs"]["train_step_v3_t8192"] = case_train(moe, S, dev, args, flush, cpu_baseline=cb)
        assert moe.device_status() == 0
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# --------------------------------------------------------------------------
# single workloads: the benchmark's other configurations (each timed alone)
# --------------------------------------------------------------------------

class L2Flush:
    """Writes a buffer twice the size of L2 so the next launch starts cold."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.buf = torch.empty(max(2 * l2, 1 << 20) // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.buf.fill_(1)


def time_launches(fn, steps, warmup, flush=None):
    """Mean device time (ms) of fn() over `steps` launches, each bracketed by
    CUDA events on the current stream, with an optional L2 flush before each."""
    import torch
    for _ in range(warmup):
        if flush:
            flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        if flush:
            flush()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def _cpu(value, unit, cores, sample):
    return {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}


def case_tiny(moe, S, dev, args, flush, cpu_baseline=True):
    """The tiny bf16 layer (T=128, d=256, 16 routed + 1 shared, top-4, I=128,
    b=0): launch-latency bound; reported as microseconds per layer call."""
    import numpy as np
    import torch

    import oracle
    sh = S.TINY
    cent = S.centroids(sh).to(dev)
    bias = S.bias(sh, zero=True).to(dev)
    layer = moe.MoELayer.build(sh.d, sh.N, sh.K, sh.I, cent, bias, lambda e: S.expert_weights(sh, e, device=dev),
                               fp8=False, gamma=sh.gamma)
    u = S.tokens(sh, device=dev)
    out = torch.empty_like(u)
    ms_eager = time_launches(lambda: layer.forward(u, out, update_bias=False), args.steps, args.warmup, flush)
    # the same call captured once in a CUDA graph and replayed (the launch-bound case graphs are for)
    graph = layer.capture(u, out, update_bias=False)
    ms = time_launches(graph.replay, args.steps, args.warmup, flush)
    R = sh.T * sh.K + sh.T
    flop = 2.0 * R * 3 * sh.I * sh.d + 2.0 * sh.T * sh.N * sh.d
    pk, src = peaks()
    res = {"workload": "tiny-bf16-layer T=128 d=256 16+1 experts top-4 I=128", "ms": ms, "us_per_layer": 1e3 * ms,
           "us_per_layer_eager": 1e3 * ms_eager, "tokens_per_s": sh.T / ms * 1e3, "dtype": "bf16",
           # gate GEMM, select | one-block count/scan/rank (it also writes the loads), scatter | GEMM1 | GEMM2 |
           # combine
           "launches": 7, "timing": "CUDA-graph replay of the layer call (eager call beside it)",
           "roofline": {"bound": "tensor", "achieved": flop / ms / 1e9, "peak": pk["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": flop / ms / 1e9 / pk["bf16_tflops"], "traffic": None,
                        "note": "launch-latency bound: 7 dependent kernels of a few microseconds each",
                        "peak_source": f"{src} bf16 burst"}}
    if cpu_baseline:
        w = {e: S.expert_weights(sh, e) for e in range(sh.N + 1)}
        t0 = time.perf_counter()
        oracle.layer_tokens(u.cpu(), cent.cpu(), bias.cpu(), sh.K, lambda e: w[e], np.arange(sh.T), fp8=False)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = _cpu(sh.T / dt, "tokens/s", oracle.threads(), f"the whole layer, all {sh.T} tokens "
                                   f"({dt:.2f} s)")
    del layer
    return res


def case_route(moe, S, dev, args, flush, cpu_baseline=True):
    """Routing + dispatch at T=16384, d=7168, 256 fp32 centroids, top-8: gate
    logits, affinities, biased top-8, gates, loads (routing from centroids
    prepared once), the stable counting sort and scatter of bf16 rows, and the
    bias update. The gate is a contraction, the rest moves bytes."""
    import numpy as np

    import oracle
    sh = S.ROUTE_V3
    T, d, N, K = sh.T, sh.d, sh.N, sh.K
    u = S.tokens(sh, device=dev)
    cent = S.centroids(sh, device=dev)
    bias = S.bias(sh, device=dev)
    L = moe.load_library()
    prepared = moe.moe_route_prepare_centroids(cent)
    ws_r = moe._ws(L.moe_route_prepared_workspace_size(T, d, N, moe.MOE_DTYPE_F32), dev)
    ws_p = moe._ws(L.moe_permute_workspace_size(T, N), dev)
    pk, src = peaks()
    idx, gates, loads, _ = moe.moe_route_prepared(u, prepared, moe.MOE_DTYPE_F32, N, bias, K, workspace=ws_r)
    moe.moe_permute(u, idx, N, workspace=ws_p)

    def step():
        moe.moe_route_prepared(u, prepared, moe.MOE_DTYPE_F32, N, bias, K, workspace=ws_r)
        moe.moe_permute(u, idx, N, workspace=ws_p)
        moe.moe_bias_update(bias, loads, T, K, sh.gamma)
    ms = time_launches(step, args.steps, args.warmup, flush)
    ms_route = time_launches(lambda: moe.moe_route_prepared(u, prepared, moe.MOE_DTYPE_F32, N, bias, K,
                                                            workspace=ws_r), args.steps, args.warmup, flush)
    ms_perm = time_launches(lambda: moe.moe_permute(u, idx, N, workspace=ws_p), args.steps, args.warmup, flush)
    # sequence-wise balance statistics of the step (sequences of 4096 tokens) from the routing's affinities
    seq_len = 4096
    _, _, _, scores = moe.moe_route_prepared(u, prepared, moe.MOE_DTYPE_F32, N, bias, K, want_scores=True,
                                             workspace=ws_r)
    ws_b = moe._ws(L.moe_route_balance_stats_workspace_size(T, N, seq_len), dev)
    ms_bal = time_launches(lambda: moe.moe_route_balance_stats(scores, idx, seq_len, workspace=ws_b), args.steps,
                           args.warmup, flush)
    bal_bytes = T * N * 4 + T * K * 4 + (T // seq_len) * N * 8
    # algorithmic bytes: u read twice (gate, scatter), the prepared centroids, the K bf16 copies
    # written, indices / gates / rows / tokens (int32 or fp32) written, bias and loads
    alg = 2 * T * d * 2 + N * 3 * d * 2 + T * K * d * 2 + T * K * 4 * 4 + N * 12
    res = {"workload": "route-dispatch-16384x7168-256e-top8", "ms": ms, "tokens_per_s": T / ms * 1e3,
           "ms_route": ms_route, "ms_permute": ms_perm,
           "permute_gbs": (T * d * 2 + T * K * d * 2 + T * K * 12) / ms_perm / 1e6,
           "balance_stats": {"seq_len": seq_len, "ms": ms_bal, "gbs": bal_bytes / ms_bal / 1e6,
                             "frac_of_hbm": bal_bytes / ms_bal / 1e6 / pk["hbm_gbs"],
                             "note": "reads the [T, N] fp32 affinities once; two launches"},
           "roofline": {"bound": "hbm", "achieved": alg / ms / 1e6, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": alg / ms / 1e6 / pk["hbm_gbs"], "traffic": None, "algorithmic_bytes": alg,
                        "peak_source": f"{src} hbm copy"},
           "l2": "flushed before each step"}
    # the gate is a contraction (three bf16 terms of the fp32 centroids), the rest moves bytes:
    # the workload's floor is the gate at the bf16 peak plus the bytes at the HBM peak, in sequence
    gate_flop = 2.0 * T * ((N + 255) // 256 * 256) * 3 * d
    floor_ms = gate_flop / pk["bf16_tflops"] / 1e9 + alg / pk["hbm_gbs"] / 1e6
    res["roofline_combined"] = {"bound": "tensor (gate) + hbm (the rest), in sequence", "floor_ms": floor_ms,
                                "frac": floor_ms / ms, "gate_flop": gate_flop,
                                "peak_source": f"{src} bf16 burst and hbm copy"}
    if cpu_baseline:
        n = 512
        uc, ec, bc = u[:n].cpu(), cent.cpu(), bias.cpu()
        t0 = time.perf_counter()
        r = oracle.route(uc, ec, bc, K)
        oracle.permute(r.topk_idx, N)
        oracle.bias_update(bc.numpy(), r.loads, n, K, sh.gamma)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = _cpu(n / dt, "tokens/s", oracle.threads(),
                                   f"routing, permutation indices and bias update of {n} of the {T} tokens "
                                   f"({dt:.2f} s)")
    return res


def case_gemm(moe, S, dev, args, flush, cpu_baseline=True):
    """The dense FP8 block-scaled GEMM: A 4096x7168 (1x128 scales, 0.1% outliers
    x100), B 4096x7168 (128x128 scales), bf16 out; tensor bound."""
    import torch

    import oracle
    cfg = S.GEMM_V3
    a, b = S.gemm_operands(cfg["M"], cfg["K"], cfg["N"], device=dev)
    qa, sa = moe.fp8_quant_1x128(a)
    qb, sb = moe.fp8_quant_128x128(b)
    qb3, sb3 = qb[None], sb[None]
    offs = torch.tensor([0, cfg["M"]], dtype=torch.int32, device=dev)
    C = moe.fp8_grouped_gemm(qa, sa, qb3, sb3, offs, moe.MOE_EPI_BF16)
    ms = time_launches(lambda: moe.fp8_grouped_gemm(qa, sa, qb3, sb3, offs, moe.MOE_EPI_BF16, C=C),
                       args.steps, args.warmup, flush)
    flop = 2.0 * cfg["M"] * cfg["N"] * cfg["K"]
    pk, src = peaks()
    peak = pk["bf16_tflops"] * FP8_OVER_BF16
    res = {"workload": "fp8-gemm-4096x4096x7168", "ms": ms, "tflops": flop / ms / 1e9,
           "roofline": {"bound": "tensor", "achieved": flop / ms / 1e9, "peak": peak, "unit": "TFLOP/s",
                        "frac": flop / ms / 1e9 / peak, "traffic": None,
                        "peak_source": f"{src} bf16 burst x {FP8_OVER_BF16}"},
           "l2": "flushed before each launch"}
    if cpu_baseline:
        rows = 16
        qa_o, sa_o = oracle.quant_1x128(a[:rows].cpu())
        qb_o, sb_o = oracle.quant_128x128(b.cpu())
        t0 = time.perf_counter()
        oracle.fp8_gemm(qa_o, sa_o, qb_o, sb_o)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = _cpu(2.0 * rows * cfg["N"] * cfg["K"] / dt / 1e12, "TFLOP/s", oracle.threads(),
                                   f"{rows} of the {cfg['M']} output rows from operands the oracle quantised "
                                   f"itself ({dt:.2f} s)")
    return res


def case_decode(moe, S, dev, args, flush, v3_layer, dsh, cpu_baseline=True):
    """A group-limited decode batch (T=64 or 256; 8 groups of 32 experts, top-4
    groups, top-8 within) through the V3 layer's resident FP8 weights; bound by
    streaming the active experts' weights from HBM."""
    import torch

    import oracle
    # the seeded bias, not the V3 layer's after its bench steps: the batch routes the same in every run
    layer = moe.MoELayer(dsh.d, dsh.N, dsh.K, dsh.I, v3_layer.centroids, S.bias(dsh, device=dev), v3_layer.w13,
                         v3_layer.w2, v3_layer.w13_scales, v3_layer.w2_scales, n_groups=dsh.n_groups,
                         topk_groups=dsh.topk_groups, gamma=dsh.gamma)
    u = S.tokens(dsh, seed=3, device=dev)
    out = torch.empty_like(u)
    ms_eager = time_launches(lambda: layer.forward(u, out, update_bias=False), args.steps, args.warmup, flush)
    graph = layer.capture(u, out, update_bias=False)   # a decode step replayed, not relaunched
    ms_graph = time_launches(graph.replay, args.steps, args.warmup, flush)
    # both ways of running a decode step are timed; the faster one is the entry's time
    ms = min(ms_graph, ms_eager)
    how = "CUDA-graph replay" if ms_graph <= ms_eager else "eager call"
    active = int((layer.loads > 0).sum().item()) + 1
    per_expert = 3 * dsh.I * dsh.d + 4 * (3 * dsh.I * dsh.d // 16384)
    alg = active * per_expert + 2 * dsh.T * dsh.d * 2
    pk, src = peaks()
    res = {"workload": dsh.name, "ms": ms, "ms_graph": ms_graph, "ms_eager": ms_eager, "tokens_per_s": dsh.T / ms * 1e3,
           "active_experts": active,
           "timing": f"the faster of a CUDA-graph replay and an eager call of the layer: {how}",
           "roofline": {"bound": "hbm", "achieved": alg / ms / 1e6, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": alg / ms / 1e6 / pk["hbm_gbs"], "traffic": None, "algorithmic_bytes": alg,
                        "peak_source": f"{src} hbm copy"},
           "l2": "flushed before each step"}
    if cpu_baseline:
        import numpy as np
        n = 2
        inputs = (u.cpu(), v3_layer.centroids.cpu(), layer.bias.cpu(),
                  lambda e: tuple(w.cpu() for w in S.expert_weights(dsh, e, device=dev)))
        toks = np.arange(n)
        r = oracle.route(inputs[0][torch.as_tensor(toks)], inputs[1], inputs[2], dsh.K, dsh.n_groups,
                         dsh.topk_groups)
        cache = {e: inputs[3](e) for e in sorted(set(r.topk_idx.ravel().tolist()) | {dsh.N})}
        t0 = time.perf_counter()
        oracle.layer_tokens(inputs[0], inputs[1], inputs[2], dsh.K, lambda e: cache[e], toks, fp8=True,
                            n_groups=dsh.n_groups, topk_groups=dsh.topk_groups)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = _cpu(n / dt, "tokens/s", oracle.threads(),
                                   f"{n} tokens: group-limited routing, FP8 quantisation of the tokens and of "
                                   f"their experts' weights, FFNs, combine ({dt:.1f} s)")
    del layer
    return res


def case_train(moe, S, dev, args, flush, cpu_baseline=True):
    """One training step of the V3 layer (T=8192, d=7168, 256 routed + 1
    shared experts, top-8, I=2048): the training forward (keeps the affinities
    and GEMM 1's products), the backward (FP8 products for dA, dX and both
    weight gradients on the tensor cores; combine, SwiGLU and gate backward),
    and SGD on the fp32 masters with the FP8 weights quantised again."""
    import numpy as np
    import torch

    import oracle
    sh = S.LAYER_V3
    T, d, N, K, I = sh.T, sh.d, sh.N, sh.K, sh.I
    G_ = N + 1
    R = T * K + T
    pk, src = peaks()
    cent = S.centroids(sh, zipf=True).to(dev)
    bias = S.bias(sh).to(dev)
    layer = moe.MoELayer.build(d, N, K, I, cent, bias, lambda e: S.expert_weights(sh, e, device=dev), fp8=True,
                               train=True, gamma=sh.gamma)
    u = S.tokens(sh, seed=5, device=dev)
    G = S.grad_out(sh, seed=5, device=dev)
    out, du = torch.empty_like(u), torch.empty_like(u)
    ms_fwd = time_launches(lambda: layer.forward_train(u, out, update_bias=False), args.steps, args.warmup, flush)
    # the backward, its stages timed by events on the launching stream
    names = ["combine_bwd", "gemm_dA", "swiglu_bwd", "gemm_dX", "gates_du_centroids", "wgrad_operands",
             "gemm_dW2", "gemm_dW13"]
    for _ in range(args.warmup):
        flush()
        layer.backward(u, G, du)
    torch.cuda.synchronize()
    runs = []
    for _ in range(args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        flush()
        layer.backward(u, G, du, stage_events=ev)
        runs.append(ev)
    torch.cuda.synchronize()
    stage = {n: statistics.mean(r[i].elapsed_time(r[i + 1]) for r in runs) for i, n in enumerate(names)}
    ms_bwd = statistics.mean(r[0].elapsed_time(r[-1]) for r in runs)
    assert moe.device_status() == 0
    # the SGD step on both masters with their re-quantisation (two launches), alone
    def sgd():
        moe.moe_sgd_requant_128x128(layer.w13_master, layer.dw13, 1e-7, layer.w13, layer.w13_scales, layer.w13t,
                                    layer.w13t_scales)
        moe.moe_sgd_requant_128x128(layer.w2_master, layer.dw2, 1e-7, layer.w2, layer.w2_scales, layer.w2t,
                                    layer.w2t_scales)
    ms_sgd = time_launches(sgd, args.steps, args.warmup, flush)
    ms_step = time_launches(lambda: layer.train_step(u, G, 1e-7, out, du), args.steps, args.warmup, flush)
    assert moe.device_status() == 0
    # rooflines: the backward's two weight-gradient GEMMs write fp32 [G, M, Nd]
    # gradients; their operands are read once from HBM (re-reads hit L2)
    Kp = ((R + 127) // 128 + G_) * 128
    n_w = G_ * 3 * I * d                                     # parameters of the experts
    rl = {
        "gemm_dA": ("tensor", 2.0 * R * d * I),
        "gemm_dX": ("tensor", 2.0 * R * d * 2 * I),
        "gemm_dW2": ("hbm", G_ * d * I * 4 + (d + I) * Kp + (d + I) * Kp // 32),
        "gemm_dW13": ("hbm", G_ * 2 * I * d * 4 + (2 * I + d) * Kp + (2 * I + d) * Kp // 32),
        "combine_bwd": ("hbm", T * d * 2 + T * K * d * 2 + R * d + R * d // 32),
        "swiglu_bwd": ("hbm", R * I * 2 + R * 2 * I * 2 * 2 + R * 2 * I + R * 2 * I // 32),
        "gates_du_centroids": ("hbm", T * d * 2 * 2 + R * d * 2 + T * K * d * 2),
        "wgrad_operands": ("hbm", R * (d + 2 * I + 2 * I + d) * 2 + Kp * (2 * d + 3 * I) * 1),
    }
    fp8_peak, fp8_src = fp8_peak_tflops(pk, ms_bwd * args.steps / 1e3)
    roof = {}
    for n, (bound, amount) in rl.items():
        if bound == "tensor":
            a = amount / (stage[n] * 1e-3) / 1e12
            roof[n] = {"bound": "tensor", "achieved": a, "peak": fp8_peak, "unit": "TFLOP/s", "frac": a / fp8_peak}
        else:
            a = amount / (stage[n] * 1e-3) / 1e9
            roof[n] = {"bound": "hbm", "achieved": a, "peak": pk["hbm_gbs"], "unit": "GB/s",
                       "frac": a / pk["hbm_gbs"]}
    sgd_bytes = n_w * (4 + 4 + 4 + 1 + 1) + n_w // 16384 * 8
    sgd_gbs = sgd_bytes / (ms_sgd * 1e-3) / 1e9
    top = max(stage, key=stage.get)
    res = {"workload": "train-step-v3-8192x7168-256e-top8-I2048", "ms": ms_step, "tokens_per_s": T / ms_step * 1e3,
           "ms_forward_train": ms_fwd, "ms_backward": ms_bwd, "ms_sgd_requant": ms_sgd,
           "backward_stages_ms": stage, "backward_rooflines": roof,
           "sgd_requant": {"bound": "hbm", "achieved": sgd_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                           "frac": sgd_gbs / pk["hbm_gbs"], "bytes": sgd_bytes,
                           "note": "reads the fp32 master and gradient, writes the master, the E4M3 codes "
                                   "and their transposed copy"},
           # the step's dominant kernel by time: the SGD re-quantisation (two launches) or a backward stage
           "roofline": (dict(bound="hbm", achieved=sgd_gbs, peak=pk["hbm_gbs"], unit="GB/s",
                             frac=sgd_gbs / pk["hbm_gbs"], kernel="sgd_requant_kernel (W13 and W2 masters)",
                             traffic=None, peak_source=f"{src} hbm copy")
                        if ms_sgd >= stage[top] else
                        dict(roof[top], kernel=f"backward stage {top}", traffic=None,
                             peak_source=f"{src} ({fp8_src})" if roof[top]["bound"] == "tensor"
                             else f"{src} hbm copy")),
           "lr": 1e-7, "l2": "flushed before each step",
           "note": "step = training forward + backward + SGD with re-quantisation of every expert weight; "
                   "at this batch the SGD over 11.3 G parameters (fp32 master and gradient) dominates"}
    if cpu_baseline:
        n = 2
        toks = torch.arange(n)
        uh, Gh = u[:n].cpu(), G[:n].cpu()
        r = oracle.route(uh, cent.cpu(), bias.cpu(), K, want_scores=True)
        cache = {e: tuple(w.cpu() for w in S.expert_weights(sh, e, device=dev))
                 for e in sorted(set(r.topk_idx.ravel().tolist()) | {N})}
        t0 = time.perf_counter()
        oracle.layer_backward(uh, cent.cpu(), bias.cpu().numpy(), K, lambda e: cache[e], Gh, fp8=True, route_all=r,
                              stack=False)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = _cpu(n / dt, "tokens/s", oracle.threads(),
                                   f"{n} tokens: the FP8 forward and backward through their {len(cache)} experts "
                                   f"(weight quantisation, products, weight gradients over 128 padded rows), "
                                   f"without the SGD ({dt:.1f} s)")
    del layer
    torch.cuda.empty_cache()
    return res


def case_dispatch(moe, S, dev, args, flush, which):
    """The V3 layer's dispatch (permute with 1x128 E4M3 quantisation and the shared
    expert's rows, `permute-fp8`) or combine (`combine`) alone, T = 8192, d = 7168,
    256 experts, top-8, on seeded ids. HBM bound."""
    import torch

    sh = S.LAYER_V3
    T, d, N, K = sh.T, sh.d, sh.N, sh.K
    pk, src = peaks()
    h = S.bits(S.key(0, "case-topk", T, N, K), 0, T * N).view(T, N)
    idx = torch.sort(torch.argsort(h, dim=1)[:, :K], dim=1).values.to(torch.int32).to(dev)
    u = S.tokens(sh, device=dev)
    L = moe.load_library()
    ws_p = moe._ws(L.moe_permute_workspace_size(T, N), dev)
    off, perm, dest, xp, xs = moe.moe_permute(u, idx, N, moe.MOE_DTYPE_E4M3, with_shared=True, workspace=ws_p)
    R = T * K + T
    if which == "permute-fp8":
        fn = lambda: moe.moe_permute(u, idx, N, moe.MOE_DTYPE_E4M3, with_shared=True, workspace=ws_p)  # noqa: E731
        alg = T * d * 2 + R * (d + d // 128 * 4) + T * K * 4 * 3 + N * 8
        workload = "permute-fp8-8192x7168-256e-top8+shared"
    else:
        y = S.normal((R, d), 0.5, S.key(0, "case-y", R, d), device=dev)
        g = torch.full((T, K), 1.0 / K, device=dev)
        out = torch.empty_like(u)
        fn = lambda: moe.moe_combine(u, y[T * K:], y, g, dest, out=out)  # noqa: E731
        alg = (K + 2) * T * d * 2 + T * d * 2 + T * K * 8
        workload = "combine-8192x7168-top8+shared"
    ms = time_launches(fn, args.steps, args.warmup, flush)
    return {"workload": workload, "ms": ms, "tokens_per_s": T / ms * 1e3,
            "roofline": {"bound": "hbm", "achieved": alg / ms / 1e6, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": alg / ms / 1e6 / pk["hbm_gbs"], "traffic": None, "algorithmic_bytes": alg,
                         "peak_source": f"{src} hbm copy"},
            "l2": "flushed before each launch"}


def grouped_fp8_operands(moe, S, dev, rows_per_group, G, Nd, Kd, seed=0):
    """Row-grouped E4M3 activations [G*rows, Kd] and G weight matrices [Nd, Kd],
    drawn N(0,1) and N(0, 1/sqrt(Kd)) and quantised by this library's kernels."""
    import torch
    M = rows_per_group * G
    a = S.normal((M, Kd), 1.0, S.key(seed, "case-a", M, Kd), device=dev)
    qa, sa = moe.fp8_quant_1x128(a)
    del a
    qb = torch.empty((G, Nd, Kd), dtype=torch.uint8, device=dev)
    sb = torch.empty((G, Nd // 128, Kd // 128), dtype=torch.float32, device=dev)
    for g in range(G):
        w = S.normal((Nd, Kd), 1.0 / math.sqrt(Kd), S.key(seed, "case-b", g, Nd, Kd), device=dev)
        moe.fp8_quant_128x128(w, qb[g], sb[g])
    offs = torch.arange(0, M + 1, rows_per_group, dtype=torch.int32, device=dev)
    return qa, sa, qb, sb, offs


def case_gemm_slice(moe, S, dev, args, flush, which):
    """One expert's average share of the V3 layer's GEMMs: 33 groups (32 routed +
    shared) of 256 rows; GEMM 1 (SwiGLU + FP8 out) or GEMM 2 (bf16 out). A small
    case for profiling the grouped GEMM."""
    G, rows = 33, 256
    Nd, Kd, epi = (4096, 7168, moe.MOE_EPI_SWIGLU_FP8) if which == 1 else (7168, 2048, moe.MOE_EPI_BF16)
    qa, sa, qb, sb, offs = grouped_fp8_operands(moe, S, dev, rows, G, Nd, Kd)
    M = G * rows
    outs = moe.fp8_grouped_gemm(qa, sa, qb, sb, offs, epi)
    C, cs = outs if epi == moe.MOE_EPI_SWIGLU_FP8 else (outs, None)
    ms = time_launches(lambda: moe.fp8_grouped_gemm(qa, sa, qb, sb, offs, epi, C=C, c_scales=cs),
                       args.steps, args.warmup, flush)
    flop = 2.0 * M * Nd * Kd
    pk, src = peaks()
    peak = pk["bf16_tflops"] * FP8_OVER_BF16
    return {"workload": f"grouped-fp8-{G}x{rows}x{Nd}x{Kd}", "ms": ms, "tflops": flop / ms / 1e9,
            "frac_of_fp8_peak": flop / ms / 1e9 / peak, "peak_source": f"{src} bf16 burst x {FP8_OVER_BF16}",
            "l2": "flushed before each launch"}


def case_wgrad_slice(moe, S, dev, args, flush):
    """The backward's dW13 GEMM for 16 experts of the V3 shape (fp32 [16, 4096,
    7168] out, 2-3 blocks of 128 tokens per expert, seeded codes and scales):
    a small case for profiling the weight-gradient mode."""
    import torch
    G, M, Nd = 16, 4096, 7168
    blocks = [2 + (e * 7) % 2 for e in range(G)]
    kofs = torch.tensor([0] + list(itertools.accumulate(blocks)), dtype=torch.int32, device=dev)
    Kp = int(kofs[-1].item()) * 128
    key = S.key(0, "wgrad-slice", G, M, Nd)
    A = (S.bits(key, 0, M * Kp, dev) % 120).to(torch.uint8).view(M, Kp)
    B = (S.bits(key, M * Kp, Nd * Kp, dev) % 120).to(torch.uint8).view(Nd, Kp)
    sa = S.uniform((Kp // 128, M), 0.5, 1.5, S.key(1, "wgrad-slice-sa"), dev)
    sb = S.uniform((Kp // 128, Nd), 0.5, 1.5, S.key(1, "wgrad-slice-sb"), dev)
    C = torch.empty((G, M, Nd), dtype=torch.float32, device=dev)
    ms = time_launches(lambda: moe.fp8_grouped_gemm_wgrad(A, sa, B, sb, kofs, out=C), args.steps, args.warmup, flush)
    pk, src = peaks()
    out_gb = C.numel() * 4 / 1e9
    return {"workload": f"wgrad-fp8-{G}x{M}x{Nd}-k{Kp}", "ms": ms, "out_gbs": out_gb / ms * 1e3,
            "frac_of_hbm": out_gb / ms * 1e3 / pk["hbm_gbs"], "peak_source": f"{src} hbm copy",
            "l2": "flushed before each launch"}


def case_dispatch_modes(moe, S, dev, args):
    """The V3 layer step under both dispatch modes of an FP8 layer, alternating in
    one process on the same weights and batches: the permutation writing the
    grouped rows (scatter, the default) and GEMM 1 gathering the quantised
    tokens by perm_token (gather). Stages by CUDA events, ms per step."""
    import torch
    sh = S.LAYER_V3
    layer = moe.MoELayer.build(sh.d, sh.N, sh.K, sh.I, S.centroids(sh, zipf=True).to(dev), S.bias(sh).to(dev),
                               lambda e: S.expert_weights(sh, e, device=dev), fp8=True, gamma=sh.gamma)
    u_bufs = [S.tokens(sh, seed=s, device=dev) for s in (0, 7)]
    out = torch.empty_like(u_bufs[0])
    n_ev = len(moe.LAYER_STAGES) + 1
    runs = {"scatter": [], "gather": []}
    for _ in range(2):
        for name, mode in (("scatter", moe.MOE_DISPATCH_SCATTER), ("gather", moe.MOE_DISPATCH_GATHER)):
            layer._desc.dispatch = mode
            for i in range(args.warmup):
                layer.forward(u_bufs[i % 2], out, update_bias=False)
            torch.cuda.synchronize()
            events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
            for i in range(args.steps):
                layer.forward(u_bufs[i % 2], out, update_bias=False, stage_events=events[i])
            torch.cuda.synchronize()
            runs[name].append({n: statistics.mean(ev[j].elapsed_time(ev[j + 1]) for ev in events)
                               for j, n in enumerate(moe.LAYER_STAGES)})
    res = {"workload": "v3-layer-fp8 dispatch modes", "l2": "inputs larger than L2 (streamed weights)"}
    for name, rs in runs.items():
        stages = {n: statistics.mean(r[n] for r in rs) for n in moe.LAYER_STAGES}
        res[name] = {"ms_per_step": sum(stages.values()), "stages_ms": stages}
    return res


def run_case(args):
    import torch

    import mixture_experts_layer_90_b300 as moe
    import synthetic as S
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)
    line = {"case": args.case, "steps": args.steps, "warmup": args.warmup, "data": "synthetic"}
    cb = not args.no_cpu_baseline
    if args.case == "gemm":
        line.update(case_gemm(moe, S, dev, args, flush, cpu_baseline=cb))
    elif args.case in ("gemm1-small", "gemm2-small"):
        line.update(case_gemm_slice(moe, S, dev, args, flush, 1 if args.case == "gemm1-small" else 2))
    elif args.case == "route":
        line.update(case_route(moe, S, dev, args, flush, cpu_baseline=cb))
    elif args.case == "tiny":
        line.update(case_tiny(moe, S, dev, args, flush, cpu_baseline=cb))
    elif args.case in ("permute-fp8", "combine"):
        line.update(case_dispatch(moe, S, dev, args, flush, args.case))
    elif args.case == "train":
        line.update(case_train(moe, S, dev, args, flush, cpu_baseline=cb))
    elif args.case == "wgrad-small":
        line.update(case_wgrad_slice(moe, S, dev, args, flush))
    elif args.case == "dispatch":
        line.update(case_dispatch_modes(moe, S, dev, args))
    elif args.case in ("decode64", "decode256"):
        sh = S.LAYER_V3
        cent = S.centroids(sh, zipf=True).to(dev)
        bias = S.bias(sh).to(dev)
        v3 = moe.MoELayer.build(sh.d, sh.N, sh.K, sh.I, cent, bias, lambda e: S.expert_weights(sh, e, device=dev),
                                fp8=True, gamma=sh.gamma)
        dsh = S.DECODE_V3[0 if args.case == "decode64" else 1]
        line.update(case_decode(moe, S, dev, args, flush, v3, dsh, cpu_baseline=cb))
    assert moe.device_status() == 0
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="time the V3 layer only")
    ap.add_argument("--case", default="layer",
                    choices=["layer", "tiny", "route", "gemm", "gemm1-small", "gemm2-small", "decode64",
                             "decode256", "permute-fp8", "combine", "train", "wgrad-small", "dispatch"],
                    help="layer: the V3 layer step with every other workload (the benchmark line); the others "
                         "time one workload alone")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.case != "layer":
        run_case(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
