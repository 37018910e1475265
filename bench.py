"""Benchmark of the packed weight-only-quantized decode GEMV/GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl wqp|reference]

Headline workload: the ternary Q2_0 GEMV at the 27B-class qkv/o projection
shape, N = K = 5120, with M = 1, 4 and 8 activation rows. One step is three
calls (M = 1, 4, 8), each on a different weight buffer. The buffers are
cycled over more than 3x the L2 size, so HBM, not L2, supplies the weights.
The metric is effective weight-stream bandwidth: packed weight bytes (codes
plus scales, not A, C or the per-tensor scale) per second. The same line
reports per-call times for the other workloads (W4A16 at 5120^2, W8A16 for
the dense-FFN shapes with the scalar and tensor-core paths, and the Q2_0
decoder-layer sequence), the roofline of the dominant kernel, an end-to-end
number through the C ABI with host buffers, and the CPU oracle timed on the
host's cores.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas: the op has no exchange step), and value = all ranks' bytes / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective weight-stream GB/s (% of GB300 HBM peak) and us/call at M=1..16"
UNIT = "GB/s"
# The step calls, for each M, the library's fastest Q2_0 path at this shape
# (measured): the warp-level tensor-core GEMM (q2_gemm_mma) at M = 1, 4 and 8.
HEADLINE = {"fmt": "q2", "N": 5120, "K": 5120, "Ms": (1, 4, 8), "tc": {1: "mma", 4: "mma", 8: "mma"}}
WORKLOAD = "Q2_0 GEMV N=5120 K=5120, one step = M=1, 4, 8 calls"   # both arms' config
KERNEL_SOURCES = {False: ["gemv_scalar.cuh", "gemv_q2.cu", "decode.cuh", "common.cuh"],
                  True: ["gemm_tc.cu", "tc.cuh", "decode.cuh", "common.cuh"],
                  "mma": ["gemm_mma.cu", "tc.cuh", "common.cuh"],
                  "stream": ["gemm_mma_stream.cu", "tc.cuh", "common.cuh"],
                  "f16": ["gemm_mma_f16.cu", "mma_f16.cuh", "tc.cuh", "decode.cuh", "common.cuh"],
                  "w4s": ["gemm_mma_w4s.cu", "mma_f16.cuh", "tc.cuh", "decode.cuh", "common.cuh"]}
# Q2_0 entry point per path key (False: scalar, True: tcgen05, "mma": mma.sync).
Q2_PATH = {False: "q2_gemv", True: "q2_gemm_tc", "mma": "q2_gemm_mma"}


# ------------------------------------------------------------------ helpers
def weight_bytes(fmt, N, K):
    from weight_only_quantized_packed_gb300 import synth

    return {"q2": synth.q2_weight_bytes, "w4": synth.w4_weight_bytes,
            "w8": synth.w8_weight_bytes}[fmt](N, K)


def peak_bf16():
    """Measured dense bf16 tensor throughput (TFLOP/s, burst), else the
    fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2070.0)), "measured"
    except Exception:
        return 6800.0, 2070.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while timing."""

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
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
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
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _code_only(text):
    """Source text without comments and blank lines: a comment edit leaves
    the compiled kernel, and so its recorded DRAM traffic, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(l.strip() for l in text.splitlines() if l.strip())


def source_hash(tc=False):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[tc]:
        with open(os.path.join(ROOT, "weight_only_quantized_packed_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key, tc=False):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_hash") == source_hash(tc):
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


def reduce_max_ms(ms: float, dist=None, device="cuda") -> float:
    """Slowest rank's time (max over ranks); identity without a group."""
    if dist is None:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_step: int, steps: int, world: int, ms_total_max: float) -> float:
    """Whole-job GB/s: all ranks' weight bytes over the slowest rank's time."""
    return world * bytes_per_step * steps / (ms_total_max * 1e-3) / 1e9


# ------------------------------------------------------------------ GPU arm
class Workload:
    """Device-resident inputs for one format/shape, weights cycled over
    enough buffers to exceed 3x L2."""

    def __init__(self, fmt, N, K, Ms, l2_bytes, seed_workload, tc=False, cap_bytes=3 << 30):
        import torch

        from tests import _gpu as G
        from weight_only_quantized_packed_gb300 import synth

        self.fmt, self.N, self.K, self.Ms, self.tc = fmt, N, K, tuple(Ms), tc
        self.wb = weight_bytes(fmt, N, K)
        self.nbuf = max(2, min(math.ceil(3 * l2_bytes / self.wb), max(2, cap_bytes // self.wb)))
        seed = synth.seed_for(seed_workload, 0)
        if fmt == "q2":
            W, _, _ = synth.q2_weights(N, K, seed)
            S = None
        elif fmt == "w4":
            W, S, _ = synth.w4_weights(N, K, seed)
        else:
            W, S = synth.w8_weights(N, K, seed)
        w0 = G.dev_u8(W)
        self.W = [w0] + [w0.clone() for _ in range(self.nbuf - 1)]
        if S is None:
            self.S = [None] * self.nbuf
        else:
            s0 = G.dev_u8(S) if fmt == "w4" else G.dev_f32(S)
            self.S = [s0] + [s0.clone() for _ in range(self.nbuf - 1)]
        self.A = {M: G.dev_bf16(synth.activations(M, K, synth.seed_for(seed_workload, M))) for M in self.Ms}
        self.C = {M: torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for M in self.Ms}
        self.i = 0

    def call(self, M, A=None, C=None, tc=None):
        import weight_only_quantized_packed_gb300 as wqp

        j = self.i % self.nbuf
        self.i += 1
        A = self.A[M] if A is None else A
        C = self.C[M] if C is None else C
        tc = self.tc if tc is None else tc
        if self.fmt == "q2" and tc == "mma":
            wqp.q2_gemm_mma(A, self.W[j], self.N, self.K, out=C)
        elif self.fmt == "q2" and tc:
            wqp.q2_gemm_tc(A, self.W[j], self.N, self.K, out=C)
        elif self.fmt == "q2":
            wqp.q2_gemv(A, self.W[j], self.N, self.K, out=C)
        elif self.fmt == "w4" and tc == "mma":
            wqp.w4a16_gemm_mma(A, self.W[j], self.S[j], self.N, self.K, out=C)
        elif self.fmt == "w4" and tc:
            wqp.w4a16_gemm_tc(A, self.W[j], self.S[j], self.N, self.K, out=C)
        elif self.fmt == "w4":
            wqp.w4a16_gemv(A, self.W[j], self.S[j], self.N, self.K, out=C)
        elif tc == "mma":
            wqp.w8a16_gemm_mma(A, self.W[j], self.S[j], self.N, self.K, out=C)
        elif tc:
            wqp.w8a16_gemm_tc(A, self.W[j], self.S[j], self.N, self.K, out=C)
        else:
            wqp.w8a16_gemm(A, self.W[j], self.S[j], self.N, self.K, out=C)

    def free(self):
        self.W = self.S = self.A = self.C = None


class GraphSteps:
    """n calls of fn captured once into a CUDA graph (launch attributes such
    as programmatic dependent launch are captured with them); replay() runs
    them with no host work in between."""

    def __init__(self, fn, n, warm=3):
        import torch

        self.n = n
        self.stream = torch.cuda.Stream()
        with torch.cuda.stream(self.stream):
            for _ in range(warm):
                fn()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            for _ in range(n):
                fn()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()


def time_calls(fn, n, warm=3, reps=3):
    """Device time per call (us): a graph of n calls, median of reps replays."""
    import torch

    g = GraphSteps(fn, n, warm)
    g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / n)
    del g
    return statistics.median(out)


# Per-SM pipe rates measured on GB300 with microbenchmarks (lane operations
# or instructions per SM clock), used for the compute view of each line:
# LOP3/PRMT/SHF/IMAD and the packed f16/bf16 multiplies 64, FFMA 128,
# mma.sync m16n8k16 0.5 (and it does not overlap the ALU pipe), the
# E4M3/E2M1 -> f16x2 conversions 32.
PIPE = {"alu": 64.0, "ffma": 128.0, "mma": 0.5, "cvt": 32.0}
# Decode work per weight of each warp-level MMA engine: (ALU lane-ops, cvt lane-ops).
MMA_DECODE = {"q2": (0.5625, 0.0), "w4": (0.5, 0.5), "w8": (0.0, 0.5)}


def compute_view(fmt, path, N, K, M, us, sm_count, f_mhz, bf16_tflops):
    """The engine's compute bound next to the HBM one: the time its pipes
    need at the measured per-SM rates, as a fraction of the call's time."""
    cyc = us * 1e-6 * f_mhz * 1e6            # SM clocks of the call
    w = float(N) * K                         # weights
    if path == "mma":
        alu, cvt = MMA_DECODE[fmt]
        mmas = w / 256.0 * ((M + 7) // 8)
        need = (w * alu / PIPE["alu"] + w * cvt / PIPE["cvt"] + mmas / PIPE["mma"]) / sm_count
        return {"engine": "mma.sync", "pipe_bound_us": round(need / (f_mhz * 1e6) * 1e6, 3),
                "frac": round(need / cyc, 4),
                "model": f"per SM: {alu} ALU + {cvt} cvt lane-ops per weight, {(M + 7) // 8} mma per 256 weights, "
                         "ALU and tensor pipes not overlapping"}
    if path is True:
        flops = 2.0 * 16 * N * K              # M padded to 16 on the MMA's N side
        return {"engine": "tcgen05", "tensor_tflops": round(flops / (us * 1e-6) / 1e12, 2),
                "frac": round(flops / (us * 1e-6) / 1e12 / bf16_tflops, 4),
                "model": "dense bf16 tensor rate (measured cuBLAS peak)"}
    fmas = w * M
    return {"engine": "scalar FFMA", "fma_tflops": round(fmas / (us * 1e-6) / 1e12, 3),
            "frac": round(fmas / cyc / (PIPE["ffma"] * sm_count), 4),
            "model": f"{sm_count} SMs x 128 FP32 lanes x {f_mhz:.0f} MHz"}


def sweep(l2, peak, sm_count, f_mhz, bf16_tflops):
    """us/call, GB/s, HBM fraction and compute view for every workload and
    engine (one line each), PDL on."""
    import torch

    import weight_only_quantized_packed_gb300 as wqp

    out = []
    names = {("q2", False): "q2_gemv", ("q2", True): "q2_gemm_tc", ("q2", "mma"): "q2_gemm_mma",
             ("w4", False): "w4a16_gemv", ("w4", True): "w4a16_gemm_tc", ("w4", "mma"): "w4a16_gemm_mma",
             ("w8", False): "w8a16_gemm", ("w8", True): "w8a16_gemm_tc", ("w8", "mma"): "w8a16_gemm_mma"}
    specs = [
        ("q2", 256, 512, (1,), False, 0),
        ("q2", 5120, 5120, (1, 4, 8, 16), False, 1),
        ("q2", 5120, 5120, (1, 4, 8, 16), True, 1),
        ("q2", 5120, 5120, (1, 4, 8, 16), "mma", 1),
        ("w4", 5120, 5120, tuple(range(1, 9)), False, 2),
        ("w4", 5120, 5120, (1, 4, 8, 16), True, 2),
        ("w4", 5120, 5120, tuple(range(1, 9)) + (16,), "mma", 2),
        ("w8", 17408, 5120, (1, 4, 8, 16), False, 3),
        ("w8", 5120, 17408, (1, 4, 8, 16), False, 3),
        ("w8", 17408, 5120, (1, 8, 16), True, 3),
        ("w8", 5120, 17408, (1, 8, 16), True, 3),
        ("w8", 17408, 5120, (1, 8, 16), "mma", 3),
        ("w8", 5120, 17408, (1, 8, 16), "mma", 3),
    ]
    wqp.set_pdl(True)
    try:
        for fmt, N, K, Ms, tc, wl in specs:
            w = Workload(fmt, N, K, Ms, l2, wl, tc=tc)
            for M in Ms:
                us = time_calls(lambda: w.call(M), max(20, min(400, int(2e5 / max(1, w.wb // 4096)))))
                gbs = w.wb / us / 1e3
                out.append({"workload": f"{names[(fmt, tc)]} N={N} K={K}", "M": M, "us": round(us, 3),
                            "gbs": round(gbs, 1), "pct_peak": round(100 * gbs / peak, 1),
                            "compute_view": compute_view(fmt, tc, N, K, M, us, sm_count, f_mhz, bf16_tflops)})
            w.free()
            torch.cuda.empty_cache()
        ws = layer_workloads((1, 4, 8, 16))
        lb = sum(w.wb for w in ws)
        for path, M in [(p, M) for p in (True, "mma") for M in (1, 4, 8, 16)]:
            us = time_calls(lambda: [w.call(M, tc=path) for w in ws], 40)
            out.append({"workload": "q2 decoder layer (qkv+o+gate_up+down), 8 layers cycled", "M": M,
                        "path": Q2_PATH[path],
                        "us_per_layer": round(us, 3), "gbs": round(lb / us / 1e3, 1),
                        "pct_peak": round(100 * lb / us / 1e3 / peak, 1)})
        del ws
        torch.cuda.empty_cache()
    finally:
        wqp.set_pdl(False)
    return out


def gpu_arm(args, rank, world, local_rank):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import weight_only_quantized_packed_gb300 as wqp

    torch.cuda.set_device(local_rank)
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    peak, sm_max_nominal, peak_kind = peaks()
    dist = None
    if world > 1:
        import torch.distributed as dist

    H = HEADLINE
    w = Workload(H["fmt"], H["N"], H["K"], H["Ms"], l2, 1)
    bytes_step = w.wb * len(H["Ms"])
    wqp.set_pdl(args.pdl)

    def step():
        for M in H["Ms"]:
            w.call(M, tc=H["tc"][M])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # The timed steps run as replays of a CUDA graph of G steps (no host work
    # between calls, as a decode loop would run them).
    G = 100 if args.steps % 100 == 0 else (50 if args.steps % 50 == 0 else args.steps)
    steps_graph = GraphSteps(step, G)
    if dist:
        dist.barrier()
    with ClockSampler(dev) as clk:
        # Keep the clock sampler's window filled with work before and after.
        t_end = time.time() + 0.3
        while time.time() < t_end:
            steps_graph.replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        # REPS timed regions, each of exactly `steps` steps bracketed by a
        # synchronize (and a barrier across ranks); the line reports their
        # median and spread.
        stream = steps_graph.stream
        reps_ms = []
        for _ in range(args.reps):
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(args.steps // G):
                    steps_graph.replay()
                e1.record(stream)
            e1.synchronize()
            reps_ms.append(e0.elapsed_time(e1))
        if dist:
            dist.barrier()
        ms_total = statistics.median(reps_ms)
        # Per-kernel durations: each call of the step alone, as a graph of
        # back-to-back calls (events on the launching stream around it).
        avg = {M: time_calls(lambda M=M: w.call(M, tc=H["tc"][M]), 200) for M in H["Ms"]}
    del steps_graph
    wqp.set_pdl(False)
    ms_total = reduce_max_ms(ms_total, dist)
    ms_step = ms_total / args.steps
    value = job_value(bytes_step, args.steps, world, ms_total)

    # Dominant kernel: the call with the largest average duration.
    Mdom = max(avg, key=avg.get)
    us_dom = avg[Mdom]
    tc_dom = H["tc"][Mdom]
    kname = Q2_PATH[tc_dom]
    achieved = w.wb / (us_dom * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "kernel": f"{kname} M={Mdom} N={H['N']} K={H['K']}",
                "algorithmic_bytes_per_launch": w.wb,
                "traffic": committed_traffic(f"{kname}_M{Mdom}_N{H['N']}_K{H['K']}", tc_dom)}
    # Compute view of the same kernel: the time its pipes need at the measured
    # per-SM rates, as a fraction of its duration.
    sm_count = props.multi_processor_count
    clk_sum = clk.summary()
    f_mhz = clk_sum["sm_mhz"] or sm_max_nominal
    bf16_tflops = peak_bf16()
    roofline["compute_view"] = compute_view(H["fmt"], tc_dom, H["N"], H["K"], Mdom, us_dom, sm_count, f_mhz,
                                            bf16_tflops)

    # End-to-end through the C ABI with host buffers (pinned): per step copy
    # the three activation blocks in, compute, copy the three outputs back.
    e2e = e2e_arm(w, H, max(20, min(args.steps, 2000)))
    e2e["value"] = round(e2e["value"] * world, 2)
    host_us = host_call_us(w, H)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded; A ~ N(0,1) bf16, ternary codes U{0,1,2}, d U[0.01,0.05] fp16)",
        "config": {"workload": WORKLOAD,
                   "paths": {str(M): Q2_PATH[H["tc"][M]] for M in H["Ms"]},
                   "timing": f"median of {args.reps} timed regions of {args.steps} steps (each a CUDA graph of "
                             f"{G} steps replayed {args.steps // G} times, synchronised on both sides)",
                   "weight_bytes_per_call": w.wb, "weight_buffers_cycled": w.nbuf,
                   "l2": f"inputs larger than L2: {w.nbuf} weight buffers = {w.nbuf * w.wb / 2**20:.0f} MiB > 3x L2 ({l2 / 2**20:.0f} MiB)",
                   "pdl": bool(args.pdl), "parallelism": f"replicas x{world}"},
        "timed_regions_ms": {"median": round(statistics.median(reps_ms), 4), "min": round(min(reps_ms), 4),
                             "max": round(max(reps_ms), 4), "n": len(reps_ms)},
        "us_per_call": {str(M): round(avg[M], 3) for M in H["Ms"]},
        "pct_of_peak": round(100 * value / world / peak, 2),
        "roofline": roofline, "e2e": e2e,
        "host_us_per_call": host_us,
        "gpu_launches": args.steps * len(H["Ms"]),
        "clocks": clk_sum,
    }
    w.free()
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_sweep:
        line["sweep"] = sweep(l2, peak, sm_count, f_mhz, bf16_tflops)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    return line


def host_call_us(w, H, n=400):
    """Host time to issue one call through the public Python API (argument
    marshalling, the C call's checks, plan and tensor-map lookups and the
    launch), per M of the step: n calls issued back to back without waiting,
    so the GPU, at about 4 us per call, keeps the launch queue short."""
    import torch

    out = {}
    for M in H["Ms"]:
        for _ in range(20):
            w.call(M, tc=H["tc"][M])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            w.call(M, tc=H["tc"][M])
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        out[str(M)] = round((t1 - t0) / n * 1e6, 2)
    out["how"] = f"{n} back-to-back calls per M through the Python binding, host wall time per call"
    return out


def e2e_arm(w, H, steps):
    """The same step end to end through the public API with host buffers:
    every step copies the three activation blocks in from pinned host memory
    (one copy: they sit in one pinned buffer), runs the three calls on views
    of one device buffer, and reads the three outputs back (one copy).
    Timed two ways: the step's API calls captured once into a CUDA graph and
    replayed per step (copies included in every replay), and the same calls
    issued from Python every step."""
    import torch

    Ms = H["Ms"]
    rows = sum(Ms)
    off = {}
    o = 0
    for M in Ms:
        off[M] = o
        o += M
    hA = torch.empty((rows, w.K), dtype=torch.bfloat16).pin_memory()
    for M in Ms:
        hA[off[M]:off[M] + M].copy_(w.A[M].cpu())
    hC = torch.empty((rows, w.N), dtype=torch.bfloat16).pin_memory()
    dA = torch.empty((rows, w.K), dtype=torch.bfloat16, device="cuda")
    dC = torch.empty((rows, w.N), dtype=torch.bfloat16, device="cuda")
    h2d = hA.numel() * 2
    d2h = hC.numel() * 2

    vA = {M: dA[off[M]:off[M] + M] for M in Ms}
    vC = {M: dC[off[M]:off[M] + M] for M in Ms}

    def step():
        dA.copy_(hA, non_blocking=True)
        for M in Ms:
            w.call(M, A=vA[M], C=vC[M], tc=H["tc"][M])
        hC.copy_(dC, non_blocking=True)

    def timed(run, n):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        run(n)
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1), time.perf_counter() - t0

    for _ in range(5):
        step()
    ms_eager, wall_eager = timed(lambda n: [step() for _ in range(n)], steps)
    # Graph of G steps (each with its two copies), replayed.
    G = 50
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(G):
            step()
    g.replay()
    reps = max(1, steps // G)

    def replay(_n):
        for _ in range(reps):
            g.replay()

    # The median of five timed regions of reps * G steps each.
    regions = [timed(replay, reps) for _ in range(5)]
    ms_graph, wall_graph = sorted(regions)[len(regions) // 2]
    del g
    bytes_step = w.wb * len(Ms)
    return {"value": bytes_step * reps * G / (ms_graph * 1e-3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": reps * G,
            "copies_per_step": {"h2d": 1, "d2h": 1},
            "how": "the step's public-API calls (H2D copy, three GEMM calls, D2H copy) captured in a CUDA graph of "
                   f"{G} steps and replayed; every step's copies run inside the timed region; the median of "
                   f"{len(regions)} timed regions of {reps * G} steps",
            "regions_ms": {"median": round(ms_graph, 4), "min": round(min(r[0] for r in regions), 4),
                           "max": round(max(r[0] for r in regions), 4)},
            "wall_s": round(wall_graph, 4),
            "eager": {"value": round(bytes_step * steps / (ms_eager * 1e-3) / 1e9, 2), "unit": UNIT, "steps": steps,
                      "how": "the same calls issued from Python every step", "wall_s": round(wall_eager, 4)}}


# ------------------------------------------------------------------ CPU oracle
def cpu_baseline(seconds=10.0, rows=None):
    """The CPU oracle, as it stands, timed on the host's cores on a bounded
    sample of the headline step: the three calls restricted to the first
    `rows` weight rows, repeated for about `seconds`."""
    import oracle
    from weight_only_quantized_packed_gb300 import synth

    oracle.build()
    H = HEADLINE
    N, K = H["N"], H["K"]
    rows = rows or N
    W, _, _ = synth.q2_weights(N, K, synth.seed_for(1, 0))
    W = W[:rows]
    As = {M: synth.activations(M, K, synth.seed_for(1, M)) for M in H["Ms"]}
    wb = synth.q2_weight_bytes(rows, K)
    t0 = time.perf_counter()
    n = 0
    while True:
        for M in H["Ms"]:
            oracle.q2_gemv(As[M], W, M, rows, K)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    cores = oracle.max_threads()
    line = {"value": round(wb * len(H["Ms"]) * n / dt / 1e9, 4), "unit": UNIT,
            "cores": cores, "kind": "oracle",
            "sample": f"{n} x (q2 M=1,4,8 over {rows} of {N} rows, K={K}); {dt:.1f} s"}
    # The same oracle on one host thread, on a sixteenth of the rows.
    rows1 = max(8, rows // 16)
    W1 = W[:rows1]
    wb1 = synth.q2_weight_bytes(rows1, K)
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        n1 = 0
        while True:
            for M in H["Ms"]:
                oracle.q2_gemv(As[M], W1, M, rows1, K)
            n1 += 1
            if time.perf_counter() - t0 >= seconds / 4:
                break
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_threads(cores)
    line["one_thread"] = {"value": round(wb1 * len(H["Ms"]) * n1 / dt1 / 1e9, 4), "unit": UNIT, "cores": 1,
                          "sample": f"{n1} x (q2 M=1,4,8 over {rows1} of {N} rows, K={K}); {dt1:.1f} s"}
    return line


def reference_arm(args, rank, world):
    """The oracle as the reference arm: rank 0 only, on the host's cores."""
    if rank != 0:
        return None
    import oracle

    oracle.build()
    H = HEADLINE
    # Size each step so that warmup + steps finish in about a minute.
    t_full = 0.7                          # s for a full step on 8 cores (measured)
    per_step = 60.0 / max(1, args.steps + args.warmup)
    rows = max(8, min(H["N"], int(H["N"] * per_step / t_full)))
    from weight_only_quantized_packed_gb300 import synth

    W, _, _ = synth.q2_weights(H["N"], H["K"], synth.seed_for(1, 0))
    W = W[:rows]
    As = {M: synth.activations(M, H["K"], synth.seed_for(1, M)) for M in H["Ms"]}
    wb = synth.q2_weight_bytes(rows, H["K"])

    def step():
        for M in H["Ms"]:
            oracle.q2_gemv(As[M], W, M, rows, H["K"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = wb * len(H["Ms"]) * args.steps / dt / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": f"{rows} of {H['N']} rows per step"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# The Q2_0 decoder layer of the sweep: qkv, o, gate+up and down (N, K).
Q2_LAYER = [(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)]


def layer_workloads(Ms):
    """The four projections of a Q2_0 decoder layer, 8 layers' weights
    cycled (702 MB, past L2): one generated buffer per shape and 7 copies."""
    ws = [Workload("q2", N, K, Ms, 0, 4, cap_bytes=0) for (N, K) in Q2_LAYER]
    for w in ws:
        w.nbuf = 8
        w.W = [w.W[0]] + [w.W[0].clone() for _ in range(7)]
    return ws


def profile_case(case, launches, pdl):
    """A fixed number of launches of one call shape (fmt:M:N:K[:tc|:mma]),
    or of decoder-layer passes (layer:M[:tc|:mma], four calls each), for ncu
    captures."""
    import torch

    import weight_only_quantized_packed_gb300 as wqp

    parts = case.split(":")
    wqp.set_pdl(bool(pdl))
    if parts[0] == "layer":
        M = int(parts[1])
        tc = {"tc": True, "mma": "mma"}.get(parts[2], False) if len(parts) > 2 else False
        ws = layer_workloads((M,))
        for _ in range(launches):
            for w in ws:
                w.call(M, tc=tc)
        nbuf = ws[0].nbuf
    else:
        fmt, M, N, K = parts[0], int(parts[1]), int(parts[2]), int(parts[3])
        tc = {"tc": True, "mma": "mma"}.get(parts[4], False) if len(parts) > 4 else False
        # About 192 MiB of cycled weights: past L2 (129 MB), well under 1 GiB on the device.
        w = Workload(fmt, N, K, (M,), 64 << 20, 9, tc=tc, cap_bytes=1 << 30)
        for _ in range(launches):
            w.call(M)
        nbuf = w.nbuf
    torch.cuda.synchronize()
    err = wqp.get_device_error()
    print(json.dumps({"case": case, "launches": launches, "buffers": nbuf, "device_error": err}))
    if err:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="wqp", choices=["wqp", "reference"])
    ap.add_argument("--pdl", type=int, default=1, help="programmatic dependent launch (1/0)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reps", type=int, default=7, help="timed regions of --steps steps; the median is reported")
    ap.add_argument("--case", default=None,
                    help="profiling mode: run --launches calls of one shape, fmt:M:N:K[:tc|:mma] "
                         "(fmt q2|w4|w8), or --launches Q2_0 decoder-layer passes, layer:M[:tc|:mma]; "
                         "weights cycled past L2; prints one status line")
    ap.add_argument("--launches", type=int, default=6)
    args = ap.parse_args()
    if args.case:
        profile_case(args.case, args.launches, args.pdl)
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", rank=rank, world_size=world)
    line = gpu_arm(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
