#!/usr/bin/env python
"""Benchmark of the INT8ConvRot (W8A8 Hadamard-rotated) linear on GB300.

Workload (default): the 448-layer sweep at M = 1024 over the six (N, K)
weight shapes and layer counts of the page "INT8ConvRot GEMM vs fp16 on M1
Max with Metal, MPSMatrix, and MLX" (section "Testing the MPS weight-only
INT8 path in isolation"): 2048x2048 x168, 256x2048 x84, 6144x256 x84,
2048x1024 x56, 8192x2048 x28, 2048x8192 x28.  One step = one call of the layer
for each of the 448 layers, each with its own activation, prepared weight and
output (synthetic, seeded; ~12 GB touched per step, far above the 129 MB L2).
The metric is whole-sweep TOPS (2*M*N*K summed over the layers, divided by
the step time); ms_per_step is the layer-count-weighted sum of per-layer
times.  Weight preparation is one-time and not timed.

Output: one JSON line on rank 0.
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "ConvRot W8A8 linear TOPS, 6-shape M=1024 sum ms; % of int8 tensor peak"
UNIT = "TOPS"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["sweep", "attn", "msweep", "lora"], default="sweep",
                    help="sweep: the 448-layer M=1024 mix (the headline); attn, msweep, lora: "
                         "the other workloads, for per-config numbers")
    ap.add_argument("--seed", type=int, default=2)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="rows per shape in the oracle sample (0 = calibrate)")
    # Profiling subsets (not the headline workload): restrict the sweep to
    # some shapes and cap the layers per shape; skip the per-kernel breakdown.
    ap.add_argument("--shapes", type=str, default="",
                    help="comma-separated shape indices 0..5 (default: all)")
    ap.add_argument("--layers-per-shape", type=int, default=0)
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--no-comparator", action="store_true",
                    help="skip the fp16 cuBLAS comparator on the same layers")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# Distributed plumbing (one process per GPU under torchrun; replicas only).
# ----------------------------------------------------------------------------

class Dist:
    def __init__(self, want: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if _cuda_ok() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if _cuda_ok() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# ----------------------------------------------------------------------------
# Clock sampling during the timed region.
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"convrot_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm.append(float(parts[2]))
                    smax.append(float(parts[3]))
                    power.append(float(parts[4]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[6:10]):
                    if val.lower() == "active":
                        reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm) // 2], "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------
# Our arm: the sweep through the C ABI.
# ----------------------------------------------------------------------------

def workload_groups(config: str):
    """Layer groups of a workload: dicts of M, N, K, R, lora_scale, count."""
    if config == "sweep":
        return [dict(M=workloads.SWEEP_M, N=N, K=K, R=0, lora_scale=0.0, count=c,
                     name=f"{N}x{K}") for N, K, c in workloads.SWEEP_SHAPES]
    if config == "attn":
        c = workloads.ATTN
        # 32 distinct copies so a step touches ~0.5 GB (more than L2).
        return [dict(M=c.M, N=c.N, K=c.K, R=0, lora_scale=0.0, count=32, name="attn")]
    if config == "msweep":
        # Small-M layers are weight streams: 16 distinct layers of each, so
        # their weights (16 x 16.8 MB) exceed L2 and a layer's time is read
        # from a multi-layer graph.
        return [dict(M=c.M, N=c.N, K=c.K, R=0, lora_scale=0.0, count=16 if c.M <= 16 else 1,
                     name=c.name) for c in workloads.m_sweep_configs()]
    if config == "lora":
        c = workloads.LORA
        return [dict(M=c.M, N=c.N, K=c.K, R=c.R, lora_scale=c.lora_scale, count=2, name="lora")]
    raise ValueError(config)


WORKLOAD_TEXT = {
    "sweep": "ConvRot W8A8 linear, 448-layer sweep at M=1024 over 6 (N,K) shapes "
             "(2048x2048 x168, 256x2048 x84, 6144x256 x84, 2048x1024 x56, "
             "8192x2048 x28, 2048x8192 x28)",
    "attn": "ConvRot W8A8 linear M=1024 N=2048 K=2048 (attention projection), "
            "32 distinct layers per step",
    "msweep": "ConvRot W8A8 linear, M in {1,16,128,4096,16384} x (N,K) in "
              "{(8192,2048),(2048,8192)}, 16 distinct layers each at M <= 16, one above",
    "lora": "ConvRot W8A8 linear with unmerged LoRA, M=4096 N=2048 K=8192 R=32 "
            "scale 0.8, 2 distinct layers per step",
}


class Sweep:
    """Device buffers for every layer of a workload and the calls of one step."""

    def __init__(self, seed: int, groups, shapes=None, cap: int = 0):
        import torch
        import w8a8_hadamard_rotated_gb300 as cr
        self.torch, self.cr = torch, cr
        self.groups = groups
        self.seed = seed
        self.layers = []
        self.counts = {}
        ws_bytes = 0
        for si, grp in enumerate(groups):
            if shapes is not None and si not in shapes:
                continue
            M, N, K, R, count = grp["M"], grp["N"], grp["K"], grp["R"], grp["count"]
            if cap:
                count = min(count, cap)
            self.counts[si] = count
            n_out = workloads.n_outliers(K)
            for i in range(count):
                g = torch.Generator(device="cuda")
                g.manual_seed(seed * 1_000_000 + si * 1000 + i)
                x = torch.randn((M, K), generator=g, device="cuda")
                cols = torch.randperm(K, generator=g, device="cuda")[:n_out]
                x[:, cols] *= workloads.OUTLIER_SCALE
                X = x.half()
                del x
                W = torch.randn((N, K), generator=g, device="cuda") / math.sqrt(K)
                Q_W = torch.empty((N, K), dtype=torch.int8, device="cuda")
                s_W = torch.empty((N,), dtype=torch.float32, device="cuda")
                img = torch.empty((N, K), dtype=torch.float16, device="cuda")
                cr.convrot_prepare_weight(W, Q_W, s_W, img)
                del W
                down = up = None
                if R:
                    down = (torch.randn((R, K), generator=g, device="cuda") * 0.01).half()
                    up = (torch.randn((N, R), generator=g, device="cuda") * 0.01).half()
                Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
                self.layers.append(dict(M=M, N=N, K=K, R=R, scale=grp["lora_scale"], shape=si,
                                        X=X, Q_W=Q_W, s_W=s_W, img=img, Y=Y, down=down, up=up))
                ws_bytes = max(ws_bytes, cr.convrot_linear_workspace_bytes(M, N, K, R, True))
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        assert cr.convrot_check_device_error() == 0
        self.ops = float(sum(2.0 * L["M"] * L["N"] * L["K"] for L in self.layers))
        self.subset = (shapes is not None) or bool(cap)
        self.bytes_touched = sum(
            L["X"].numel() * 2 + L["img"].numel() * 2 + L["Y"].numel() * 2 + L["s_W"].numel() * 4
            for L in self.layers)

    def call(self, L):
        self.cr.convrot_linear(L["X"], L["Q_W"], L["s_W"], L["Y"], self.ws, W_img=L["img"],
                               lora_down=L["down"], lora_up=L["up"], lora_scale=L["scale"])

    def step(self):
        for L in self.layers:
            self.call(L)

    def layers_only(self, shape_index: int):
        for L in self.layers:
            if L["shape"] == shape_index:
                self.call(L)

    def gemm_only(self, shape_index: int):
        cr = self.cr
        for L in self.layers:
            if L["shape"] == shape_index:
                cr.convrot_linear_gemm(L["M"], L["K"], L["Q_W"], L["s_W"], L["Y"], self.ws,
                                       W_img=L["img"], lora_up=L["up"], lora_scale=L["scale"])

    def prologue_only(self, shape_index: int):
        cr = self.cr
        for L in self.layers:
            if L["shape"] == shape_index:
                cr.convrot_linear_prologue(L["X"], L["N"], self.ws, lora_down=L["down"],
                                           with_weight_image=True)

    def first_layer_of(self, shape_index: int):
        for L in self.layers:
            if L["shape"] == shape_index:
                return L
        raise KeyError(shape_index)

    def launches_per_step(self) -> int:
        # What the library launches per call under its engine choice (one
        # kernel for a small-M layer; rotate+quantize, [LoRA down, LoRA up,]
        # GEMM otherwise).
        return sum(self.cr.convrot_linear_kernel_count(L["M"], L["N"], L["K"], L["R"], True)
                   for L in self.layers)


def graph_of(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # eager run first (lazy init, errors surface here)
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    stream.synchronize()
    return g


def replay(torch, stream, g, reps: int = 1):
    # CUDAGraph.replay() launches on the current stream: make it `stream`.
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()


def time_graph(torch, stream, g, reps: int) -> float:
    """Average ms per replay, CUDA events on the replay stream."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    replay(torch, stream, g, reps)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def clock_stop(clocks):
    return clocks.stop()


def run_ours(args, dist: Dist):
    import torch
    import w8a8_hadamard_rotated_gb300 as cr

    cr.build()
    cr.load()
    torch.cuda.set_device(dist.local_rank)
    peaks, peak_src = load_peaks()
    shapes = {int(v) for v in args.shapes.split(",")} if args.shapes else None
    groups = workload_groups(args.config)
    sweep = Sweep(args.seed + dist.rank, groups, shapes=shapes, cap=args.layers_per_shape)
    stream = torch.cuda.Stream()
    g_step = graph_of(torch, stream, sweep.step)

    # Warm-up, then exactly K timed steps bracketed by barrier + synchronize.
    replay(torch, stream, g_step, args.warmup)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    replay(torch, stream, g_step, args.steps)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - w0) * 1e3 / args.steps
    dist.barrier()
    clock_info = clock_stop(clocks)
    ms_local = e0.elapsed_time(e1) / args.steps
    # The device time of a step can never exceed its wall time.
    assert ms_local <= wall_ms * 1.05 + 0.05, (ms_local, wall_ms)
    ms = dist.max(ms_local)
    detail = cr.convrot_check_device_error()
    if detail:
        raise RuntimeError(f"device error flag {detail} after the timed region")

    # Per-kernel breakdown: each shape's whole layers, GEMM stage and prologue
    # alone, each back to back in a graph over that shape's layers, timed
    # with CUDA events on the launching stream.  (A small-M layer runs as one
    # kernel; its GEMM and prologue stages are the two-kernel path's.)
    per_shape = []
    gemm_ms_total = 0.0
    pro_ms_total = 0.0
    flops_total = 0.0
    reps = max(3, min(20, args.steps // 5 or 3))
    for si, grp in enumerate(groups):
        if args.no_breakdown or si not in sweep.counts:
            continue
        count = sweep.counts[si]
        M, N, K = grp["M"], grp["N"], grp["K"]
        gg = graph_of(torch, stream, lambda: sweep.gemm_only(si))
        gp = graph_of(torch, stream, lambda: sweep.prologue_only(si))
        gl = graph_of(torch, stream, lambda: sweep.layers_only(si))
        replay(torch, stream, gg, 2)
        replay(torch, stream, gp, 2)
        replay(torch, stream, gl, 2)
        t_gemm = time_graph(torch, stream, gg, reps) / count
        t_pro = time_graph(torch, stream, gp, reps) / count
        t_layer = time_graph(torch, stream, gl, reps) / count
        flops = 2.0 * M * N * K
        pbytes = 3.0 * M * K + 4.0 * M  # algorithmic: fp16 X in, int8 codes out, s_X
        per_shape.append({
            "M": M, "N": N, "K": K, "R": grp["R"], "layers": count,
            "layer_us": round(t_layer * 1e3, 3),
            "kernels_per_layer": cr.convrot_linear_kernel_count(M, N, K, grp["R"], True),
            "gemm_us": round(t_gemm * 1e3, 3), "prologue_us": round(t_pro * 1e3, 3),
            "gemm_tflops": round(flops / (t_gemm * 1e-3) / 1e12, 1),
            "prologue_gbs": round(pbytes / (t_pro * 1e-3) / 1e9, 1),
        })
        gemm_ms_total += count * t_gemm
        pro_ms_total += count * t_pro
        flops_total += count * flops
        del gg, gp, gl
    assert cr.convrot_check_device_error() == 0
    if per_shape:
        gemm_tflops = flops_total / (gemm_ms_total * 1e-3) / 1e12
        pro_bytes = sum(sweep.counts[si] * (3.0 * groups[si]["M"] * groups[si]["K"]
                                            + 4.0 * groups[si]["M"]) for si in sweep.counts)
        pro_alg_gbs = pro_bytes / (pro_ms_total * 1e-3) / 1e9
    else:
        gemm_tflops = pro_alg_gbs = float("nan")

    # The pages' question, "does W8A8 beat fp16?", on this GPU: the same
    # layers as a plain fp16 product (torch.mm, i.e. cuBLAS) into the same Y
    # buffers, one graph, timed like the step.  A comparator only.
    comparator = w8a16 = None
    if not args.no_comparator and args.config == "sweep":
        comparator = fp16_comparator(torch, stream, sweep, reps=max(3, min(20, args.steps)),
                                     ms_w8a8=ms)
        w8a16 = w8a16_comparator(torch, stream, sweep, reps=max(3, min(20, args.steps)),
                                 ms_w8a8=ms)

    # End to end through the host-buffer entry point: per layer, H2D of X from
    # pinned memory, the layer, D2H of Y; the step ends when Y is on the host.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, sweep, stream, dist)

    # Ceilings of the two exact int8 product engines on this GPU, measured
    # live (back-to-back MMAs on resident operands, every SM).
    engines = engine_peaks(cr)
    # Quantization error of the layer against the unquantized fp64 X W^T, on
    # a row sample of the first layer of each group.
    qerr = quant_error(torch, sweep, groups)

    value = dist.world * sweep.ops / (ms * 1e-3) / 1e12
    launches_per_step = sweep.launches_per_step()
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8",
        "data": "synthetic (seeded normal activations with 1% x50 outlier columns, "
                "normal weights std 1/sqrt(K); weights prepared on the GPU, untimed)",
        "config": {
            "workload": WORKLOAD_TEXT[args.config],
            "layers": len(sweep.layers), "total_tops_per_step": sweep.ops / 1e12,
            "l2": f"inputs larger than L2: {sweep.bytes_touched / 1e9:.1f} GB of distinct "
                  "activations, weights and outputs per step",
            "launch": f"one CUDA graph per step ({len(sweep.layers)} x convrot_linear)",
            "weight_operand": "fp16 image of the int8 weight (exact)",
            "parallelism": f"replicas x{dist.world}",
            "subset": sweep.subset,
        },
        "weighted_sum_ms": round(ms, 4),
        "wall_ms_per_step": round(wall_ms, 4),
        "roofline": dominant_gemm_roofline(per_shape, peaks, peak_src, len(sweep.layers),
                                           engines),
        "gemm_all_shapes": {
            "achieved": round(gemm_tflops, 1), "unit": "TFLOP/s",
            "frac": round(gemm_tflops / peaks["bf16_tflops"], 4),
            "frac_of_int8_engine_peak": (round(gemm_tflops / engines["tcgen05_f16_tflops"], 4)
                                         if engines else None),
            "note": "every GEMM launch of the step: sum of 2MNK over the sum of per-shape "
                    "GEMM-only graph times",
        },
        "prologue_roofline": {
            "bound": "hbm", "achieved": round(pro_alg_gbs, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(pro_alg_gbs / peaks["hbm_gbs"], 4),
            "algorithmic_bytes": "3*M*K + 4*M per call (fp16 X in, int8 codes out, fp32 s_X)",
            "note": "the kernel writes the codes as an fp16 image (4*M*K + 4*M actual bytes)",
        },
        "gemm_ms_per_step": round(gemm_ms_total, 4),
        "prologue_ms_per_step": round(pro_ms_total, 4),
        "per_shape": per_shape,
        "engine_peaks": engines,
        "quant_error": qerr,
        "clocks": clock_info,
        "gpu_launches": launches_per_step * args.steps,
    }
    if e2e:
        result["e2e"] = e2e
    if comparator:
        result["fp16_comparator"] = comparator
    if w8a16:
        result["w8a16_comparator"] = w8a16
    if args.config != "sweep":
        result["metric"] = f"ConvRot W8A8 linear TOPS ({args.config} workload)"
        result.pop("weighted_sum_ms")
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and args.config == "sweep":
        result["cpu_baseline"] = cpu_baseline(args, budget_s=20.0)
    return result


# DRAM traffic of one GEMM launch (dram__bytes_read.sum + dram__bytes_write.sum)
# from an ncu capture, keyed by (M, N, K), with a hash of the kernel sources it
# was taken on: reported only while the sources are unchanged.
GEMM_TRAFFIC_CAPTURES = {
    (1024, 2048, 2048): {"bytes": 12665600, "sources": "b16542c24224e439",
                         "profile": "profiles/gemm_tc_2048x2048_m1024_ncu.md"},
}
GEMM_SOURCES = ("gemm_tc.cu", "common.cuh", "epilogue.cuh", "fwht.cuh", "kernels.h")


def gemm_sources_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    root = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "w8a8_hadamard_rotated_gb300", "csrc")
    for f in GEMM_SOURCES:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def engine_peaks(cr):
    """Measured ceilings of the exact int8 product engines (convrot_measure_engine_peak):
    tcgen05 kind::f16 on integer operands (the large-M paths), mma.sync
    m16n8k16 f16 (the small-M GEMM at M >= 3), dp4a (the one-kernel small-M
    layer) and mma.sync m16n8k32 s8 (the small-M GEMM's other kernel).  Best
    of three runs of ~5-40 ms each."""
    out = {}
    for eng, key, reps in ((cr.CONVROT_PEAK_MMA_S8, "mma_sync_s8_tops", 20000),
                           (cr.CONVROT_PEAK_TCGEN05_F16, "tcgen05_f16_tflops", 20000),
                           (cr.CONVROT_PEAK_MMA_F16, "mma_sync_f16_tflops", 20000),
                           (cr.CONVROT_PEAK_DP4A, "dp4a_tops", 20000)):
        best = 0.0
        for _ in range(3):
            ops, ms = cr.convrot_measure_engine_peak(eng, reps)
            best = max(best, ops / (ms * 1e-3) / 1e12)
        out[key] = round(best, 1)
    out["note"] = ("back-to-back instructions on operands already in registers / shared "
                   "memory, all SMs, no loads: sm_103a has no integer tcgen05 MMA, so the "
                   "int8 x int8 -> int32 product runs on tcgen05 kind::f16 with exact operands "
                   "(large M; the int8 tensor peak of this GPU), on mma.sync m16n8k16 f16 with "
                   "exact operands (the small-M GEMM at M >= 3), on dp4a (the one-kernel "
                   "small-M layer at M <= 2) or on mma.sync s8 (the small-M GEMM's other kernel)")
    return out


def quant_error(torch, sweep: Sweep, groups, rows: int = 128):
    """Relative L2 and max-abs error of the layer's fp16 Y against the
    unquantized product X W^T (+ LoRA) in fp64, on the first `rows` rows of
    the first layer of each group (W rebuilt from the same generator)."""
    out = []
    for si, grp in enumerate(groups):
        if si not in sweep.counts:
            continue
        L = sweep.first_layer_of(si)
        M, N, K = L["M"], L["N"], L["K"]
        r = min(rows, M)
        g = torch.Generator(device="cuda")
        g.manual_seed(sweep.seed * 1_000_000 + si * 1000 + 0)
        torch.randn((M, K), generator=g, device="cuda")
        torch.randperm(K, generator=g, device="cuda")
        W = torch.randn((N, K), generator=g, device="cuda") / math.sqrt(K)
        sweep.call(L)
        torch.cuda.synchronize()
        x = L["X"][:r].double()
        ref = x @ W.double().t()
        if L["R"]:
            ref += L["scale"] * (x @ L["down"].double().t()) @ L["up"].double().t()
        y = L["Y"][:r].double()
        d = y - ref
        out.append({"M": M, "N": N, "K": K, "R": L["R"], "rows": r,
                    "rel_l2": float(d.norm() / ref.norm()),
                    "max_abs": float(d.abs().max()),
                    "max_abs_ref": float(ref.abs().max())})
        del W, ref, x, y, d
    return out


def dominant_gemm_roofline(per_shape, peaks, peak_src, layers, engines=None):
    """Roofline of the dominant kernel: the tensor-core GEMM on the shape that
    takes the largest share of the step's GEMM time; achieved = 2MNK of one
    launch / that shape's average launch time (CUDA events, GEMM-only graph)."""
    if not per_shape:
        return {"bound": "tensor", "achieved": None, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": None, "traffic": None}
    top = max(per_shape, key=lambda x: x["layers"] * x["gemm_us"])
    M, N, K = top["M"], top["N"], top["K"]
    ach = 2.0 * M * N * K / (top["gemm_us"] * 1e-6) / 1e12
    # At M <= 16 the GEMM stage is the small-M GEMM on the warp MMA (the
    # library's automatic path), above it the tcgen05 GEMM.
    small = M <= 16
    kname = ("small-M GEMM (skinny_f16_kernel: mma.sync m16n8k16 f16, exact int8 operands)"
             if small else "gemm_tc_kernel (tcgen05 kind::f16, exact int8 operands)")
    eng_key = "mma_sync_f16_tflops" if small else "tcgen05_f16_tflops"
    cap = GEMM_TRAFFIC_CAPTURES.get((M, N, K))
    traffic = cap["bytes"] if cap and cap["sources"] == gemm_sources_hash() else None
    return {
        "bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
        "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": traffic,
        "traffic_unit": "bytes per launch",
        "algorithmic_bytes": M * K + N * K + 2 * M * N + 4 * M + 4 * N,
        "operand_image_bytes": 2 * M * K + 2 * N * K,
        "traffic_note": "the operands travel as exact fp16 images of the int8 codes "
                        "(no integer MMA on sm_103a); Y stays in L2 at kernel end",
        "kernel": f"{kname} on M={M} N={N} K={K}, {top['layers']} of {layers} layers",
        "peak_source": f"{peak_src} bf16 dense burst (f16 runs at the bf16 rate)",
        "frac_of_int8_engine_peak": (round(ach / engines[eng_key], 4)
                                     if engines else None),
        "int8_engine_peak_source": ("mma.sync m16n8k16 f16" if small else "tcgen05 kind::f16")
                                   + " back-to-back MMAs measured live (engine_peaks)",
    }


def fp16_comparator(torch, stream, sweep: Sweep, reps: int, ms_w8a8: float):
    """Y = X W^T in fp16 with fp32 accumulation (torch.mm -> cuBLAS) for every
    layer of the step, with seeded random fp16 weights of the same shapes."""
    weights = []
    for i, L in enumerate(sweep.layers):
        g = torch.Generator(device="cuda")
        g.manual_seed(7_000_000 + i)
        weights.append((torch.randn((L["N"], L["K"]), generator=g, device="cuda")
                        / math.sqrt(L["K"])).half())

    def step():
        for L, W in zip(sweep.layers, weights):
            torch.mm(L["X"], W.t(), out=L["Y"])

    g = graph_of(torch, stream, step)
    replay(torch, stream, g, 3)
    ms = time_graph(torch, stream, g, reps)
    del g, weights
    return {
        "impl": "torch.mm fp16 x fp16 -> fp16 (cuBLAS), same 448 layers and X/Y buffers",
        "ms_per_step": round(ms, 4), "tops": round(sweep.ops / (ms * 1e-3) / 1e12, 2),
        "w8a8_speedup": round(ms / ms_w8a8, 3),
        "note": "fp16 is a different (unquantized) product; reported as context only",
    }


def w8a16_comparator(torch, stream, sweep: Sweep, reps: int, ms_w8a8: float):
    """The weight-only layer on the same 448 layers: X_rot = X H in fp16
    (convrot_rotate, this library's kernel), then Y = X_rot W_deq^T with
    W_deq = Q_W * s_W dequantized to fp16 once, untimed (torch.mm -> cuBLAS).
    Dequantizing ahead of time makes this a lower bound for any W8A16 kernel
    (the pages' weight-only design decodes the weight on every call)."""
    cr = sweep.cr
    deq, rot = [], {}
    for L in sweep.layers:
        deq.append((L["Q_W"].float() * L["s_W"][:, None]).half())
        key = (L["M"], L["K"])
        if key not in rot:
            rot[key] = torch.empty((L["M"], L["K"]), dtype=torch.float16, device="cuda")

    def step():
        for L, W in zip(sweep.layers, deq):
            xr = rot[(L["M"], L["K"])]
            cr.convrot_rotate(L["X"], xr)
            torch.mm(xr, W.t(), out=L["Y"])

    g = graph_of(torch, stream, step)
    replay(torch, stream, g, 3)
    ms = time_graph(torch, stream, g, reps)
    del g, deq, rot
    return {
        "impl": "convrot_rotate (fp16 X H) + torch.mm fp16 (cuBLAS) with the weight "
                "dequantized to fp16 once, same 448 layers and X/Y buffers",
        "ms_per_step": round(ms, 4), "tops": round(sweep.ops / (ms * 1e-3) / 1e12, 2),
        "w8a8_speedup": round(ms / ms_w8a8, 3),
        "note": "weight-only (activations unquantized); dequantizing ahead of time makes "
                "it a lower bound for a W8A16 kernel; context only",
    }


E2E_STREAMS = 3


def run_e2e(args, sweep: Sweep, stream, dist: Dist):
    """The sweep through convrot_linear_host: every layer copies its X from
    pinned host memory and its Y back, with the layers dealt round-robin to
    E2E_STREAMS streams (a workspace and host output buffers each), so that
    one layer's copies overlap the others' kernels.  The step is captured once
    as a CUDA graph (the side streams fork from and join the timing stream)
    and timed on the host clock around replay + synchronize."""
    import torch
    cr = sweep.cr
    ns = E2E_STREAMS
    xs, ys = {}, {}
    for si in sweep.counts:
        L = sweep.first_layer_of(si)
        xs[si] = L["X"].cpu().pin_memory()
        for j in range(ns):
            ys[si, j] = torch.empty((L["M"], L["N"]), dtype=torch.float16).pin_memory()
    ws_bytes = max(cr.convrot_linear_host_workspace_bytes(L["M"], L["N"], L["K"], L["R"], True)
                   for L in sweep.layers)
    wss = [torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") for _ in range(ns)]
    streams = [torch.cuda.Stream() for _ in range(ns)]
    h2d = sum(2 * L["M"] * L["K"] for L in sweep.layers)
    d2h = sum(2 * L["M"] * L["N"] for L in sweep.layers)

    def issue():
        fork = torch.cuda.Event()
        fork.record(stream)
        for sj in streams:
            sj.wait_event(fork)
        for i, L in enumerate(sweep.layers):
            j = i % ns
            si = L["shape"]
            with torch.cuda.stream(streams[j]):
                cr.convrot_linear_host(xs[si], L["Q_W"], L["s_W"], ys[si, j], wss[j], W_img=L["img"],
                                       lora_down=L["down"], lora_up=L["up"],
                                       lora_scale=L["scale"])
        for sj in streams:
            join = torch.cuda.Event()
            join.record(sj)
            stream.wait_event(join)

    with torch.cuda.stream(stream):
        issue()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        issue()

    def step():
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()

    steps = max(3, min(args.steps, 20))
    for _ in range(3):
        step()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = dist.max((time.perf_counter() - t0) / steps)
    assert cr.convrot_check_device_error() == 0
    return {"value": round(dist.world * sweep.ops / dt / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(dt * 1e3, 3), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": f"convrot_linear_host (pinned host X and Y), layers dealt to {ns} streams, "
                   "one CUDA graph per step, host clock around replay + synchronize"}


# ----------------------------------------------------------------------------
# The oracle on the host cores (cpu_baseline and the reference arm).
# ----------------------------------------------------------------------------

class OracleSweep:
    """The oracle's per-call path on a row sample of each sweep shape."""

    def __init__(self, seed: int):
        import oracle
        self.oracle = oracle
        self.shapes = []
        for si, (N, K, count) in enumerate(workloads.SWEEP_SHAPES):
            W = workloads.make_w(N, K, seed * 1000 + si)
            prep = oracle.prepare_weight(W)  # one-time, untimed
            X = workloads.make_x(workloads.SWEEP_M, K, seed * 1000 + si)
            self.shapes.append((N, K, count, X, prep["Q_W"], prep["s_W"]))

    def run(self, rows: int) -> float:
        """Seconds for one call per shape on `rows` rows; returns the time."""
        t = 0.0
        import numpy as np
        for (N, K, count, X, Q_W, s_W) in self.shapes:
            sel = np.arange(rows)
            t0 = time.perf_counter()
            self.oracle.linear(X, Q_W, s_W, rows=sel, tie_bound=False)
            t += time.perf_counter() - t0
        return t

    def ops(self, rows: int) -> float:
        return float(sum(2 * rows * N * K for (N, K, *_rest) in self.shapes))

    def weighted_ops_and_time(self, rows: int):
        import numpy as np
        ops, t = 0.0, 0.0
        for (N, K, count, X, Q_W, s_W) in self.shapes:
            sel = np.arange(rows)
            t0 = time.perf_counter()
            self.oracle.linear(X, Q_W, s_W, rows=sel, tie_bound=False)
            dt = time.perf_counter() - t0
            ops += count * 2.0 * rows * N * K
            t += count * dt
        return ops, t


def cpu_baseline(args, budget_s: float):
    ors = OracleSweep(args.seed)
    threads = ors.oracle.threads_used()
    rows = args.cpu_rows
    if not rows:
        # Calibrate on one row per core, then size the sample to the budget.
        probe = max(1, threads)
        _, t = ors.weighted_ops_and_time(probe)
        rows = int(max(probe, min(workloads.SWEEP_M, probe * budget_s / max(t, 1e-6))))
        rows = max(probe, rows // probe * probe)
    ops, t = ors.weighted_ops_and_time(rows)
    return {"value": round(ops / t / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {rows} of 1024 rows of each of the 6 shapes, each shape's time "
                      f"weighted by its layer count (rows are independent); weight prep untimed",
            "seconds": round(t, 2)}


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return None
    ors = OracleSweep(args.seed)
    threads = ors.oracle.threads_used()
    # Each step: one pass over a row sample of all six shapes.  The sample has
    # at least one row per host core (the oracle parallelizes over rows), and
    # grows with the time the --steps/--warmup run may take (a few minutes).
    if args.cpu_rows:
        rows = args.cpu_rows
    else:
        t1 = ors.run(threads)  # one pass over the six shapes, one row per core
        per_step_budget = 120.0 / max(1, args.steps + args.warmup)
        rows = threads * int(max(1, min(workloads.SWEEP_M // threads,
                                        per_step_budget / max(t1, 1e-6))))
    for _ in range(args.warmup):
        ors.run(rows)
    w_ops, w_t, wall = 0.0, 0.0, 0.0
    for _ in range(args.steps):
        w0 = time.perf_counter()
        ops, t = ors.weighted_ops_and_time(rows)
        wall += time.perf_counter() - w0
        w_ops += ops
        w_t += t
    # The rate of the sweep's mix: each shape's time weighted by its layer count.
    value = w_ops / w_t / 1e12
    sample = (f"first {rows} of 1024 rows of each of the 6 shapes per step (one call per "
              "shape), the sweep's rate from each shape's time weighted by its layer count; "
              "weight prep untimed")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        # Time actually spent per step (one pass over the row sample of the six
        # shapes); the whole sweep's time at this rate is in its own key.
        "ms_per_step": round(wall / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8",
        "data": "synthetic (same recipe as the GPU arm, numpy generators)",
        "config": {"workload": WORKLOAD_TEXT["sweep"],
                   "layers": sum(c for (_, _, c) in workloads.SWEEP_SHAPES),
                   "parallelism": "host cores",
                   "rows_per_shape": rows},
        "sweep_ms_extrapolated": round(
            sum(2.0 * workloads.SWEEP_M * N * K * c for (N, K, c) in workloads.SWEEP_SHAPES)
            / (value * 1e12) * 1e3, 1),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _finite(o):
    """Replaces NaN/inf floats by None so the line is strict JSON."""
    if isinstance(o, float):
        return o if math.isfinite(o) else None
    if isinstance(o, dict):
        return {k: _finite(v) for k, v in o.items()}
    if isinstance(o, list):
        return [_finite(v) for v in o]
    return o


def main():
    args = parse_args()
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            res = run_reference(args, dist)
        else:
            res = run_ours(args, dist)
        if dist.rank == 0 and res is not None:
            print(json.dumps(_finite(res)), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
