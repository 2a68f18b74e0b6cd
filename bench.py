"""Benchmark: packed-weight GB/s of the M = 1 decode product on one GB300.

Workload (one step): the decode-time products of a Qwen3-0.6B-shaped stack
with MLX affine 4-bit, group-size-64 weights -- 28 layers of q_proj 2048x1024,
k_proj and v_proj 1024x1024, gate_proj and up_proj 3072x1024, down_proj
1024x3072, plus lm_head 151936x1024 -- 169 qm_apply calls on distinct
weights (302 MB packed, more than the 129 MB L2), each on its own synthetic
bf16 activation row. The step is captured once in a CUDA graph and replayed.

`value` is packed weight bytes per second over the timed steps (inputs
resident in HBM); `e2e` repeats the step with its activations copied in from
pinned host memory and every result copied back, inside the timed region.

--impl reference times the oracle (oracle/, plain C in float64) on the host
cores over a bounded sample of the same workload. Under torchrun (N > 1) each
rank runs an independent replica (the product does not shard here).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from packed_qmatmul_gb300 import synth  # noqa: E402

LAYERS = synth.QWEN3_0_6B_LAYERS
SHAPES = synth.QWEN3_0_6B_LAYER
LM_HEAD = synth.QWEN3_0_6B_LM_HEAD
METRIC = "packed-weight GB/s (M=1 GEMV)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill", "experts", "take"],
                    help="decode: the headline M=1 step; prefill: Q8_0 products at M >= 128; "
                         "experts: MXFP4 apply_experts; take: quantized embedding take + dequant")
    ap.add_argument("--T", type=int, default=None, help="experts: tokens (default 4096)")
    ap.add_argument("--bits", type=int, default=4)
    ap.add_argument("--M", type=int, default=None)
    ap.add_argument("--no-detail", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--unfused", action="store_true",
                    help="decode: one qm_apply per product (169 calls) instead of one qm_apply_many "
                         "per group of products that read the same activations (85 calls)")
    ap.add_argument("--only", default=None,
                    help="profiling aid: a step of just the projections whose name ends with this")
    return ap.parse_args()


def workload_list(bits):
    """[(name, n, k)] for one step, in call order."""
    out = []
    for layer in range(LAYERS):
        for name, (n, k) in SHAPES.items():
            out.append((f"layers.{layer}.{name}", n, k))
    out.append(("lm_head", *LM_HEAD))
    return out


def packed_bytes(n, k, bits, gs=64):
    return n * k * bits // 8 + 2 * n * (k // gs) * 2


def config_dict(bits, M, fused=True):
    calls = ("85 calls on distinct weights: per layer one qm_apply_many over q/k/v and one over gate/up "
             "(products that read the same activations share a launch) and qm_apply for down_proj; "
             "qm_apply for lm_head") if fused else "169 qm_apply calls on distinct weights"
    return {
        "workload": f"qwen3-0.6b-shaped decode step: 28 x (q 2048x1024, k/v 1024x1024, gate/up "
                    f"3072x1024, down 1024x3072) + lm_head 151936x1024, MLX affine {bits}-bit gs64, "
                    f"M={M}, {calls}",
        "format": "mlx_affine", "bits": bits, "group_size": 64, "M": M,
        "weight_bytes_per_step": sum(packed_bytes(n, k, bits) for _, n, k in workload_list(bits)),
        "l2": "inputs larger than L2 (distinct weights per layer, 302 MB at 4-bit)",
        "graph": "step captured once as a CUDA graph",
    }


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (clocks and throttle reasons)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
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
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def build_step(bits, M, device, only=None):
    import torch

    import packed_qmatmul_gb300 as qm

    g = synth.rng(1)
    items = []
    for name, n, k in workload_list(bits):
        if only and not name.endswith(only):
            continue
        w = synth.affine_weight(g, n, k, bits=bits, group_size=64)
        qw = qm.QWeight.from_arrays(w, device, flags=qm.QM_WEIGHT_STATIC)  # model weights do not change
        x = torch.from_numpy(synth.activations(g, M, k).view(np.int16)).to(device).view(torch.bfloat16)
        y = torch.empty((M, n), dtype=torch.bfloat16, device=device)
        items.append((name, n, k, qw, x, y))
    return items


FUSED_GROUPS = (("q_proj", "k_proj", "v_proj"), ("gate_proj", "up_proj"))


def step_groups(items, fused=True):
    """The step's calls in order: lists of items that read the same activations
    (q/k/v, gate/up of one layer) when fused, every other product alone."""
    groups, i = [], 0
    while i < len(items):
        g = [items[i]]
        for fg in FUSED_GROUPS if fused else ():
            if items[i][0].endswith(fg[0]):
                layer = items[i][0][:-len(fg[0])]
                for name in fg[1:]:
                    j = i + len(g)
                    if j < len(items) and items[j][0] == layer + name:
                        g.append(items[j])
        groups.append(g)
        i += len(g)
    return groups


def call_group(g, stream):
    """One call of the step: qm_apply for a lone product, qm_apply_many for a group
    (the group's first activations, which every member reads)."""
    import packed_qmatmul_gb300 as qm

    if len(g) == 1:
        qm.qm_apply(g[0][3], g[0][4], g[0][5], stream)
    else:
        qm.qm_apply_many([it[3] for it in g], g[0][4], [it[5] for it in g], stream)


def group_algo_bytes(g, bits, M):
    """Packed weights, the activations once, every output."""
    return sum(packed_bytes(n, k, bits) + 2 * M * n for _, n, k, *_ in g) + 2 * M * g[0][2]


def time_graph(step, stream, steps, warmup, clock_index=None):
    """Captures `step` once as a CUDA graph; returns (seconds for `steps`
    replays timed with CUDA events on `stream`, clock summary or None)."""
    import torch

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(clock_index) if clock_index is not None else None
    if clk:
        clk.__enter__()
        time.sleep(0.3)  # let the sampler start
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    if clk:
        clk.__exit__(None, None, None)
    return ev0.elapsed_time(ev1) / 1e3, (clk.summary() if clk else None)


PREFILL_METRIC = "TFLOP/s (M>=128 qmatmul)"


def prefill_items(M, dev, only=None):
    """GGUF Q8_0 weights 4096x4096, 14336x4096, 4096x14336 with x [M, k] and y [M, n]."""
    import torch

    import packed_qmatmul_gb300 as qm

    g = synth.rng(2)
    items = []
    for n, k in synth.Q8_0_SHAPES:
        if only and f"{n}x{k}" != only:
            continue
        qw = qm.QWeight.from_arrays(synth.q8_0_weight(g, n, k), dev)
        x = torch.from_numpy(synth.activations(g, M, k).view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
        items.append((n, k, qw, x, y))
    return items


def run_prefill(args, rank, world):
    """GGUF Q8_0 products 4096x4096, 14336x4096 and 4096x14336 at M tokens
    (2048 by default): one step = the three qm_apply calls, graph-captured."""
    import torch

    import packed_qmatmul_gb300 as qm
    from packed_qmatmul_gb300 import build as qbuild

    qbuild.build()
    qm.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    M = args.M or 2048
    items = prefill_items(M, dev, args.only)
    flops = sum(2.0 * M * n * k for n, k, *_ in items)
    wbytes = sum(n * (k // 32) * 34 for n, k, *_ in items)
    stream = torch.cuda.Stream()

    def step():
        for _, _, qw, x, y in items:
            qm.qm_apply(qw, x, y, stream)

    elapsed, clocks = time_graph(step, stream, args.steps, args.warmup, dev.index)
    qm.qm_device_status(stream)
    if world > 1:
        import torch.distributed as tdist
        t = torch.tensor([elapsed], device=dev)
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
        elapsed = float(t.item())
    tflops = flops * args.steps * world / elapsed / 1e12
    achieved = flops * args.steps / elapsed / 1e12
    peaks = load_peaks()
    peak = peaks.get("bf16_tflops", 1900.0)
    return {
        "metric": PREFILL_METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16xbf16->f32",
        "data": "synthetic (seeded)",
        "config": {"workload": f"GGUF Q8_0 qmatmul, W 4096x4096, 14336x4096, 4096x14336, M={M}"
                               + (f" (only {args.only})" if args.only else ""),
                   "M": M, "weight_bytes_per_step": wbytes, "flops_per_step": flops,
                   "l2": ("weights 143 MB per step, more than L2" if not args.only else
                          f"profiling aid: weights {wbytes / 1e6:.0f} MB per step, L2 not flushed")},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "gemm_kernel<Q8_0> (every launch of the step)",
                     "peak_source": "measured bf16 dense, burst" if "bf16_tflops" in peaks else "fallback"},
        "gpu_launches": len(items) * args.steps,
        "clocks": clocks,
    }


def _reduce_max(elapsed, dev, world):
    if world > 1:
        import torch
        import torch.distributed as tdist
        t = torch.tensor([elapsed], device=dev)
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
        return float(t.item())
    return elapsed


def _setup():
    import torch

    import packed_qmatmul_gb300 as qm
    from packed_qmatmul_gb300 import build as qbuild

    qbuild.build()
    qm.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    return dev


EXPERTS_SHAPE = (32, 5760, 2880)


def experts_step(T, dev):
    """One apply_experts call: 32 MXFP4 experts [5760, 2880], ids [T, 4]
    distinct per token and uniform over the experts, x [T, 2880]. Returns
    (step, flops, weight bytes of the experts the ids use, launches)."""
    import torch

    import packed_qmatmul_gb300 as qm

    w, ids, x = synth.moe_config(T)
    E, n, k = w["shape"]
    qw = qm.QWeight.from_arrays(w, dev)
    ids_d = torch.from_numpy(ids).to(dev)
    x_d = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((T, ids.shape[1], n), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(qm.qm_apply_experts_workspace(qw, T, ids.shape[1]), 256), dtype=torch.uint8,
                     device=dev)
    used = len(np.unique(ids))
    wbytes = used * (n * k // 2 + n * k // 32)
    flops = 2.0 * ids.size * n * k
    tensor = ids.size > 32 * E
    launches = 4 if tensor else 3  # route count + route scatter + (gather + grouped GEMM | grouped GEMV)

    def step(stream):
        qm.qm_apply_experts(qw, ids_d, x_d, y, ws, stream)

    return step, flops, wbytes, launches, tensor


EXPERTS_TFLOPS = "TFLOP/s (MXFP4 apply_experts)"
EXPERTS_GBS = "packed-weight GB/s (MXFP4 apply_experts, few tokens)"


def run_experts(args, rank, world):
    import torch

    import packed_qmatmul_gb300 as qm

    dev = _setup()
    T = args.T or 4096
    fn, flops, wbytes, launches, tensor = experts_step(T, dev)
    stream = torch.cuda.Stream()
    elapsed, clocks = time_graph(lambda: fn(stream), stream, args.steps, args.warmup, dev.index)
    qm.qm_device_status(stream)
    elapsed = _reduce_max(elapsed, dev, world)
    t_step = elapsed / args.steps
    peaks = load_peaks()
    if tensor:
        peak = peaks.get("bf16_tflops", 1900.0)
        value, unit, metric = flops * world / t_step / 1e12, "TFLOP/s", EXPERTS_TFLOPS
        roof = {"bound": "tensor", "achieved": round(flops / t_step / 1e12, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(flops / t_step / 1e12 / peak, 4), "traffic": traffic("experts_gemm", T == 4096)[0],
                "traffic_source": traffic("experts_gemm", T == 4096)[1],
                "kernel": "grouped gemm_kernel<MXFP4> with routing and gather in the step time",
                "peak_source": "measured bf16 dense, burst" if "bf16_tflops" in peaks else "fallback"}
    else:
        peak = peaks.get("hbm_gbs", 6800.0)
        value, unit, metric = wbytes * world / t_step / 1e9, "GB/s", EXPERTS_GBS
        roof = {"bound": "hbm", "achieved": round(wbytes / t_step / 1e9, 2), "peak": peak, "unit": "GB/s",
                "frac": round(wbytes / t_step / 1e9 / peak, 4), "traffic": traffic("experts_gemv", T == 64)[0],
                "traffic_source": traffic("experts_gemv", T == 64)[1],
                "kernel": "grouped gemv_kernel<MXFP4> with routing in the step time",
                "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"}
    return {
        "metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16xbf16->f32" if tensor else "f16xf16->f32",
        "data": "synthetic (seeded)",
        "config": {"workload": f"MXFP4 apply_experts, 32 experts [5760, 2880] (gate_up), T={T} tokens x top-4, "
                               "ids distinct per token, uniform", "T": T, "topk": 4,
                   "flops_per_step": flops, "weight_bytes_used": wbytes,
                   "l2": "expert weights 282 MB, more than L2", "graph": "step captured once as a CUDA graph"},
        "roofline": roof, "gpu_launches": launches * args.steps, "clocks": clocks,
    }


TAKE_METRIC = "GB/s (quantized embedding take + full dequant)"


def take_step(dev):
    """Affine 4-bit gs64 table 151936 x 1024: take of 4096 uniform ids into
    bf16 [4096, 1024], then dequant of the whole table to bf16. Returns
    (take fn, dequant fn, packed-take fn, bytes of each)."""
    import torch

    import packed_qmatmul_gb300 as qm

    g = synth.rng(5)
    n, k = LM_HEAD
    qw = qm.QWeight.from_arrays(synth.affine_weight(g, n, k, bits=4, group_size=64), dev)
    nid = 4096
    ids = torch.from_numpy(synth.uniform_ids(g, nid, n)).to(dev)
    dense = torch.empty((nid, k), dtype=torch.bfloat16, device=dev)
    table = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
    row = packed_bytes(1, k, 4)
    shapes = qw.part_shapes((nid,))
    outs = [None if sh is None else torch.empty(sh, dtype=torch.uint8, device=dev) for sh in shapes]
    take_bytes = nid * (row + 2 * k) + nid * 4
    deq_bytes = n * (row + 2 * k)
    ptake_bytes = 2 * nid * row + nid * 4

    def take(stream):
        qm.qm_take(qw, 0, ids, None, None, None, dense, stream)

    def deq(stream):
        qm.qm_dequant(qw, table, stream)

    def ptake(stream):
        qm.qm_take(qw, 0, ids, outs[0], outs[1], outs[2], None, stream)

    return take, deq, ptake, take_bytes, deq_bytes, ptake_bytes


def run_take(args, rank, world):
    import torch

    import packed_qmatmul_gb300 as qm

    dev = _setup()
    take, deq, ptake, tb, db, pb = take_step(dev)
    stream = torch.cuda.Stream()

    def step():
        take(stream)
        deq(stream)

    elapsed, clocks = time_graph(step, stream, args.steps, args.warmup, dev.index)
    t_deq, _ = time_graph(lambda: deq(stream), stream, args.steps, args.warmup)
    qm.qm_device_status(stream)
    elapsed = _reduce_max(elapsed, dev, world)
    t_step = elapsed / args.steps
    t_d = t_deq / args.steps
    peaks = load_peaks()
    peak = peaks.get("hbm_gbs", 6800.0)
    return {
        "metric": TAKE_METRIC, "value": round((tb + db) * world / t_step / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "dtype_note": "values decoded to f32, rounded once to bf16", "data": "synthetic (seeded)",
        "config": {"workload": "MLX affine 4-bit gs64 table 151936x1024: take of 4096 uniform ids to bf16 "
                               "[4096, 1024] + dequant of the whole table to bf16",
                   "bytes_per_step": tb + db, "take_bytes": tb, "dequant_bytes": db,
                   "l2": "the dequant writes 311 MB (more than L2) between takes",
                   "graph": "step captured once as a CUDA graph"},
        "roofline": {"bound": "hbm", "achieved": round(db / t_d / 1e9, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(db / t_d / 1e9 / peak, 4), "traffic": traffic("dequant")[0],
                     "traffic_source": traffic("dequant")[1],
                     "kernel": "decode_rows_kernel<affine,4> (the full dequant, timed alone)",
                     "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"},
        "gpu_launches": 2 * args.steps, "clocks": clocks,
    }


def chain_time(calls, stream, reps=10, warmup=3):
    """Seconds per call of a CUDA graph that runs `calls` (callables taking the
    stream) once each, in order, replayed `reps` times after `warmup`."""
    el, _ = time_graph(lambda: [c(stream) for c in calls], stream, reps, warmup)
    return el / (reps * len(calls))


def other_workloads(dev, stream):
    """The other configs' headline numbers, for the default run's detail. Each
    sub-L2 problem is timed as a graph chain over distinct weights, tables or
    outputs whose total exceeds twice the L2, so no call reads what an earlier
    one left in L2."""
    import torch

    import packed_qmatmul_gb300 as qm

    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    tc = peaks.get("bf16_tflops", 1900.0)
    out = {}
    # prefill: the TFLOP/s half of the metric (Q8_0, the three shapes per step)
    for M in (128, 2048):
        items = prefill_items(M, dev)
        flops = sum(2.0 * M * n * k for n, k, *_ in items)
        t = chain_time([lambda st, it=it: qm.qm_apply(it[2], it[3], it[4], st) for it in items], stream) * len(items)
        out[f"prefill_q8_0_M{M}"] = {"TFLOP/s": round(flops / t / 1e12, 1), "frac": round(flops / t / 1e12 / tc, 4),
                                     "ms_per_step": round(t * 1e3, 4),
                                     "shapes": "4096x4096, 14336x4096, 4096x14336"}
        del items
        torch.cuda.empty_cache()
    # Q8_0 14336 x 4096 at M = 1: five distinct weights (312 MB)
    g = synth.rng(6)
    n, k = 14336, 4096
    ws = [qm.QWeight.from_arrays(synth.q8_0_weight(g, n, k), dev, flags=qm.QM_WEIGHT_STATIC) for _ in range(5)]
    xs = [torch.from_numpy(synth.activations(g, 1, k).view(np.int16)).to(dev).view(torch.bfloat16) for _ in ws]
    ys = [torch.empty((1, n), dtype=torch.bfloat16, device=dev) for _ in ws]
    t = chain_time([lambda st, i=i: qm.qm_apply(ws[i], xs[i], ys[i], st) for i in range(len(ws))], stream, 20)
    b = n * (k // 32) * 34
    out["q8_0_14336x4096_M1"] = {"us": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1),
                                 "frac": round(b / t / 1e9 / hbm, 4)}
    del ws, xs, ys
    torch.cuda.empty_cache()
    # the embedding-table shape, 151936 x 1024 affine 4-bit gs64, four distinct
    # tables (350 MB): lm_head at M = 1, take of 4096 uniform ids, full dequant
    g = synth.rng(5)
    n, k = LM_HEAD
    tabs = [qm.QWeight.from_arrays(synth.affine_weight(g, n, k, bits=4, group_size=64), dev,
                                   flags=qm.QM_WEIGHT_STATIC) for _ in range(4)]
    row = packed_bytes(1, k, 4)
    xs = [torch.from_numpy(synth.activations(g, 1, k).view(np.int16)).to(dev).view(torch.bfloat16) for _ in tabs]
    ys = [torch.empty((1, n), dtype=torch.bfloat16, device=dev) for _ in tabs]
    t = chain_time([lambda st, i=i: qm.qm_apply(tabs[i], xs[i], ys[i], st) for i in range(4)], stream, 20)
    out["lm_head_M1"] = {"us": round(t * 1e6, 2), "GB/s": round(n * row / t / 1e9, 1),
                         "frac": round(n * row / t / 1e9 / hbm, 4)}
    del xs, ys
    nid, R = 4096, 64  # 64 takes of fresh ids into distinct outputs: 151 MB packed, 537 MB dense
    ids = [torch.from_numpy(synth.uniform_ids(g, nid, n)).to(dev) for _ in range(R)]
    shapes = tabs[0].part_shapes((nid,))
    pouts = [[None if sh is None else torch.empty(sh, dtype=torch.uint8, device=dev) for sh in shapes]
             for _ in range(R)]
    t = chain_time([lambda st, i=i: qm.qm_take(tabs[i % 4], 0, ids[i], pouts[i][0], pouts[i][1], pouts[i][2],
                                               None, st) for i in range(R)], stream)
    pb = 2 * nid * row + nid * 4
    out["take_packed_4096"] = {"us": round(t * 1e6, 2), "GB/s": round(pb / t / 1e9, 1),
                               "frac": round(pb / t / 1e9 / hbm, 4),
                               "bytes": "packed rows read and written once, plus the ids"}
    del pouts
    torch.cuda.empty_cache()
    douts = [torch.empty((nid, k), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    t = chain_time([lambda st, i=i: qm.qm_take(tabs[i % 4], 0, ids[i], None, None, None, douts[i], st)
                    for i in range(R)], stream)
    tb = nid * (row + 2 * k) + nid * 4
    out["take_dense_4096"] = {"us": round(t * 1e6, 2), "GB/s": round(tb / t / 1e9, 1),
                              "frac": round(tb / t / 1e9 / hbm, 4),
                              "bytes": "packed rows read, bf16 rows written, plus the ids"}
    del douts, ids
    table = torch.empty((n, k), dtype=torch.bfloat16, device=dev)  # 311 MB written per call: past L2
    t = chain_time([lambda st: qm.qm_dequant(tabs[0], table, st)], stream)
    db = n * (row + 2 * k)
    out["dequant_table"] = {"ms": round(t * 1e3, 4), "GB/s": round(db / t / 1e9, 1), "frac": round(db / t / 1e9 / hbm, 4)}
    del tabs, table
    torch.cuda.empty_cache()
    for T in (64, 1024, 4096):
        fn, flops, wbytes, _, tensor = experts_step(T, dev)
        el, _ = time_graph(lambda: fn(stream), stream, 10, 3)
        t = el / 10
        out[f"experts_T{T}"] = {"ms": round(t * 1e3, 4), "TFLOP/s": round(flops / t / 1e12, 1),
                                "weight GB/s": round(wbytes / t / 1e9, 1),
                                "path": "grouped tcgen05 GEMM" if tensor else "grouped GEMV"}
        del fn
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world):
    import torch

    import packed_qmatmul_gb300 as qm
    from packed_qmatmul_gb300 import build as qbuild

    qbuild.build()
    qm.load_library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    bits, M = args.bits, (args.M or 1)
    fused = not args.unfused
    items = build_step(bits, M, dev, args.only)
    groups = step_groups(items, fused)
    step_bytes = sum(packed_bytes(n, k, bits) for _, n, k, *_ in items)
    launches_per_step = len(groups)
    stream = torch.cuda.Stream()

    def step():
        for g in groups:
            call_group(g, stream)

    dist = world > 1
    if dist:
        import torch.distributed as tdist
        tdist.barrier()
    elapsed, clocks = time_graph(step, stream, args.steps, args.warmup, dev.index)
    qm.qm_device_status(stream)
    if dist:
        t = torch.tensor([elapsed], device=dev)
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
        elapsed = float(t.item())
        tdist.barrier()
    ms_per_step = elapsed / args.steps * 1e3
    value = step_bytes * args.steps * world / elapsed / 1e9
    # the dominant kernel: the one-token kernel of the layer projections (all
    # but lm_head), their launches captured and timed alone on the same stream
    layers = [g for g in groups if g[0][0] != "lm_head"] if M == 1 and not args.only else groups
    lay_algo = sum(group_algo_bytes(g, bits, M) for g in layers)

    def layer_step():
        for g in layers:
            call_group(g, stream)

    lay_el, _ = time_graph(layer_step, stream, args.steps, args.warmup)
    avg_launch = lay_el / (args.steps * len(layers))
    achieved = lay_algo / len(layers) / avg_launch / 1e9

    e2e = run_e2e(groups, stream, args, step_bytes)

    peaks = load_peaks()
    peak = peaks.get("hbm_gbs", 6800.0)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32",
        "dtype_note": "codes enter f16 tensor-core products as exact small integers, activations as exact "
                      "power-of-two rescaled f16; sums and scales at f32",
        "data": "synthetic (seeded; weights and activations drawn as the workload states)",
        "config": config_dict(bits, M, fused),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": traffic("decode", bits == 4 and M == 1 and not args.only and fused)[0],
                     "traffic_source": traffic("decode", bits == 4 and M == 1 and not args.only and fused)[1],
                     "algorithmic_bytes_per_launch": round(lay_algo / len(layers)),
                     "launch_us": round(avg_launch * 1e6, 3),
                     "kernel": (f"gemv1_kernel<affine,{bits}> (the {len(layers)} layer launches of the step"
                                + (", q/k/v and gate/up one grid each" if fused else "")
                                + ", timed alone as a graph of the same launches; lm_head runs gemv_kernel)")
                               if M == 1 and not args.only else f"the step's {len(layers)} product launches",
                     "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if args.only:
        res["config"]["workload"] += f" (profiling aid: only *{args.only})"
    if not args.no_detail and not args.only and rank == 0:
        res["detail"] = detail_measurements(args, dev, stream, fused)
        res["detail"].update(other_workloads(dev, stream))
        pf = res["detail"].get("prefill_q8_0_M2048")
        if pf:  # the metric's TFLOP/s half, on the Q8_0 prefill config
            res["tflops_m2048"] = {"metric": PREFILL_METRIC, "value": pf["TFLOP/s"], "unit": "TFLOP/s",
                                   "frac": pf["frac"], "peak_source": "measured bf16 dense, burst",
                                   "config": "GGUF Q8_0 W 4096x4096, 14336x4096, 4096x14336 at M=2048"}
    return res


def run_e2e(groups, stream, args, step_bytes):
    """Same step through the public API with host buffers: every call's
    activation rows copied in from pinned host memory as one transfer, the
    step's calls (no graph), every result copied back as one transfer, inside
    the timed region."""
    import torch

    gx = [g[0][4] for g in groups]  # each call's activations
    ys_all = [it[5] for g in groups for it in g]
    dev = gx[0].device
    y_sizes = [y.numel() for y in ys_all]
    hx = torch.cat([x.reshape(-1).cpu() for x in gx]).pin_memory()
    hy = torch.empty(sum(y_sizes), dtype=torch.bfloat16).pin_memory()
    dx = torch.empty_like(hx, device=dev)
    dy = torch.empty(sum(y_sizes), dtype=torch.bfloat16, device=dev)
    xs, ox = [], 0
    for x in gx:
        xs.append(dx[ox:ox + x.numel()].view(x.shape))
        ox += x.numel()
    ys, oy = [], 0
    for y in ys_all:
        ys.append(dy[oy:oy + y.numel()].view(y.shape))
        oy += y.numel()
    # the same calls on the staged buffers
    staged, yi = [], 0
    for g, x in zip(groups, xs):
        staged.append([(it[0], it[1], it[2], it[3], x, ys[yi + j]) for j, it in enumerate(g)])
        yi += len(g)
    h2d = hx.numel() * hx.element_size()
    d2h = hy.numel() * hy.element_size()

    def step():
        dx.copy_(hx, non_blocking=True)
        for g in staged:
            call_group(g, stream)
        hy.copy_(dy, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step()
    stream.synchronize()
    steps = max(1, min(args.steps, 20))
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(steps):
            step()
    stream.synchronize()
    el = time.perf_counter() - t0
    return {"value": round(step_bytes * steps / el / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": f"the step's {len(groups)} calls from Python (no graph); all activation rows H2D as one "
                    "copy before them and all results D2H as one copy after, pinned host memory"}


def detail_measurements(args, dev, stream, fused=True):
    """Secondary numbers (not the headline): 8-bit, M in {2, 4, 8}, and the
    4-bit M = 1 step the other way (one call per product, or grouped)."""
    import torch

    out = {}
    for bits, M, fz in ((8, 1, fused), (4, 2, fused), (4, 4, fused), (4, 8, fused), (4, 1, not fused)):
        items = build_step(bits, M, dev)
        groups = step_groups(items, fz)
        sb = sum(packed_bytes(n, k, bits) for _, n, k, *_ in items)

        def step():
            for g in groups:
                call_group(g, stream)

        reps = 20
        el, _ = time_graph(step, stream, reps, 3)
        key = f"affine{bits}_M{M}" + ("" if fz == fused else ("_grouped" if fz else "_one_call_per_product"))
        out[key] = {"GB/s": round(sb * reps / el / 1e9, 1), "ms_per_step": round(el / reps * 1e3, 4),
                    "calls_per_step": len(groups)}
        del items
        torch.cuda.empty_cache()
    return out


# DRAM bytes (read + write) per launch of each roofline kernel, from one ncu
# capture, with the commit whose kernel was measured. A kernel changed after its
# capture has None here (reported as null) until it is captured again.
TRAFFIC = {
    "decode": (2580267.0, "66cf0e5"),
    "experts_gemm": (539.0e6, "aa657a9"),
    "experts_gemv": (None, None),
    "dequant": (337.4e6, "6d4178e"),
}


def traffic(key, applies=True):
    if not applies or key not in TRAFFIC or TRAFFIC[key][0] is None:
        return None, None
    v, commit = TRAFFIC[key]
    return v, f"ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, kernel as of commit {commit}"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# ---------------------------------------------------------------- oracle (CPU)
def oracle_sample(bits):
    """One twenty-eighth of the step: one layer's six projections and 1/28 of
    lm_head's rows -- the same mix of shapes, so the same rate."""
    g = synth.rng(1)
    items = []
    for name, (n, k) in SHAPES.items():
        items.append((n, k, synth.affine_weight(g, n, k, bits=bits, group_size=64),
                      synth.activations(g, 1, k)))
    n, k = LM_HEAD
    nh = n // LAYERS
    items.append((nh, k, synth.affine_weight(g, nh, k, bits=bits, group_size=64),
                  synth.activations(g, 1, k)))
    return items


def time_oracle(bits, min_seconds=10.0, reps=None):
    import oracle

    items = oracle_sample(bits)
    ows = [(oracle.Weight(oracle.AFFINE, w["shape"], w["codes"], w["scales"], w["biases"], bits=bits,
                          group_size=64), x) for n, k, w, x in items]
    sb = sum(packed_bytes(n, k, bits) for n, k, _, _ in items)
    oracle.apply(*ows[0])  # build + page in
    done, t0 = 0, time.perf_counter()
    while True:
        for w, x in ows:
            oracle.apply(w, x)
        done += 1
        el = time.perf_counter() - t0
        if (reps is not None and done >= reps) or (reps is None and el >= min_seconds):
            break
    return sb * done / el / 1e9, el, done, oracle.num_threads()


def cpu_baseline(bits):
    v, el, reps, cores = time_oracle(bits, min_seconds=10.0)
    return {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"1/28 of the step (one layer's 6 projections + 5426 lm_head rows), "
                      f"repeated {reps}x in {el:.1f} s"}


def run_reference(args):
    import oracle

    oracle.build()
    bits = args.bits
    for _ in range(args.warmup):
        time_oracle(bits, reps=1)
    v, el, reps, cores = time_oracle(bits, reps=max(1, args.steps))
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / reps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_dict(bits, 1),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: 1/28 of the workload (one layer's six "
                                       "projections + 5426 lm_head rows)"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
    if args.workload in ("prefill", "experts", "take"):
        res = {"prefill": run_prefill, "experts": run_experts, "take": run_take}[args.workload](args, rank, world)
        if rank == 0:
            print(json.dumps(res))
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()
        return
    res = run_ours(args, rank, world)
    if rank == 0 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(args.bits)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
