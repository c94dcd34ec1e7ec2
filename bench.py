"""Benchmark of the W2A8 ternary GEMV path on GB300.

Workload: the M=1 GEMV sweep over the BitNet-2B decode shapes of the W2A8
kernel page (§7.1 table; §一 model shape) -- wqkv 3840x2560 (3 scale
segments), wo 2560x2560, w13 13824x2560 (2 segments), w2 2560x6912 --
with i.i.d. ternary weights (P(0) = 0.35), N(0,1) fp32 activation rows and
bf16 weight scales in [0.5, 2).

One step = one pass of the hot path over one batch of synthetic input:
  1. bw_quant_act on the step's 64 fp32 activation rows (48 of K=2560,
     16 of K=6912): per-row absmax to int8 + scale;
  2. 64 bw_gemv_w2a8 calls: R = 16 replicas x the 4 shapes, each replica a
     distinct weight buffer (278 MB in total, over twice the 126 MB L2, so
     every call streams its weights from HBM).
The quantisation and the 64 GEMVs (in decode-layer order, one chain of
programmatic dependent launches) are each captured once as a CUDA graph;
CUDA events between the two give the GEMV kernel's own time inside the
timed region.

value = packed weight bytes per step / step time (GB/s, all GPUs).
The reference arm (--impl reference) times the CPU oracle, its output rows
split over every host core, on a bounded sample of the same workload, in
the same unit.
Multi-GPU: replicas only (the path has no exchange step); each rank runs the
same workload on its own GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("W2A8 ternary GEMV µs/call & weight GB/s vs HBM peak (M=1); "
          "layer-stack tok/s")
WORKLOAD = ("M=1 W2A8 GEMV sweep over the BitNet-2B decode shapes: wqkv "
            "3840x2560, wo 2560x2560, w13 13824x2560, w2 2560x6912")
SHAPES = ["wqkv", "wo", "w13", "w2"]
REPLICAS = 16
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of the TMA GEMV kernel, measured with
# ncu (dram__bytes_read.sum + dram__bytes_write.sum, median of the captured
# launches of the bench's own sweep), with the SHA-256 of the kernel's
# source files at the time.  The bench reports them only while those files
# are unchanged, so a changed kernel reports null until it is re-measured.
TRAFFIC_SOURCES = ("bit_gemv_bitlinear_gb300/csrc/bw_pipe.cuh",
                   "bit_gemv_bitlinear_gb300/csrc/bw_gemv_tma.cu")
MEASURED_DRAM = {
    "sha256": "3c98a6960de8fbbe9072a9dc07d6e568f97d69fc9be013c5cd0f8eceb8620333",
    "bytes": {"wqkv": 2479232, "wo": 1659648, "w13": 8868736, "w2": 4449408}}


def traffic_sources_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic():
    """ncu DRAM bytes per GEMV launch (mean over the 4 shapes), or None if
    the kernel changed since they were taken."""
    if (not MEASURED_DRAM["bytes"]
            or MEASURED_DRAM["sha256"] != traffic_sources_sha()):
        return None
    b = MEASURED_DRAM["bytes"]
    return round(sum(b[n] for n in SHAPES) / len(SHAPES))


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--replicas", type=int, default=REPLICAS)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-stack", action="store_true",
                   help="skip the layer-stack tok/s measurement")
    p.add_argument("--no-batched", action="store_true",
                   help="skip the batched M = 4/16/64 timings")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the single-shape timings of the 2560x2560 "
                        "and large-shape configurations")
    p.add_argument("--no-attn", action="store_true",
                   help="skip the decode-attention timings")
    p.add_argument("--attn", action="store_true",
                   help="only time the decode attention (us/call, KV GB/s)")
    p.add_argument("--attn-contexts", default=None, metavar="L[,L...]",
                   help="--attn: context lengths (default 512,4096)")
    p.add_argument("--attn-rotate", type=int, default=0,
                   help="--attn: caches per graph (0: the read rows of "
                        "4x L2)")
    p.add_argument("--stack", action="store_true",
                   help="only time the 30-layer decode stack (tok/s)")
    p.add_argument("--stack-layers", type=int, default=None,
                   help="--stack: layers (default 30)")
    p.add_argument("--stack-steps", type=int, default=None,
                   help="--stack: decode steps per run (default 256)")
    p.add_argument("--stack-kv", type=int, default=0, metavar="S",
                   help="--stack: attend over a KV cache of S positions "
                        "(the steps are tokens 0.. of one sequence)")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="bounded CPU work for the oracle baseline")
    p.add_argument("--single", default=None, metavar="N,K[,M]",
                   help="time one GEMV shape alone over rotating weight "
                        "buffers (CUDA graph of back-to-back calls)")
    p.add_argument("--iters", type=int, default=2000)
    p.add_argument("--rotate", type=int, default=0,
                   help="--single: weight buffers (0: enough for 4x L2)")
    p.add_argument("--eager", action="store_true",
                   help="--single: launch eagerly instead of a CUDA graph")
    p.add_argument("--lut", action="store_true",
                   help="--single: time the pair-table (LUT) variant "
                        "bw_gemv_w2a8_lut instead of the dp4a GEMV")
    p.add_argument("--gemm", action="store_true",
                   help="--single: time the prefill call bw_gemm_w2a8 "
                        "(256-token tensor-core tiles)")
    p.add_argument("--no-lut", action="store_true",
                   help="skip the LUT-variant comparison")
    p.add_argument("--cold", action="store_true",
                   help="--single: isolated calls, L2 flushed before each "
                        "(median of --iters, at most 200), launch included")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def job_time_ms(torch, local_ms, world, device):
    """Whole-job time of a timed region that every rank entered after the
    same barrier: the maximum over ranks (an all-reduce; no-op at N=1)."""
    if world == 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(world, bytes_per_rank_step, ms_per_step):
    """Whole-job GB/s: every rank moves the same bytes per step (replicas),
    in the whole job's time per step."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def algorithmic_bytes(N, K, n_ws):
    """Packed weights + int8 x + bf16 y + fp32 s + bf16 ws of one call."""
    return N * K // 4 + K + 2 * N + 4 + 2 * n_ws


def weight_bytes(N, K):
    return N * K // 4


def read_all_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed
    region (200 ms period)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(),
                                 f"bw_bench_clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                smax.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def build_workload(torch, bw, dev, replicas, seed):
    """Weights (repacked, one buffer per replica), scales, activations."""
    shapes = {}
    for si, name in enumerate(SHAPES):
        N, K, bounds = synth.DECODE_SHAPES[name]
        canon = synth.canonical_weights(seed + si, N, K)
        canon_d = torch.from_numpy(canon).to(dev)
        packed0 = bw.bw_repack(canon_d, N, K)
        packed = [packed0] + [packed0.clone() for _ in range(replicas - 1)]
        ws = synth.bf16_uniform(seed + si, len(bounds) - 1)
        ws_d = torch.from_numpy(ws.view(np.int16)).to(dev).view(torch.bfloat16)
        shapes[name] = dict(N=N, K=K, bounds=bounds, canon=canon, ws=ws,
                            packed=packed, ws_d=ws_d)
    # Activation rows of one step: for every replica and shape, one N(0,1)
    # row of length K; grouped by K for the quantisation launches.
    rows = {}
    for name in SHAPES:
        K = shapes[name]["K"]
        rows.setdefault(K, []).append(name)
    # The fp32 rows of all K groups are views of one device buffer, and the
    # outputs of all calls views of another, so that a step's inputs and
    # results each move in one host<->device copy.
    act = {}
    total_in = sum(replicas * len(names) * K for K, names in rows.items())
    xf_all = torch.empty((total_in,), dtype=torch.float32, device=dev)
    off = 0
    for K, names in rows.items():
        count = replicas * len(names)
        xf = synth.normal_f32(seed + K, count * K).reshape(count, K)
        xf_d = xf_all[off:off + count * K].view(count, K)
        xf_d.copy_(torch.from_numpy(xf))
        off += count * K
        act[K] = dict(names=names, xf=xf, xf_d=xf_d,
                      q_d=torch.empty((count, K), dtype=torch.int8,
                                      device=dev),
                      s_d=torch.empty((count,), dtype=torch.float32,
                                      device=dev))
    act_all = xf_all
    total_out = replicas * sum(shapes[n]["N"] for n in SHAPES)
    out_all = torch.empty((total_out,), dtype=torch.bfloat16, device=dev)
    outs, off = {}, 0
    for name in SHAPES:
        N = shapes[name]["N"]
        outs[name] = []
        for _ in range(replicas):
            outs[name].append(out_all[off:off + N].view(1, N))
            off += N
    return shapes, act, outs, act_all, out_all


def act_row(act, shapes, name, r):
    """(q row view, s element view) of replica r of a shape."""
    K = shapes[name]["K"]
    a = act[K]
    idx = r * len(a["names"]) + a["names"].index(name)
    return a["q_d"][idx:idx + 1], a["s_d"][idx:idx + 1]


def check_sample(bw, shapes, act, outs):
    """Cheap parity check of the bench's own outputs: 64 sampled rows of
    replica 0 of every shape against the oracle."""
    import oracle
    for name in SHAPES:
        sh = shapes[name]
        N, K = sh["N"], sh["K"]
        q_d, s_d = act_row(act, shapes, name, 0)
        q = q_d.cpu().numpy()
        s = s_d.cpu().numpy()
        sel = (synth.u64(1, 77, 64) % np.uint64(N)).astype(np.int64)
        y = outs[name][0].view(__import__("torch").int16).cpu().numpy() \
            .view(np.uint16)[0]
        seg = np.searchsorted(np.asarray(sh["bounds"]), sel, side="right") - 1
        for i, n in enumerate(sel):
            ref = oracle.gemv(q, sh["canon"][n:n + 1], s,
                              sh["ws"][seg[i]:seg[i] + 1], [0, 1], 1, K)[0, 0]
            g = synth.bf16_bits_to_f32(np.array([y[n]], np.uint16))[0]
            r_ = synth.bf16_bits_to_f32(np.array([ref], np.uint16))[0]
            ulp = 2.0 ** (np.floor(np.log2(max(abs(r_), 1e-38))) - 7)
            if abs(float(g) - float(r_)) > ulp:
                raise AssertionError(f"bench output mismatch {name} row {n}")
    return True


def run_ours(args):
    import torch
    import bit_gemv_bitlinear_gb300 as bw

    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    R = args.replicas
    seed = synth.base_seed(1)
    shapes, act, outs, act_all, out_all = build_workload(torch, bw, dev, R,
                                                         seed)
    stream = torch.cuda.Stream(device=dev)

    def launch_quant():
        for K, a in act.items():
            bw.bw_quant_act(a["xf_d"], a["q_d"], a["s_d"], stream=stream)

    def launch_shape(name):
        sh = shapes[name]
        for r in range(R):
            q_d, s_d = act_row(act, shapes, name, r)
            bw.bw_gemv_w2a8(q_d, sh["packed"][r], s_d, sh["ws_d"],
                            sh["bounds"], sh["N"], sh["K"], y=outs[name][r],
                            stream=stream)

    def launch_gemvs():
        """The 64 GEMVs in decode-layer order: replica by replica, wqkv, wo,
        w13, w2 -- one programmatic-dependent-launch chain."""
        for r in range(R):
            for name in SHAPES:
                sh = shapes[name]
                q_d, s_d = act_row(act, shapes, name, r)
                bw.bw_gemv_w2a8(q_d, sh["packed"][r], s_d, sh["ws_d"],
                                sh["bounds"], sh["N"], sh["K"],
                                y=outs[name][r], stream=stream)

    # Capture the two parts of a step as CUDA graphs (after an eager warm-up).
    with torch.cuda.stream(stream):
        launch_quant()
        launch_gemvs()
    stream.synchronize()
    graphs = {}
    parts = ["quant", "gemv"]
    for part in parts:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if part == "quant":
                launch_quant()
            else:
                launch_gemvs()
        graphs[part] = g
    torch.cuda.synchronize()

    def step(evs=None):
        with torch.cuda.stream(stream):
            if evs is not None:
                evs[0].record(stream)
            for i, part in enumerate(parts):
                graphs[part].replay()
                if evs is not None:
                    evs[i + 1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    check_sample(bw, shapes, act, outs)

    K_steps = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)]
           for _ in range(K_steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    start.record(stream)
    for k in range(K_steps):
        step(evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    bw.bw_device_error(stream)   # raises if a bounded device wait ran out
    total_ms = start.elapsed_time(end)
    part_ms = {p: 0.0 for p in parts}
    for k in range(K_steps):
        for i, p in enumerate(parts):
            part_ms[p] += evs[k][i].elapsed_time(evs[k][i + 1])
    total_ms = job_time_ms(torch, total_ms, world, dev)

    wbytes_step = R * sum(weight_bytes(shapes[n]["N"], shapes[n]["K"])
                          for n in SHAPES)
    ms_per_step = total_ms / K_steps
    value = job_value(world, wbytes_step, ms_per_step)

    # The GEMV kernel's own time: the events around the GEMV graph of every
    # timed step.
    alg_total = K_steps * R * sum(
        algorithmic_bytes(shapes[n]["N"], shapes[n]["K"],
                          len(shapes[n]["bounds"]) - 1) for n in SHAPES)
    gemv_ms = part_ms["gemv"]
    peak, peak_kind = read_peaks()
    achieved = alg_total / (gemv_ms * 1e-3) / 1e9
    per_call = per_shape_times(torch, bw, shapes, act, outs, R, stream,
                               reps=max(1, min(50, K_steps)))
    gemv_launches = len(SHAPES) * R
    quant_launches = len(act)

    # End to end: the same step with host buffers -- one pinned H2D of the
    # step's fp32 activation rows, the step, one D2H of all its outputs.
    host_in = act_all.cpu().pin_memory()
    host_out = torch.empty_like(out_all, device="cpu").pin_memory()
    h2d = host_in.numel() * 4
    d2h = host_out.numel() * 2

    def e2e_step():
        with torch.cuda.stream(stream):
            act_all.copy_(host_in, non_blocking=True)
            for part in parts:
                graphs[part].replay()
            host_out.copy_(out_all, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(K_steps):
        e2e_step()
    e_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = job_time_ms(torch, e_start.elapsed_time(e_end), world, dev) / K_steps
    e2e_value = job_value(world, wbytes_step, e2e_ms)

    lut_line = None
    if rank == 0 and not args.no_lut:
        lut_line = run_lut_comparison(torch, bw, dev)
    configs_line = None
    if rank == 0 and not args.no_configs:
        configs_line = run_config_shapes(torch, bw, dev, peak)

    stack_line = stack_kv_line = None
    if not args.no_stack:
        stack_line = run_stack_timing(torch, bw, dev)
        stack_kv_line = run_stack_timing(torch, bw, dev,
                                         kv_positions=ATTN_S)
    batched_line = prefill_line = None
    if rank == 0 and not args.no_batched:
        batched_line = run_batched(torch, bw, dev, peak)
        prefill_line = run_prefill(torch, bw, dev, read_all_peaks())
    attn_line = None
    if rank == 0 and not args.no_attn:
        attn_line = run_attn_timing(torch, bw, dev, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(shapes, act, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": K_steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int8",
            "data": "synthetic",
            "config": {
                "workload": WORKLOAD,
                "replicas": R,
                "gemv_calls_per_step": gemv_launches,
                "weight_bytes_per_step": wbytes_step,
                "l2": "inputs larger than L2: 16 distinct weight buffers "
                      "per shape, 278 MB per step vs 126 MB L2",
                "graphs": "per step: one graph of the quantisation launches, "
                          "one graph of the 64 GEMV launches",
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "per_call": per_call,
            "roofline": {
                "bound": "hbm",
                "kernel": "gemv_w2a8_pipe_kernel",
                "achieved": round(achieved, 1),
                "peak": peak,
                "peak_kind": peak_kind,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": measured_traffic(),
                "traffic_unit": "bytes per GEMV launch (ncu)",
                "alg_bytes_per_launch": round(alg_total / (K_steps * R
                                                           * len(SHAPES))),
            },
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 5)},
            "gpu_launches": (gemv_launches + quant_launches) * K_steps,
            "clocks": clocks,
        }
        if configs_line is not None:
            line["configs"] = configs_line
        if lut_line is not None:
            line["lut_variant"] = lut_line
        if stack_line is not None:
            line["layer_stack"] = stack_line
        if stack_kv_line is not None:
            line["layer_stack_kv"] = stack_kv_line
        if batched_line is not None:
            line["batched"] = batched_line
        if prefill_line is not None:
            line["prefill"] = prefill_line
        if attn_line is not None:
            line["attn_decode"] = attn_line
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


STACK_LAYERS, STACK_STEPS = 30, 256


def run_stack_timing(torch, bw, dev, n_layers=STACK_LAYERS,
                     steps=STACK_STEPS, reps=3, kv_positions=0):
    """The BitNet-2B-shaped decode layer stack (dim 2560, ffn 6912, 20/5
    heads): `steps` decode steps through `n_layers` layers.  One layer's
    random ternary weights are generated and copied into n_layers distinct
    device buffers (521 MB for 30 layers, so every step streams all weights
    from HBM).  kv_positions = 0: independent steps with the one-token
    attention; > 0: a stack with a KV cache of that many positions, the
    steps being tokens 0 .. steps - 1 of one sequence (the cache reset
    before every timed run).  Returns tok/s and the derived figures."""
    dim, ffn, nh, nkv = 2560, 6912, 20, 5
    seed = synth.base_seed(4)
    w = synth.stack_weights(seed, 1, dim, ffn, nh, nkv)
    L0 = w["layers"][0]
    base = {}
    for name in ("wqkv", "wo", "w13", "w2"):
        canon = L0[name]
        base[name] = bw.bw_repack(torch.from_numpy(canon).to(dev),
                                  canon.shape[0], canon.shape[1] * 4)
    ws = torch.from_numpy(L0["ws"].view(np.int16)).to(dev).view(torch.bfloat16)
    gam = torch.from_numpy(L0["gammas"]).to(dev)
    layers = [{k: (v if i == 0 else v.clone()) for k, v in base.items()}
              | {"ws": ws, "gammas": gam} for i in range(n_layers)]
    stack = bw.Stack(layers, dim, ffn, nh, nkv, w["eps"],
                     max_positions=kv_positions, theta=ATTN_THETA)
    h_in = torch.from_numpy(synth.step_inputs(seed, steps, dim)).to(dev)
    h_out = torch.empty_like(h_in)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        stack.run(h_in[:4], h_out[:4], stream=stream)
    stream.synchronize()
    best = None
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            if kv_positions:
                stack.reset_kv(stream=stream)
            e0.record(stream)
            stack.run(h_in, h_out, stream=stream)
            e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    bw.bw_device_error(stream)
    stack.close()
    layer_bytes = sum(int(base[k].numel()) for k in base)
    us_tok = best * 1e3 / steps
    res = {"layers": n_layers, "steps": steps,
           "tok_s": round(steps / (best * 1e-3), 1),
           "us_per_token": round(us_tok, 2),
           "weight_bytes_per_token": layer_bytes * n_layers,
           "weight_GBps": round(layer_bytes * n_layers / (us_tok * 1e3), 1),
           "timing": f"best of {reps} runs of {steps} steps, CUDA events"}
    if kv_positions:
        res["launches_per_token"] = 5 * n_layers
        res["execution"] = ("one launch per GEMV and one per attention, each "
                            "step replayed from a CUDA graph")
    else:
        res["launches_per_call"] = 1
        res["execution"] = ("one persistent cooperative kernel per call "
                            f"({steps} steps x {n_layers} layers x 4 GEMVs)")
    if kv_positions:
        res["attention"] = (f"KV cache of {kv_positions} positions; tokens "
                            f"0..{steps - 1} of one sequence per run")
    else:
        res["attention"] = "one-token context (independent steps)"
    return res


def per_shape_times(torch, bw, shapes, act, outs, R, stream, reps=50):
    """Informational, after the timed region: µs per call of each shape,
    from a graph of its R calls back to back."""
    res = {}
    for name in SHAPES:
        sh = shapes[name]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(R):
                q_d, s_d = act_row(act, shapes, name, r)
                bw.bw_gemv_w2a8(q_d, sh["packed"][r], s_d, sh["ws_d"],
                                sh["bounds"], sh["N"], sh["K"],
                                y=outs[name][r], stream=stream)
        with torch.cuda.stream(stream):
            g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * R)
        ab = algorithmic_bytes(sh["N"], sh["K"], len(sh["bounds"]) - 1)
        res[name] = {"N": sh["N"], "K": sh["K"], "us_per_call": round(us, 3),
                     "weight_GBps": round(weight_bytes(sh["N"], sh["K"])
                                          / (us * 1e3), 1),
                     "alg_GBps": round(ab / (us * 1e3), 1)}
    return res


def oracle_gemv_threads(oracle, q, canon, s, ws, bounds, N, K, threads):
    """The oracle's GEMV over `threads` contiguous slices of output rows, run
    on a thread pool: each slice is one call of the unmodified oracle (its C
    code releases the GIL), with the weight-scale segments cut to the slice.
    Rows are independent, so the result equals one call over all rows."""
    import concurrent.futures as cf
    cuts = [N * i // threads for i in range(threads + 1)]
    bounds = np.asarray(bounds)

    def part(i):
        lo, hi = cuts[i], cuts[i + 1]
        if hi <= lo:
            return np.empty((q.shape[0] if q.ndim == 2 else 1, 0), np.uint16)
        seg_lo = int(np.searchsorted(bounds, lo, side="right") - 1)
        seg_hi = int(np.searchsorted(bounds, hi - 1, side="right") - 1)
        b = [lo] + [int(v) for v in bounds[seg_lo + 1:seg_hi + 1]] + [hi]
        b = [v - lo for v in b]
        return oracle.gemv(q, canon[lo:hi], s, ws[seg_lo:seg_hi + 1], b,
                           hi - lo, K)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return np.concatenate(list(ex.map(part, range(threads))), axis=1)


def oracle_step(oracle, shapes, act, threads):
    """One replica's step through the oracle: the quantisation of its rows,
    then the 4 decode-shape GEMVs; returns the packed weight bytes."""
    wb = 0
    for K, a in act.items():
        oracle.quant_act(a["xf"][: len(a["names"])])
    for name in SHAPES:
        sh = shapes[name]
        K = sh["K"]
        a = act[K]
        q, s = oracle.quant_act(a["xf"][a["names"].index(name)])
        if threads == 1:
            oracle.gemv(q, sh["canon"], s, sh["ws"], sh["bounds"], sh["N"], K)
        else:
            oracle_gemv_threads(oracle, q, sh["canon"], s, sh["ws"],
                                sh["bounds"], sh["N"], K, threads)
        wb += weight_bytes(sh["N"], K)
    return wb


def oracle_stack_token(oracle, seconds):
    """The oracle's decoder layers at the BitNet-2B shape (dim 2560, ffn 6912,
    20/5 heads, one-token attention, the bench stack's seeded weights): one
    token through as many of the 30 layers as a bounded time allows, one
    core; returns tok/s for the 30-layer stack."""
    dim, ffn, nh, nkv = 2560, 6912, 20, 5
    seed = synth.base_seed(4)
    w = synth.stack_weights(seed, 1, dim, ffn, nh, nkv)
    L0 = w["layers"][0]
    h = synth.step_inputs(seed, 1, dim)[0]
    t0 = time.perf_counter()
    layers = 0
    while layers < STACK_LAYERS:
        h = oracle.layer(h, dim, ffn, nh, nkv, w["eps"], L0["wqkv"], L0["wo"],
                         L0["w13"], L0["w2"], L0["ws"], L0["gammas"])
        layers += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"tok_s": round(layers / (dt * STACK_LAYERS), 4), "cores": 1,
            "sample": f"{layers} layer(s) of one token in {dt:.1f} s on one "
                      f"thread, scaled to {STACK_LAYERS} layers"}


def cpu_baseline(shapes, act, seconds):
    """The oracle as it stands on whole steps of the workload restricted to
    one replica, repeated for a bounded time: on every host core (output
    rows split over a thread pool), and on one core.  Beside it, the oracle's
    decoder layers in tok/s."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    res = {}
    for threads in (cores, 1):
        t0 = time.perf_counter()
        reps, wbytes = 0, 0
        while True:
            wbytes += oracle_step(oracle, shapes, act, threads)
            reps += 1
            if time.perf_counter() - t0 >= seconds / 2:
                break
        dt = time.perf_counter() - t0
        res[threads] = (wbytes / dt / 1e9, reps, dt)
    v, reps, dt = res[cores]
    v1, reps1, dt1 = res[1]
    return {"value": round(v, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} pass(es) of quant + the 4 decode-shape GEMVs "
                      f"(one replica), {dt:.1f} s, output rows split over "
                      f"{cores} threads",
            "single_core": {"value": round(v1, 4), "unit": "GB/s",
                            "cores": 1,
                            "sample": f"{reps1} pass(es), {dt1:.1f} s on one "
                                      f"thread"},
            "layer_stack": oracle_stack_token(oracle, seconds / 2)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch  # noqa: F401  (only for the shared generators' dtype use)
    seed = synth.base_seed(1)
    shapes, act = {}, {}
    for si, name in enumerate(SHAPES):
        N, K, bounds = synth.DECODE_SHAPES[name]
        shapes[name] = dict(N=N, K=K, bounds=bounds,
                            canon=synth.canonical_weights(seed + si, N, K),
                            ws=synth.bf16_uniform(seed + si, len(bounds) - 1))
    for name in SHAPES:
        K = shapes[name]["K"]
        act.setdefault(K, {"names": []})["names"].append(name)
    for K, a in act.items():
        count = len(a["names"])
        a["xf"] = synth.normal_f32(seed + K, count * K).reshape(count, K)

    import oracle
    oracle.build()

    cores = os.cpu_count() or 1

    def one_step():
        return oracle_step(oracle, shapes, act, cores)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    wb = 0
    for _ in range(args.steps):
        wb += one_step()
    dt = time.perf_counter() - t0
    value = wb / dt / 1e9
    sample = (f"each step: quant + the 4 decode-shape GEMVs of one replica "
              f"(1/{REPLICAS} of a GPU step); {args.steps} steps in "
              f"{dt:.1f} s, output rows split over {cores} host threads")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "replicas": 1,
                   "implementation": "CPU oracle (plain C; output rows "
                                     f"split over {cores} threads)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                         "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_shape(torch, bw, dev, N, K, M, iters=2000, rotate=0, eager=False,
               lut=False, gemm=False):
    """Microseconds per bw_gemv_w2a8 call of one shape (bw_gemv_w2a8_lut
    with `lut`, the prefill call bw_gemm_w2a8 with `gemm`), back to back on
    one stream (a CUDA graph of up to 64 calls unless `eager`), cycling
    through enough copies of the weights that they exceed L2 (weights,
    tokens and scales are seeded synthetic data)."""
    seed = synth.base_seed(2, 1)
    canon = synth.canonical_weights(seed, N, K)
    packed0 = bw.bw_repack(torch.from_numpy(canon).to(dev), N, K)
    wb = weight_bytes(N, K)
    rot = rotate or max(2, -(-4 * 126 * 2**20 // wb))
    rot = min(rot, max(2, (8 << 30) // max(wb, 1)))
    packed = [packed0] + [packed0.clone() for _ in range(rot - 1)]
    xf = torch.from_numpy(synth.normal_f32(seed, M * K).reshape(M, K)).to(dev)
    q, s_ = bw.bw_quant_act(xf)
    ws = torch.ones(1, device=dev).to(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    per_graph = max(rot, min(iters, 64))
    gemv = bw.bw_gemv_w2a8_lut if lut else bw.bw_gemv_w2a8
    work = (torch.empty((bw.bw_gemm_workspace_bytes(M, K),),
                        dtype=torch.uint8, device=dev) if gemm else None)

    def launches():
        for i in range(per_graph):
            if gemm:
                bw.bw_gemm_w2a8(q, packed[i % rot], s_, ws, [0, N], N, K, y=y,
                                workspace=work, stream=stream)
            else:
                gemv(q, packed[i % rot], s_, ws, [0, N], N, K, y=y,
                     stream=stream)

    with torch.cuda.stream(stream):
        launches()
    stream.synchronize()
    if eager:
        def run():
            with torch.cuda.stream(stream):
                launches()
    else:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launches()

        def run():
            with torch.cuda.stream(stream):
                g.replay()
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    reps = max(1, iters // per_graph)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(reps):
        run()
    end.record(stream)
    torch.cuda.synchronize()
    bw.bw_device_error(stream)
    us = start.elapsed_time(end) * 1e3 / (reps * per_graph)
    ab = algorithmic_bytes(N, K, 1) + (M - 1) * (K + 2 * N + 4)
    return {"us": us, "rotate": rot, "calls": reps * per_graph,
            "weight_bytes": wb, "alg_bytes": ab}


# The single-call configurations: one 2560 x 2560 GEMV with one weight scale,
# and the large M = 1 shapes whose weights (70.8 and 17.7 MB) far exceed L2.
CONFIG_SHAPES = (("single_2560x2560", 2560, 2560),
                 ("large_55296x5120", 55296, 5120),
                 ("large_13824x5120", 13824, 5120))


def run_config_shapes(torch, bw, dev, peak_gbs):
    """us per call of each single-call configuration, back to back in a CUDA
    graph over rotating weight buffers (their total over 4x L2), with the
    weight GB/s and the fraction of the measured HBM copy peak on the
    algorithmic bytes (weights + x + y + scales)."""
    out = {"timing": "graph of calls back to back over rotating weight "
                     "buffers (over 4x L2), CUDA events",
           "kernel": "gemv_w2a8_pipe_kernel"}
    for name, N, K in CONFIG_SHAPES:
        t = time_shape(torch, bw, dev, N, K, 1, iters=1024)
        us = t["us"]
        out[name] = {"N": N, "K": K, "us_per_call": round(us, 3),
                     "weight_GBps": round(t["weight_bytes"] / (us * 1e3), 1),
                     "alg_GBps": round(t["alg_bytes"] / (us * 1e3), 1),
                     "hbm_frac": round(t["alg_bytes"] / (us * 1e3) / peak_gbs,
                                       4),
                     "weight_buffers": t["rotate"]}
    return out


# The pair-table (LUT) variant against the dp4a decode, same kernel template.
LUT_CASES = ((1, 2560, 2560), (1, 13824, 2560), (4, 13824, 2560))


def run_lut_comparison(torch, bw, dev):
    """us per call of bw_gemv_w2a8_lut and bw_gemv_w2a8 at M = 1 and 4 (graph
    of calls over rotating weight buffers), and their ratio."""
    out = {"timing": "graph of calls back to back over rotating weight "
                     "buffers (over 4x L2), CUDA events", "cases": {}}
    for M, N, K in LUT_CASES:
        d = time_shape(torch, bw, dev, N, K, M, iters=1024)
        lt = time_shape(torch, bw, dev, N, K, M, iters=1024, lut=True)
        out["cases"][f"M{M}_{N}x{K}"] = {
            "dp4a_us": round(d["us"], 3), "lut_us": round(lt["us"], 3),
            "lut_over_dp4a": round(lt["us"] / d["us"], 3)}
    return out


BATCHED_N, BATCHED_K, BATCHED_M = 13824, 2560, (4, 16, 64)
PREFILL_M = (256, 512, 1024, 2048)


def run_prefill(torch, bw, dev, peaks):
    """Prompt-sized W2A8 GEMMs (the W2A8 page's §一 prefill) at 13824 x 2560
    through bw_gemm_w2a8 (the token conversion plus 256-token tcgen05 tiles):
    us per call (graph of calls over rotating weight buffers) and TFLOP/s
    (2 M N K per call) against the measured dense bf16 rate -- the path runs
    kind::f16 MMAs, whose nominal rate equals bf16's.  Beside it, the same
    product through bw_gemv_w2a8's 128-token tiles."""
    out = {"shape": [BATCHED_N, BATCHED_K],
           "kernel": "tok_fp16_kernel + gemm_kernel (tcgen05, 128 weight "
                     "rows x 256 tokens per CTA)",
           "per_m": {}}
    for M in PREFILL_M:
        t = time_shape(torch, bw, dev, BATCHED_N, BATCHED_K, M,
                       iters=max(8, 8192 // M), gemm=True)
        t128 = time_shape(torch, bw, dev, BATCHED_N, BATCHED_K, M,
                          iters=max(8, 8192 // M))
        us = t["us"]
        tflops = 2.0 * M * BATCHED_N * BATCHED_K / (us * 1e-6) / 1e12
        out["per_m"][str(M)] = {
            "us_per_call": round(us, 2), "tflops": round(tflops, 1),
            "frac_of_measured_bf16_sustained":
                round(tflops / peaks["bf16_tflops_sustained"], 4)
                if peaks.get("bf16_tflops_sustained") else None,
            "frac_of_nominal_dense_fp16": round(tflops / 2250.0, 4),
            "gemv_128_token_tiles_us": round(t128["us"], 2)}
    return out


def run_batched(torch, bw, dev, peak_gbs):
    """The batched known-token GEMM (M = 4, 16, 64 at 13824 x 2560): us per
    call, weight GB/s, and the fractions of the measured HBM copy peak and
    of the nominal dense fp16 tensor rate (2.25 PFLOP/s) the call reaches."""
    out = {"shape": [BATCHED_N, BATCHED_K], "per_m": {}}
    for M in BATCHED_M:
        t = time_shape(torch, bw, dev, BATCHED_N, BATCHED_K, M, iters=1024)
        us = t["us"]
        flops = 2.0 * M * BATCHED_N * BATCHED_K
        out["per_m"][str(M)] = {
            "us_per_call": round(us, 3),
            "kernel": "tc_gemv_kernel (tcgen05)" if M >= 8
                      else "gemv_w2a8_pipe_kernel (dp4a)",
            "weight_GBps": round(t["weight_bytes"] / (us * 1e3), 1),
            "hbm_frac": round(t["alg_bytes"] / (us * 1e3) / peak_gbs, 4),
            "tensor_frac_nominal": round(flops / (us * 1e-6) / 2.25e15, 4),
        }
    return out


ATTN_H, ATTN_HKV, ATTN_D, ATTN_S = 20, 5, 128, 4096
ATTN_CONTEXTS = (512, 4096)
ATTN_THETA = 500000.0


def run_attn_timing(torch, bw, dev, peak_gbs, contexts=ATTN_CONTEXTS,
                    iters=1024, rotate=0):
    """bw_attn_decode at the BitNet-2B attention shape (20 query heads over
    5 KV heads of 128, a 4096-position bf16 cache) for contexts of L tokens
    (the new token at position L - 1): us per call in a graph of calls back
    to back, each on its own cache so that the keys and values it reads
    (2 Hkv L D bf16 = 2560 L bytes) come from HBM.  One cache of seeded
    synthetic N(0,1) values is generated and copied.  Timed twice: as
    bw_attn_decode (every input read after the preceding call) and with
    BW_ATTN_PAST_READY (the position and the rows before it read and copied
    before the dependency wait, which this chain allows: no call writes the
    position or another call's cache), as the KV stack runs it."""
    H, Hkv, D, S = ATTN_H, ATTN_HKV, ATTN_D, ATTN_S
    seed = synth.base_seed(5)
    case = synth.attn_case(seed, H, Hkv, D, S, 0)

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)) \
            .to(dev).view(torch.bfloat16)

    qkv = dev_bf16(case["qkv"])
    kc0, vc0 = dev_bf16(case["kc"]), dev_bf16(case["vc"])
    ws = torch.zeros((bw.bw_attn_workspace_bytes(H, Hkv, D, S),),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((H, D), dtype=torch.float32, device=dev)
    res = {"heads": H, "kv_heads": Hkv, "head_dim": D, "cache_positions": S,
           "theta": ATTN_THETA,
           "kernel": "attn_cluster_kernel (one cluster of up to 16 CTAs per "
                     "KV head, merge in distributed shared memory)",
           "timing": "graph of calls back to back, one cache per call, "
                     "the caches' read rows over 4x L2",
           "contexts": {}}
    stream = torch.cuda.Stream(device=dev)
    for L in contexts:
        kv_bytes = 2 * Hkv * L * D * 2
        rot = rotate or max(2, -(-4 * 126 * 2**20 // kv_bytes))
        kcs = kc0.unsqueeze(0).repeat(rot, 1, 1, 1)
        vcs = vc0.unsqueeze(0).repeat(rot, 1, 1, 1)
        pos = torch.tensor([L - 1], dtype=torch.int32, device=dev)
        times = {}
        for flags in (0, bw.BW_ATTN_PAST_READY):
            def launches():
                for i in range(rot):
                    bw.bw_attn_decode_ex(qkv, pos, H, Hkv, kcs[i], vcs[i],
                                         theta=ATTN_THETA, out=out,
                                         workspace=ws, flags=flags,
                                         stream=stream)

            with torch.cuda.stream(stream):
                launches()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                launches()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
            torch.cuda.synchronize()
            reps = max(1, iters // rot)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            bw.bw_device_error(stream)
            times[flags] = e0.elapsed_time(e1) * 1e3 / (reps * rot)
            del g
        us, us_pr = times[0], times[bw.BW_ATTN_PAST_READY]
        res["contexts"][str(L)] = {
            "us_per_call": round(us, 3),
            "kv_bytes_per_call": kv_bytes,
            "kv_GBps": round(kv_bytes / (us * 1e3), 1),
            "hbm_frac": round(kv_bytes / (us * 1e3) / peak_gbs, 4),
            "caches_rotated": rot,
            "past_ready": {
                "us_per_call": round(us_pr, 3),
                "kv_GBps": round(kv_bytes / (us_pr * 1e3), 1),
                "hbm_frac": round(kv_bytes / (us_pr * 1e3) / peak_gbs, 4)},
        }
        del kcs, vcs
        torch.cuda.empty_cache()
    return res


def time_cold(torch, bw, dev, N, K, M, reps=50):
    """Microseconds of one isolated bw_gemv_w2a8 call: a 512 MB buffer is
    written first (L2 holds no weights), then events bracket the call alone
    on an otherwise idle stream, so the launch latency is included (the
    way the pages time their kernel).  Median of `reps`."""
    seed = synth.base_seed(2, 2)
    canon = synth.canonical_weights(seed, N, K)
    packed = bw.bw_repack(torch.from_numpy(canon).to(dev), N, K)
    xf = torch.from_numpy(synth.normal_f32(seed, M * K).reshape(M, K)).to(dev)
    q, s_ = bw.bw_quant_act(xf)
    ws = torch.ones(1, device=dev).to(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty((512 << 20,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    times = []
    with torch.cuda.stream(stream):
        for i in range(reps + 3):
            flush.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            stream.synchronize()
            e0.record(stream)
            bw.bw_gemv_w2a8(q, packed, s_, ws, [0, N], N, K, y=y,
                            stream=stream)
            e1.record(stream)
            stream.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) * 1e3)
    bw.bw_device_error(stream)
    return statistics.median(times)


def run_single(args):
    """One shape over rotating weight buffers; also the command the kernel
    profiles are taken with."""
    import torch
    import bit_gemv_bitlinear_gb300 as bw

    dims = [int(v) for v in args.single.split(",")]
    N, K = dims[0], dims[1]
    M = dims[2] if len(dims) > 2 else 1
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.cold:
        reps = max(1, min(args.iters, 200))
        us = time_cold(torch, bw, dev, N, K, M, reps=reps)
        print(json.dumps({"single": [N, K, M], "cold": True, "calls": reps,
                          "us_per_call": round(us, 3),
                          "weight_GBps": round(weight_bytes(N, K)
                                               / (us * 1e3), 1),
                          "timing": "median of isolated calls after a "
                                    "512 MB write, launch included"}),
              flush=True)
        return
    t = time_shape(torch, bw, dev, N, K, M, iters=args.iters,
                   rotate=args.rotate, eager=args.eager, lut=args.lut,
                   gemm=args.gemm)
    us = t["us"]
    kernel = ("pair-table (LUT)" if args.lut else
              "prefill (bw_gemm_w2a8)" if args.gemm else "bw_gemv_w2a8")
    print(json.dumps({"single": [N, K, M], "rotate": t["rotate"],
                      "kernel": kernel,
                      "tflops": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1),
                      "graph": not args.eager, "calls": t["calls"],
                      "us_per_call": round(us, 3),
                      "weight_GBps": round(t["weight_bytes"] / (us * 1e3), 1),
                      "alg_GBps": round(t["alg_bytes"] / (us * 1e3), 1)}),
          flush=True)


def main():
    args = parse_args()
    if args.single:
        run_single(args)
    elif args.attn and args.impl != "reference":
        import torch
        import bit_gemv_bitlinear_gb300 as bw
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        peak, _ = read_peaks()
        ctx = (tuple(int(v) for v in args.attn_contexts.split(","))
               if args.attn_contexts else ATTN_CONTEXTS)
        print(json.dumps({"attn_decode": run_attn_timing(
            torch, bw, dev, peak, contexts=ctx,
            iters=min(args.iters, 1024), rotate=args.attn_rotate)}),
            flush=True)
    elif args.stack and args.impl != "reference":
        import torch
        import bit_gemv_bitlinear_gb300 as bw
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"layer_stack": run_stack_timing(
            torch, bw, dev, args.stack_layers or STACK_LAYERS,
            args.stack_steps or STACK_STEPS,
            kv_positions=args.stack_kv)}),
              flush=True)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
