#!/usr/bin/env python
"""Benchmark of one EXL3 trellis MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: the GLM-5.3-Flash-shaped decode step (288 routed experts, top-8,
hidden 4096, intermediate 2048, K=2 codes, 4 bf16 tokens, plus an fp16 shared
expert), synthetic seeded data.  One JSON line on rank 0.

ours:      the CUDA library through its C ABI; the step is captured once in a
           CUDA graph and replayed; L2 is flushed (512 MiB written, then 512
           MiB read, so no dirty line is left) before every timed step.  A
           second graph of the same forward with per-stage CUDA events inside
           gives the stage times and the dominant kernel's duration for the
           roofline.  e2e: the same forward through the public API with
           pinned-host inputs copied in and the output copied out inside the
           timed region.
reference: the CPU oracle as it stands, on this host, on a bounded sample
           (one (token, expert) pair per step).
Under torchrun (N > 1) every rank runs its own token batch (weak scaling).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "decode"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="decode (default), verify3, verify4, prefill: parity/profiling cases")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count (smaller device footprint for profilers)")
    ap.add_argument("--layer", type=int, default=0, help="layer of a stacked workload (long)")
    ap.add_argument("--hadamard", action="store_true",
                    help="format v2: the workload's layer with the 128-point Hadamard rotation")
    ap.add_argument("--mixed", action="store_true",
                    help="every expert tensor K3 or K4 (seeded), the 3.5 bpw mixed recipe")
    ap.add_argument("--shared-coded", action="store_true",
                    help="the shared expert trellis-coded as one more expert (weight 1), "
                         "replacing a dense one")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own token batch (weak scaling: every rank runs its own)."""
    return seed + 1000 * rank


def max_over_ranks(value: float, device, world: int) -> float:
    """The largest of the ranks' values (the job's wall time is its slowest rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the (max) time."""
    return world * tokens_per_step * steps / (total_ms / 1e3)


# Issue-slot peak of the trellis decode (weights/s): 128 lane-instructions per
# SM and clock, 152 SMs, 2070 MHz maximum clock; K = 2 and 4 need 4 integer
# instructions per weight (window, multiply, correction, mask-xor: two on the
# ALU pipe, two on the FMA pipe), K = 3 needs 3 on the 64-lane ALU pipe
# (window, mask, mask-xor) besides the multiply.
DECODE_PEAK = {kk: 152 * 2.070e9 * (128 / 4 if kk in (2, 4) else 64 / 3) for kk in (2, 3, 4)}


def expert_work(spec, counts, per: int):
    """Algorithmic work of the two expert stages ("gate_up", "down") of one
    step: weight decodes (every active expert's weights once per unit of
    `per` tokens: a GEMV token group or a tensor-core tile), the same divided
    by the decode peak of each expert's width (seconds at peak), and code +
    side-vector bytes of the active experts.  counts: tokens per expert."""
    H, I = spec.hidden, spec.inter
    side_b = (H + I) * 2
    dec_w = {"gate_up": 0, "down": 0}
    dec_t = {"gate_up": 0.0, "down": 0.0}
    code_bytes = {"gate_up": 0, "down": 0}
    for e, c in enumerate(counts):
        if c <= 0:
            continue
        u = (int(c) + per - 1) // per
        for pr in range(3):
            st = "down" if pr == 2 else "gate_up"
            kk = spec.width(pr, e)
            dec_w[st] += u * H * I
            dec_t[st] += u * H * I / DECODE_PEAK[kk]
            code_bytes[st] += H * I * kk // 8 + side_b
    return dec_w, dec_t, code_bytes


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant stage's launches in one step, from ncu captures summarised under
# profiles/ (decode: gemv_kernel_K2_decode.md; prefill: the big- and
# small-tile kernels of the gate/up stage, prefill_gemm_dram.md); reported
# only while the kernel sources hash to what was captured (otherwise null).
NCU_TRAFFIC = {
    ("decode", "gate_up"): 128.116736e6 + 4.404480e6,
    ("prefill", "gate_up"): 4072320512,  # big-tile + small-tile launches
    ("prefill", "down"): 2429370624,
    ("decode", "down"): 63.692288e6 + 0.870144e6,
}
NCU_SOURCES = {
    "decode": {
        "trellis_quantized_moe_exl3_gb300/csrc/moe_gemv.cu": "d195d448e473addceaac4a0d4c850cd1e9550ed8",
        "trellis_quantized_moe_exl3_gb300/csrc/common.cuh": "4009ec5d411a93aadb8d82381585cf05645c8e6c",
    },
    "prefill": {
        "trellis_quantized_moe_exl3_gb300/csrc/moe_gemm.cu": "6b460aa5a90cb5bd2a19b8ac321fa9d9eacfb102",
        "trellis_quantized_moe_exl3_gb300/csrc/common.cuh": "4009ec5d411a93aadb8d82381585cf05645c8e6c",
        "trellis_quantized_moe_exl3_gb300/csrc/umma.cuh": "b447c8cca474276a478c6b77fc3e35111d3004a0",
        "trellis_quantized_moe_exl3_gb300/csrc/pipeline.cuh": "90e55f7d8ddca6b4f57fedbba41ac44ecb974179",
    },
}


def ncu_traffic(workload, kernel):
    import hashlib
    srcs = NCU_SOURCES.get(workload)
    if not srcs or (workload, kernel) not in NCU_TRAFFIC:
        return None
    for rel, digest in srcs.items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha1(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return NCU_TRAFFIC[(workload, kernel)]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


# ----------------------------------------------------------------------------- oracle timing
def oracle_pair_rate(wl, spec, x, logits, n_pairs, shared_w=None, codes=None):
    """Time the CPU oracle on n_pairs (token, expert) pairs of token 0 and the
    shared expert of token 0; returns (tokens/s, seconds used, sample text)."""
    import numpy as np

    import oracle
    from trellis_quantized_moe_exl3_gb300 import synth
    codes = codes if codes is not None else [synth.layer_codes(spec, p) for p in range(3)]
    sides = [synth.side_vectors(spec, p) for p in range(3)]
    ol = oracle.Layer(spec.num_experts, spec.hidden, spec.inter, spec.K, codes,
                      [s[0] for s in sides], [s[1] for s in sides], fp8_round=spec.fp8_round,
                      shared_w=shared_w, hadamard=spec.hadamard, shared_coded=spec.shared_coded,
                      expert_K=np.array(spec.expert_K, np.uint8) if spec.expert_K else None)
    ids, w, _, _ = oracle.route(logits, wl.top_k)
    t0 = time.perf_counter()
    for j in range(n_pairs):
        t, jj = divmod(j, wl.top_k)
        ol.expert_pair(x[t % wl.T], wl.act == "bf16", int(ids[t % wl.T, jj]), float(w[t % wl.T, jj]))
    t_pairs = (time.perf_counter() - t0) / n_pairs
    t1 = time.perf_counter()
    if shared_w is not None:
        ol.shared_row(x[0], wl.act == "bf16")
    t_shared = time.perf_counter() - t1
    kp = wl.top_k + int(spec.shared_coded)  # the coded shared expert costs one more pair
    per_token = kp * t_pairs + t_shared
    sample = (f"{n_pairs} (token, expert) pair(s) of the {wl.T}-token {wl.name} workload"
              + (" + the shared expert of one token" if shared_w is not None else "")
              + f"; tokens/s = 1 / ({kp} x pair time"
              + (" + shared time)" if shared_w is not None else ")"))
    return 1.0 / per_token, time.perf_counter() - t0, sample


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from trellis_quantized_moe_exl3_gb300 import synth
    wl, spec = pick_workload(args)
    x = synth.activations(wl.seed, wl.T, spec.hidden, wl.act)
    logits = synth.router_logits(spec.seed, wl.T, spec.num_experts, wl.routing)
    codes = [synth.layer_codes(spec, p) for p in range(3)]
    sides = [synth.side_vectors(spec, p) for p in range(3)]
    sw = synth.shared_weights(spec) if spec.shared else None
    ol = oracle.Layer(spec.num_experts, spec.hidden, spec.inter, spec.K, codes,
                      [s[0] for s in sides], [s[1] for s in sides], shared_w=sw,
                      fp8_round=spec.fp8_round, hadamard=spec.hadamard,
                      shared_coded=spec.shared_coded,
                      expert_K=np.array(spec.expert_K, np.uint8) if spec.expert_K else None)
    ids, w, _, _ = oracle.route(logits, wl.top_k)
    pairs = [(t, j) for t in range(wl.T) for j in range(wl.top_k)]
    for s in range(args.warmup):
        t, j = pairs[s % len(pairs)]
        ol.expert_pair(x[t], wl.act == "bf16", int(ids[t, j]), float(w[t, j]))
    ts = time.perf_counter()
    if sw is not None:
        ol.shared_row(x[0], wl.act == "bf16")
    t_shared = time.perf_counter() - ts
    t0 = time.perf_counter()
    for s in range(args.steps):
        t, j = pairs[(args.warmup + s) % len(pairs)]
        ol.expert_pair(x[t], wl.act == "bf16", int(ids[t, j]), float(w[t, j]))
    t_pair = (time.perf_counter() - t0) / args.steps
    kp = wl.top_k + int(spec.shared_coded)  # the coded shared expert costs one more pair
    per_token = kp * t_pair + t_shared
    value = 1.0 / per_token
    sample = (f"one (token, expert) pair of the {wl.T}-token {wl.name} workload per step; tokens/s = "
              f"1 / ({kp} x mean pair time"
              + (" + shared-expert time of one token)" if sw is not None else ")"))
    line = {
        "impl": "reference", "metric": "moe_layer_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_token * 1e3 * wl.T, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def pick_workload(args):
    import dataclasses

    from trellis_quantized_moe_exl3_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    spec = wl.layers[args.layer]
    if args.layer:
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-layer{args.layer}")
    if args.experts:
        spec = dataclasses.replace(spec, num_experts=args.experts)
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-E{args.experts}")
    if args.hadamard:
        spec = dataclasses.replace(spec, hadamard=True)
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-hadamard")
    if args.shared_coded:
        spec = dataclasses.replace(spec, shared=False, shared_coded=True)
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-sharedcoded")
    if args.mixed:
        spec = dataclasses.replace(spec, expert_K=synth.mixed_widths(spec.seed, spec.n_coded))
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-mixedK34")
    return wl, spec


def workload_config(wl):
    s = wl.layers[0]
    return {"workload": (f"{wl.name}: {s.num_experts} experts top-{wl.top_k}, hidden {s.hidden}, "
                         f"inter {s.inter}, K={list(s.K)}, T={wl.T} {wl.act}"
                         + (", + fp16 shared expert" if s.shared else "")
                         + (", + trellis-coded shared expert" if s.shared_coded else "")
                         + (", Hadamard rotation (format v2)" if s.hadamard else "")
                         + (", every expert tensor K3 or K4 (seeded)" if s.expert_K else "")),
            "T": wl.T, "top_k": wl.top_k, "experts": s.num_experts, "hidden": s.hidden,
            "inter": s.inter, "K": list(s.K), "fp8_round": s.fp8_round, "hadamard": s.hadamard,
            "l2": "flushed before every timed step (512 MiB written, then 512 MiB read)"}


# ----------------------------------------------------------------------------- ours
def run_ours(args):
    import ctypes

    import numpy as np
    import torch

    from trellis_quantized_moe_exl3_gb300 import _lib, synth
    from trellis_quantized_moe_exl3_gb300 import build as lib_build
    from trellis_quantized_moe_exl3_gb300.api import Layer, route

    world, rank, local = dist_env()
    lib_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    wl, spec = pick_workload(args)
    codes = [synth.layer_codes(spec, p) for p in range(3)]
    sides = [synth.side_vectors(spec, p) for p in range(3)]
    sw = synth.shared_weights(spec) if spec.shared else None
    # every rank runs its own token batch (weak scaling)
    x_np = synth.activations(rank_seed(wl.seed, rank), wl.T, spec.hidden, wl.act)
    lg_np = synth.router_logits(rank_seed(spec.seed, rank), wl.T, spec.num_experts, wl.routing)

    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    d_codes = [t16(c) for c in codes]
    d_suh = [t16(s[0]).view(torch.float16) for s in sides]
    d_svh = [t16(s[1]).view(torch.float16) for s in sides]
    d_sw = [t16(a).view(torch.float16) for a in sw] if sw else None
    layer = Layer(d_codes, d_suh, d_svh, spec.K, fp8_round=spec.fp8_round, shared=d_sw,
                  hadamard=spec.hadamard, shared_coded=spec.shared_coded, expert_K=spec.expert_K)
    x = t16(x_np).view(torch.bfloat16)
    lg = torch.from_numpy(lg_np).to(dev)
    T, k = wl.T, wl.top_k
    ws = layer.workspace(T, k, dev)
    out = torch.empty_like(x)
    # L2 flush: write 512 MiB (4x L2), then read it back, so the lines left in
    # L2 are clean and no write-back of the flush competes with the step
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)

    def flush_l2():
        flush.fill_(1)
        flush.sum()

    s = torch.cuda.Stream(device=dev)
    L = _lib.lib()
    with torch.cuda.stream(s):
        for _ in range(2):
            layer.forward(x, lg, k, out=out, ws=ws, stream=s)
    torch.cuda.synchronize()

    # routing of this batch (host side, outside any timing): the per-expert
    # counts behind the algorithmic work of each kernel
    _, _, r_off, _ = route(lg, k)
    counts = torch.diff(r_off).cpu().numpy()
    if spec.shared_coded:  # its segment holds every token
        counts = np.append(counts, T)
    n_active = int((counts > 0).sum())

    # headline graph: the forward alone
    use_graph = True
    c0 = L.exl3_launch_count()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=s):
            layer.forward(x, lg, k, out=out, ws=ws, stream=s)
    except Exception:
        use_graph = False
    launches_per_step = int(L.exl3_launch_count() - c0)

    # stage graph: the same forward with stage-boundary events inside
    n_ev = _lib.EXL3_NUM_STAGE_EVENTS
    stage_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    with torch.cuda.stream(s):
        for e in stage_ev:
            e.record(s)
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * n_ev)(*[e.cuda_event for e in stage_ev])
    _lib.check(L.exl3_layer_set_stage_events(layer.handle, arr, n_ev), "set_stage_events")
    g_stage = None
    if use_graph:
        g_stage = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g_stage, stream=s):
                layer.forward(x, lg, k, out=out, ws=ws, stream=s)
        except Exception:
            g_stage = None
    L.exl3_layer_set_stage_events(layer.handle, None, 0)

    def step():
        if use_graph:
            g.replay()
        else:
            layer.forward(x, lg, k, out=out, ws=ws, stream=s)

    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            flush_l2()
            step()
    torch.cuda.synchronize()

    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except ValueError:
            pass
    clocks = ClockSampler(gpu_index)
    start_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    end_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(s):
        for i in range(args.steps):
            flush_l2()
            start_ev[i].record(s)
            step()
            end_ev[i].record(s)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(start_ev, end_ev)]
    tot = max_over_ranks(float(np.sum(step_ms)), dev, world)
    ms_per_step = tot / args.steps
    value = job_tokens_per_s(world, T, args.steps, tot)

    # stage times: the stage graph (or eager forwards with the events set)
    stage_ms = np.zeros(n_ev - 1)
    stage_live = g_stage is not None
    if not stage_live:
        L.exl3_layer_set_stage_events(layer.handle, arr, n_ev)
    with torch.cuda.stream(s):
        for i in range(args.steps):
            flush_l2()
            if stage_live:
                g_stage.replay()
            else:
                layer.forward(x, lg, k, out=out, ws=ws, stream=s)
            stage_ev[-1].synchronize()
            for j in range(n_ev - 1):
                stage_ms[j] += stage_ev[j].elapsed_time(stage_ev[j + 1])
    L.exl3_layer_set_stage_events(layer.handle, None, 0)
    stage_ms /= args.steps

    # e2e: public API with host buffers, copies inside the timed region
    x_host = torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).view(torch.bfloat16).pin_memory()
    lg_host = torch.from_numpy(lg_np).pin_memory()
    out_host = torch.empty((T, spec.hidden), dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(x)
    lg_d = torch.empty_like(lg)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    with torch.cuda.stream(s):
        for i in range(args.warmup + args.steps):
            flush_l2()
            e0.record(s)
            x_d.copy_(x_host, non_blocking=True)
            lg_d.copy_(lg_host, non_blocking=True)
            layer.forward(x_d, lg_d, k, out=out, ws=ws, stream=s)
            out_host.copy_(out, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            if i >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
    e2e_tot = max_over_ranks(float(np.sum(e2e_ms)), dev, world)
    e2e_value = job_tokens_per_s(world, T, args.steps, e2e_tot)

    # roofline of the dominant expert kernel (the larger of gate/up and down)
    hbm, bf16_tf, src = peaks()
    H, I = spec.hidden, spec.inter
    stage_names = _lib.STAGE_NAMES
    P = T * (k + int(spec.shared_coded))          # pairs, the coded shared expert's included
    gemm_path = P >= 16 * spec.n_coded
    dec_w, dec_t, code_bytes = expert_work(spec, counts, 512 if gemm_path else 8)
    flops = {"gate_up": 2.0 * P * H * I * 2, "down": 2.0 * P * H * I}
    dom = max(("gate_up", "down"), key=lambda n: stage_ms[stage_names.index(n)])
    dom_ms = float(stage_ms[stage_names.index(dom)])
    peak_wps = dec_w[dom] / dec_t[dom]   # the widths' peaks, weighted by their decodes
    dec_rate = dec_w[dom] / (dom_ms / 1e3)
    hbm_rate = code_bytes[dom] / (dom_ms / 1e3) / 1e9
    if gemm_path:
        tf = flops[dom] / (dom_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": tf, "peak": bf16_tf,
                "unit": "TFLOP/s", "frac": tf / bf16_tf, "traffic": ncu_traffic(wl.name, dom),
                "traffic_unit": "bytes per step of the stage's launches (ncu)",
                "algorithmic_flops": flops[dom], "ms": dom_ms,
                "peak_source": f"{src} (bf16_tflops burst; the fp16 dense rate equals bf16)",
                "alu_view": {"achieved": dec_rate / 1e9, "peak": peak_wps / 1e9,
                             "unit": "Gweight/s", "frac": dec_rate / peak_wps,
                             "weight_decodes": dec_w[dom]}}
    else:
        traffic = ncu_traffic(wl.name, dom)
        roof = {"bound": "alu", "kernel": dom, "achieved": dec_rate / 1e9,
                "peak": peak_wps / 1e9, "unit": "Gweight/s", "frac": dec_rate / peak_wps,
                "traffic": traffic, "traffic_unit": "bytes per launch (ncu)",
                "weight_decodes": dec_w[dom], "ms": dom_ms,
                "peak_source": "derived: 152 SMs x 2070 MHz x 128 issue slots / instructions per weight",
                "hbm_view": {"achieved": hbm_rate, "peak": hbm, "unit": "GB/s",
                             "frac": hbm_rate / hbm, "algorithmic_bytes": code_bytes[dom],
                             "peak_source": f"{src} (hbm_gbs, burst)"}}
    step_bytes = code_bytes["gate_up"] + code_bytes["down"] + (3 * H * I * 2 if sw else 0)
    line = {
        "metric": "moe_layer_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16",
        "arithmetic": "integer trellis decode; fp16 MMA operands, fp32 accumulate; "
                      "bf16 activations in and out",
        "data": "synthetic (seeded PCG64): uniform uint16 codes, side vectors 1+0.1N(0,1), "
                "N(0,1) activations and router logits",
        "config": {**workload_config(wl), "cuda_graph": use_graph, "n_active_experts": n_active,
                   "path": "gemm (tcgen05)" if gemm_path else "gemv (mma.sync)",
                   "stage_times": "separate graph with stage events" if stage_live else "eager re-run"},
        "roofline": roof,
        "step_roofline": {"bytes": step_bytes, "achieved_gbs": step_bytes / (ms_per_step / 1e3) / 1e9,
                          "frac": step_bytes / (ms_per_step / 1e3) / 1e9 / hbm,
                          "what": "code + side-vector + shared-expert bytes of one step / step time"},
        "stage_ms": {n: float(v) for n, v in zip(stage_names, stage_ms)},
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2 + lg_host.numel() * 4),
                "d2h_bytes_per_step": int(out_host.numel() * 2),
                "ms_per_step": e2e_tot / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline and not args.experts:
        # one whole token: its top_k (token, expert) pairs (+ its shared expert)
        rate, secs, sample = oracle_pair_rate(wl, spec, x_np, lg_np, wl.top_k, shared_w=sw,
                                              codes=codes)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": sample, "seconds": secs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
