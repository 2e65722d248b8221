#!/usr/bin/env python
"""Benchmark of one EXL3 trellis MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode,verify3,verify4,prefill]

Workloads (synthetic seeded data, the GLM-5.3-Flash MoE layer shape: 288
routed experts, top-8, hidden 4096, intermediate 2048): the decode step (K2,
4 bf16 tokens, plus an fp16 shared expert), the speculative-verify batch (32
tokens, K3 and K4) and the prefill layer (K4 with the E4M3 rule, 7168
tokens), the last one also with FP8 x FP8 products ("prefill+fp8": E4M3
activation rows with an fp32 scale each, tcgen05 kind::f8f6f4).  By default
all five run, one after the other, and rank 0 prints ONE JSON line: its
top-level numbers are the decode step's, and "configs" holds one block per
workload with the same fields.

ours:      the CUDA library through its C ABI; the step is captured once in a
           CUDA graph and replayed; L2 is flushed (512 MiB written, then 512
           MiB read, so no dirty line is left) before every timed step.  A
           second graph of the same forward with per-stage CUDA events inside
           gives the stage times and the dominant kernel's duration for the
           roofline.  e2e: the same forward through the public API with
           pinned-host inputs copied in and the output copied out inside the
           timed region.
reference: the CPU oracle as it stands, on this host's cores: a step is one
           token of the workload (its top_k (token, expert) pairs, plus the
           shared expert, each on its own thread).
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

WORKLOADS = ("decode", "verify3", "verify4", "prefill", "prefill+fp8")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=",".join(WORKLOADS),
                    help="comma-separated workloads (decode, verify3, verify4, prefill, long; "
                         "a '+fp8' suffix selects FP8 x FP8 products); the first gives the "
                         "line's top-level numbers")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count (smaller device footprint for profilers)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the token count (small cases for profilers)")
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
# dominant stage's launch in one decode or verify step, from ncu captures of
# this bench's decode and verify workloads (the GEMV gate/up and down
# launches); reported only while the kernel sources hash to what was
# captured (otherwise null).
# The prefill stages have no full-size capture (their counters come from a
# 64-expert case), so their traffic is null.
NCU_TRAFFIC = {
    ("decode", "gate_up"): 128107264 + 3334656,
    ("decode", "down"): 63692800 + 86016,
    ("verify3", "gate_up"): 828007680 + 9542656,
    ("verify3", "down"): 410294784 + 5534208,
    ("verify4", "gate_up"): 1121739520 + 9833472,
    ("verify4", "down"): 557677824 + 5964800,
}
_GEMV_SOURCES = {
    "trellis_quantized_moe_exl3_gb300/csrc/moe_gemv.cu": "5584e0cb62598beb959c3f571892cc9a5342db4b",
    "trellis_quantized_moe_exl3_gb300/csrc/common.cuh": "91ce3402e4abd315dd1aaa25eaa71d9884431157",
    "trellis_quantized_moe_exl3_gb300/csrc/pipeline.cuh": "1f11aa433c95c15ed0fd2ec1605b876b5f7100cc",
}
NCU_SOURCES = {"decode": _GEMV_SOURCES, "verify3": _GEMV_SOURCES, "verify4": _GEMV_SOURCES}


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
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_layer(spec, codes=None):
    import numpy as np

    import oracle
    from trellis_quantized_moe_exl3_gb300 import synth
    codes = codes if codes is not None else [synth.layer_codes(spec, p) for p in range(3)]
    sides = [synth.side_vectors(spec, p) for p in range(3)]
    sw = synth.shared_weights(spec) if spec.shared else None
    return oracle.Layer(spec.num_experts, spec.hidden, spec.inter, spec.K, codes,
                        [s[0] for s in sides], [s[1] for s in sides], fp8_round=spec.fp8_round,
                        shared_w=sw, hadamard=spec.hadamard, shared_coded=spec.shared_coded,
                        expert_K=np.array(spec.expert_K, np.uint8) if spec.expert_K else None,
                        act_fp8=spec.act_fp8)


class OracleTokens:
    """One token of a workload through the CPU oracle as it stands: the
    token's top_k (token, expert) pairs (the coded shared expert's pair
    included) and the dense shared expert, each a task on its own thread (the
    C oracle releases the GIL), so a step uses min(tasks, host cores) cores."""

    def __init__(self, wl, spec, x, logits, codes=None):
        import oracle
        self.wl, self.spec, self.x = wl, spec, x
        self.ol = oracle_layer(spec, codes)
        self.ids, self.w, _, _ = oracle.route(logits, wl.top_k)
        self.n_tasks = wl.top_k + int(spec.shared_coded) + int(spec.shared)
        self.cores = max(1, min(self.n_tasks, host_cores()))

    def _tasks(self, t):
        wl, spec, bf = self.wl, self.spec, self.wl.act == "bf16"
        jobs = [(lambda j=j: self.ol.expert_pair(self.x[t], bf, int(self.ids[t, j]),
                                                 float(self.w[t, j])))
                for j in range(wl.top_k)]
        if spec.shared_coded:
            jobs.append(lambda: self.ol.expert_pair(self.x[t], bf, spec.num_experts, 1.0))
        if spec.shared:
            jobs.append(lambda: self.ol.shared_row(self.x[t], bf))
        return jobs

    def step(self, t) -> float:
        """Seconds of wall time for token t."""
        import concurrent.futures as cf
        jobs = self._tasks(t % self.wl.T)
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=self.cores) as ex:
            list(ex.map(lambda f: f(), jobs))
        return time.perf_counter() - t0

    def sample_text(self, n):
        return (f"{n} token(s) of the {self.wl.T}-token {self.wl.name} workload, each step one "
                f"token: its {self.n_tasks} expert evaluations (top-{self.wl.top_k} pairs"
                + (" + the coded shared expert" if self.spec.shared_coded else "")
                + (" + the dense shared expert" if self.spec.shared else "")
                + f") on {self.cores} threads; tokens/s = tokens / wall time")


def oracle_baseline(wl, spec, x, logits, n_tokens=2, codes=None):
    ot = OracleTokens(wl, spec, x, logits, codes)
    secs = [ot.step(t) for t in range(n_tokens)]
    tot = sum(secs)
    return {"value": n_tokens / tot, "unit": "tokens/s", "cores": ot.cores, "kind": "oracle",
            "sample": ot.sample_text(n_tokens), "seconds": tot, "host_cores": host_cores()}


def pick_workload(args, name):
    import dataclasses

    from trellis_quantized_moe_exl3_gb300 import synth
    fp8_ops = name.endswith("+fp8")
    name = name[:-4] if fp8_ops else name
    wl = synth.WORKLOADS[name]
    spec = wl.layers[args.layer if name == "long" else 0]
    if name == "long" and args.layer:
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-layer{args.layer}")
    if args.experts:
        spec = dataclasses.replace(spec, num_experts=args.experts)
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-E{args.experts}")
    if args.tokens:
        wl = dataclasses.replace(wl, T=args.tokens, name=f"{wl.name}-T{args.tokens}")
    if args.hadamard:
        spec = dataclasses.replace(spec, hadamard=True)
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-hadamard")
    if args.shared_coded:
        spec = dataclasses.replace(spec, shared=False, shared_coded=True)
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-sharedcoded")
    if args.mixed:
        spec = dataclasses.replace(spec, expert_K=synth.mixed_widths(spec.seed, spec.n_coded))
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}-mixedK34")
    if fp8_ops:  # the E4M3 operand needs the E4M3 rule
        spec = dataclasses.replace(spec, act_fp8=True, fp8_round=True)
        wl = dataclasses.replace(wl, layers=(spec,), name=f"{wl.name}+fp8")
    return wl, spec


def workload_config(wl, spec):
    """The workload's identity: the same keys on both arms."""
    s = spec
    return {"workload": (f"{wl.name}: {s.num_experts} experts top-{wl.top_k}, hidden {s.hidden}, "
                         f"inter {s.inter}, K={list(s.K)}, T={wl.T} {wl.act}"
                         + (", E4M3-rounded codebook" if s.fp8_round else "")
                         + (", + fp16 shared expert" if s.shared else "")
                         + (", + trellis-coded shared expert" if s.shared_coded else "")
                         + (", Hadamard rotation (format v2)" if s.hadamard else "")
                         + (", every expert tensor K3 or K4 (seeded)" if s.expert_K else "")
                         + (", FP8 x FP8 products (E4M3 activation rows)" if s.act_fp8 else "")),
            "T": wl.T, "top_k": wl.top_k, "experts": s.num_experts, "hidden": s.hidden,
            "inter": s.inter, "K": list(s.K), "fp8_round": s.fp8_round, "hadamard": s.hadamard,
            "act_fp8": s.act_fp8, "routing": wl.routing,
            "l2": "flushed before every timed step (512 MiB written, then 512 MiB read)"}


def line_config(blocks):
    first = blocks[0]
    cfg = dict(first["config"])
    cfg["workloads"] = [b["name"] for b in blocks]
    return cfg


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from trellis_quantized_moe_exl3_gb300 import synth
    names = [n for n in args.workload.split(",") if n]
    blocks = []
    for i, name in enumerate(names):
        wl, spec = pick_workload(args, name)
        x = synth.activations(wl.seed, wl.T, spec.hidden, wl.act)
        logits = synth.router_logits(spec.seed, wl.T, spec.num_experts, wl.routing)
        ot = OracleTokens(wl, spec, x, logits)
        # the first workload takes the full --steps/--warmup; the others a
        # bounded sample of two tokens each, so the run stays within minutes
        warm, steps = (args.warmup, args.steps) if i == 0 else (0, 2)
        for t in range(warm):
            ot.step(t)
        secs = [ot.step(warm + t) for t in range(steps)]
        ms = 1e3 * sum(secs) / steps
        value = 1e3 / ms
        blocks.append({"name": name, "config": workload_config(wl, spec), "value": value,
                       "unit": "tokens/s", "ms_per_step": ms, "steps": steps, "warmup": warm,
                       "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": ot.cores,
                                        "kind": "oracle", "sample": ot.sample_text(steps),
                                        "host_cores": host_cores()}})
        del ot
    top = blocks[0]
    line = {
        "impl": "reference", "metric": "moe_layer_tokens_per_s", "value": top["value"],
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": top["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": line_config(blocks),
        "cpu_baseline": top["cpu_baseline"],
        "e2e": {"value": top["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "configs": {b["name"]: {k: v for k, v in b.items() if k != "name"} for b in blocks},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ours
def measure_workload(args, name, dev, world, rank, local):
    """Time one workload on this rank's GPU; returns its block of the line."""
    import ctypes

    import numpy as np
    import torch

    from trellis_quantized_moe_exl3_gb300 import _lib, synth
    from trellis_quantized_moe_exl3_gb300.api import Layer, route

    wl, spec = pick_workload(args, name)
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
                  hadamard=spec.hadamard, shared_coded=spec.shared_coded, expert_K=spec.expert_K,
                  act_fp8=spec.act_fp8)
    act_t = torch.bfloat16 if wl.act == "bf16" else torch.float16
    x = t16(x_np).view(act_t)
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
    x_host = torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).view(act_t).pin_memory()
    lg_host = torch.from_numpy(lg_np).pin_memory()
    out_host = torch.empty((T, spec.hidden), dtype=act_t).pin_memory()
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

    roof = roofline(wl, spec, counts, T, k, stage_ms, sw is not None)
    block = {
        "name": name, "config": workload_config(wl, spec), "value": value, "unit": "tokens/s",
        "ms_per_step": ms_per_step, "steps": args.steps, "warmup": args.warmup,
        "roofline": roof["roofline"], "step_roofline": roof["step"],
        "stage_ms": {n: float(v) for n, v in zip(_lib.STAGE_NAMES, stage_ms)},
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2 + lg_host.numel() * 4),
                "d2h_bytes_per_step": int(out_host.numel() * 2),
                "ms_per_step": e2e_tot / args.steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "run": {"cuda_graph": use_graph, "n_active_experts": n_active,
                "path": roof["path"], "launches_per_step": launches_per_step,
                "stage_times": "separate graph with stage events" if stage_live else "eager re-run"},
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline and not args.experts and not args.tokens:
        block["cpu_baseline"] = oracle_baseline(wl, spec, x_np, lg_np, 2, codes=codes)
    block["dtype"] = "e4m3" if spec.act_fp8 else "f16"
    del layer, d_codes, d_suh, d_svh, d_sw, ws, flush, g, g_stage
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return block


def roofline(wl, spec, counts, T, k, stage_ms, has_shared):
    """Roofline of the dominant expert stage (the larger of gate/up and down):
    decode-sized steps against HBM on the active experts' code and
    side-vector bytes (with the decode issue-slot view beside it),
    prefill-sized steps against the dense tensor peak on 2 P H I flops per
    projection (with the decode view beside it)."""
    from trellis_quantized_moe_exl3_gb300 import _lib
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
    alu_view = {"achieved": dec_rate / 1e9, "peak": peak_wps / 1e9, "unit": "Gweight/s",
                "frac": dec_rate / peak_wps, "weight_decodes": dec_w[dom],
                "peak_source": "derived: 152 SMs x 2070 MHz x 128 issue slots / "
                               "instructions per weight"}
    traffic = ncu_traffic(wl.name, dom)
    if gemm_path:
        tf = flops[dom] / (dom_ms / 1e3) / 1e12
        # FP8 products: the measured bf16 peak times the nominal fp8 : bf16
        # ratio (4.5 : 2.25 PFLOP/s dense)
        peak_tf = bf16_tf * (2.0 if spec.act_fp8 else 1.0)
        roof = {"bound": "tensor", "kernel": dom, "achieved": tf, "peak": peak_tf,
                "unit": "TFLOP/s", "frac": tf / peak_tf, "traffic": traffic,
                "traffic_unit": "bytes per step of the stage's launches (ncu)",
                "algorithmic_flops": flops[dom], "ms": dom_ms,
                "peak_source": (f"{src} bf16_tflops burst x 2 (nominal fp8 : bf16 dense ratio)"
                                if spec.act_fp8 else
                                f"{src} (bf16_tflops burst; the fp16 dense rate equals bf16)"),
                "alu_view": alu_view}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": hbm_rate, "peak": hbm,
                "unit": "GB/s", "frac": hbm_rate / hbm, "traffic": traffic,
                "traffic_unit": "bytes per launch (ncu)",
                "algorithmic_bytes": code_bytes[dom], "ms": dom_ms,
                "peak_source": f"{src} (hbm_gbs, burst)",
                "alu_view": alu_view}
    step_bytes = code_bytes["gate_up"] + code_bytes["down"] + (3 * H * I * 2 if has_shared else 0)
    ms_step = float(sum(stage_ms))
    step = {"bytes": step_bytes, "achieved_gbs": step_bytes / (ms_step / 1e3) / 1e9,
            "frac": step_bytes / (ms_step / 1e3) / 1e9 / hbm,
            "what": "code + side-vector + shared-expert bytes of one step / step time"}
    return {"roofline": roof, "step": step,
            "path": "gemm (tcgen05)" if gemm_path else "gemv (mma.sync)"}


def merge_clocks(blocks):
    sms, mx, reasons, n = [], None, set(), 0
    for b in blocks:
        c = b["clocks"]
        if c.get("sm_mhz") is not None:
            sms.append(c["sm_mhz"])
        mx = c.get("sm_max_mhz") or mx
        reasons |= set(c.get("reasons", []))
        n += c.get("samples", 0)
    return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
            "reasons": sorted(reasons), "samples": n,
            "per_workload": {b["name"]: b["clocks"].get("sm_mhz") for b in blocks}}


def run_ours(args):
    import torch

    from trellis_quantized_moe_exl3_gb300 import build as lib_build

    world, rank, local = dist_env()
    lib_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    names = [n for n in args.workload.split(",") if n]
    blocks = [measure_workload(args, n, dev, world, rank, local) for n in names]
    top = blocks[0]
    line = {
        "metric": "moe_layer_tokens_per_s", "value": top["value"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": top["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16",
        "arithmetic": "integer trellis decode; fp16 MMA operands, fp32 accumulate; "
                      "bf16 activations in and out",
        "data": "synthetic (seeded PCG64): uniform uint16 codes, side vectors 1+0.1N(0,1), "
                "N(0,1) activations and router logits",
        "config": line_config(blocks),
        "roofline": top["roofline"],
        "e2e": top["e2e"],
        "gpu_launches": top["gpu_launches"],
        "clocks": merge_clocks(blocks),
        "configs": {b["name"]: {kk: v for kk, v in b.items() if kk != "name"} for b in blocks},
    }
    if "cpu_baseline" in top:
        line["cpu_baseline"] = top["cpu_baseline"]
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
