"""Host logic of bench.py's multi-GPU path (one replica per rank, weak
scaling), run as two gloo ranks on the CPU: every rank gets its own token
batch, the job time is the slowest rank's, and the job throughput counts the
tokens of all ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r pretends its timed steps took 10 + r ms
        mine = 10.0 + rank
        got = bench.max_over_ranks(mine, torch.device("cpu"), world)
        out[rank] = (got, bench.rank_seed(7, rank))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 11.0          # both ranks report the max
    assert res[0][1] != res[1][1]                  # distinct token batches


def test_job_throughput_counts_every_rank():
    # 2 ranks x 4 tokens x 10 steps in 5 ms = 16,000 tokens/s
    assert bench.job_tokens_per_s(2, 4, 10, 5.0) == pytest.approx(16000.0)
    assert bench.max_over_ranks(3.0, torch.device("cpu"), 1) == 3.0


def test_expert_work_accounting():
    """The bench's algorithmic work of the expert stages: decodes once per
    unit of tokens, code bytes at each expert's width, and the decode peak of
    a mixed-width stage weighted by its decodes."""
    import dataclasses

    import bench
    from trellis_quantized_moe_exl3_gb300 import synth
    spec = synth.LayerSpec(seed=0, num_experts=3, hidden=256, inter=128, K=(2, 2, 4))
    counts = [0, 9, 8]  # expert 1: two groups of <= 8 tokens; expert 2: one
    dec_w, dec_t, code_b = bench.expert_work(spec, counts, 8)
    H, I = 256, 128
    assert dec_w == {"gate_up": 3 * 2 * H * I, "down": 3 * H * I}
    assert code_b == {"gate_up": 2 * (2 * H * I * 2 // 8 + 2 * (H + I) * 2),
                      "down": 2 * (H * I * 4 // 8 + (H + I) * 2)}
    assert abs(dec_w["gate_up"] / dec_t["gate_up"] - bench.DECODE_PEAK[2]) < 1e-3
    mixed = dataclasses.replace(spec, expert_K=((3, 3, 3), (3, 4, 2), (4, 4, 4)))
    dec_w, dec_t, code_b = bench.expert_work(mixed, counts, 8)
    # expert 1 (2 units) gate K3 + up K4, expert 2 (1 unit) gate and up K4
    want_t = H * I * (2 / bench.DECODE_PEAK[3] + 2 / bench.DECODE_PEAK[4] + 2 / bench.DECODE_PEAK[4])
    assert abs(dec_t["gate_up"] - want_t) < 1e-15
    assert code_b["down"] == H * I * 2 // 8 + H * I * 4 // 8 + 2 * (H + I) * 2


def test_workload_overrides_for_profiling():
    """--experts and --tokens shrink a workload (for profiler captures) and
    rename it, leaving the other fields as they were."""
    import argparse

    import bench
    from trellis_quantized_moe_exl3_gb300 import synth
    args = argparse.Namespace(layer=0, experts=64, tokens=1024, hadamard=False,
                              shared_coded=False, mixed=False)
    wl, spec = bench.pick_workload(args, "prefill+fp8")
    base = synth.WORKLOADS["prefill"]
    assert wl.T == 1024 and spec.num_experts == 64
    assert spec.act_fp8 and spec.fp8_round and spec.K == base.layers[0].K
    assert wl.top_k == base.top_k and wl.routing == base.routing
    assert "E64" in wl.name and "T1024" in wl.name
    args = argparse.Namespace(layer=0, experts=0, tokens=0, hadamard=False,
                              shared_coded=False, mixed=False)
    wl, spec = bench.pick_workload(args, "prefill")
    assert wl.T == base.T and spec.num_experts == base.layers[0].num_experts and not spec.act_fp8
