"""Expert parallelism, host logic, as two (and three) gloo ranks on the CPU.

Each rank takes its block of experts from expert_range, computes its partial
sum over the pairs of those experts (here with the CPU oracle, one
(token, expert) pair at a time; rank 0 adds the dense shared expert), and
ep_sum all-reduces the partials.  Every rank must end with the whole layer
output the oracle computes in one piece (fp64, up to the order of the sums)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from trellis_quantized_moe_exl3_gb300.ep import ep_sum, expert_range


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_expert_ranges_partition():
    for E in (1, 8, 9, 288, 289, 1024):
        for world in (1, 2, 3, 4, 7, 8):
            rs = [expert_range(r, world, E) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == E
            for (a0, a1), (b0, b1) in zip(rs, rs[1:]):
                assert a1 == b0 and a0 <= a1
            sizes = [b - a for a, b in rs]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        expert_range(2, 2, 8)


def _layer_case(coded):
    import oracle
    from trellis_quantized_moe_exl3_gb300 import synth
    spec = synth.LayerSpec(seed=210 + coded, num_experts=8, hidden=256, inter=128, K=(2, 3, 2),
                           shared=not coded, shared_coded=bool(coded))
    codes = [synth.layer_codes(spec, p) for p in range(3)]
    sides = [synth.side_vectors(spec, p) for p in range(3)]
    sw = synth.shared_weights(spec) if spec.shared else None
    ol = oracle.Layer(spec.num_experts, spec.hidden, spec.inter, spec.K, codes,
                      [s[0] for s in sides], [s[1] for s in sides], shared_w=sw,
                      shared_coded=spec.shared_coded)
    T, k = 6, 3
    x = synth.activations(211, T, spec.hidden, "bf16")
    logits = synth.router_logits(211, T, spec.num_experts, "normal")
    return spec, ol, x, logits, T, k


def _rank_main(rank, world, port, coded, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        spec, ol, x, logits, T, k = _layer_case(coded)
        ids, w, _, _ = oracle.route(logits, k)

        def partial(e0, e1, with_shared):
            y = np.zeros((T, spec.hidden))
            for t in range(T):
                for j in range(k):
                    if e0 <= ids[t, j] < e1:
                        y[t] += ol.expert_pair(x[t], True, int(ids[t, j]), float(w[t, j]))
                if spec.shared_coded and e0 <= spec.num_experts < e1:
                    y[t] += ol.expert_pair(x[t], True, spec.num_experts, 1.0)
                if spec.shared and with_shared:
                    y[t] += ol.shared_row(x[t], True)
            return torch.from_numpy(y)

        y = ep_sum(partial, spec.n_coded)
        out[rank] = y.numpy().tobytes()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,coded", [(2, 0), (3, 1)])
def test_gloo_ranks_sum_to_the_whole_layer(world, coded):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, coded, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    spec, ol, x, logits, T, k = _layer_case(coded)
    ref = ol.forward(x, True, logits, k)
    for r in range(world):
        got = np.frombuffer(res[r], dtype=np.float64).reshape(T, spec.hidden)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())
