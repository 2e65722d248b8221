"""Expert parallelism over the ranks of a torch.distributed process group.

Each rank owns a contiguous block of experts, routes every token (routing
is deterministic, so every rank builds the same tables), computes the pairs
of its own experts through the C ABI (exl3_moe_forward_experts, fp32
partial sums; rank 0 also adds the dense shared expert), and one all-reduce
per layer sums the partials; the sum is then rounded once, with the
residual, by exl3_round_output.  Page "GLM-5.3 Flash EXL3 for 2x DGX
Sparks", section Why the overlay exists: the split layer's partial outputs
are summed with one all-reduce per layer.

The host logic (ranges, reduction) lives in expert_range and ep_sum, which
take the partial-sum computation as a function, so it runs the same way with
the CUDA library or, in tests, with any other implementation of the sum.
"""
from __future__ import annotations


def expert_range(rank: int, world: int, num_experts: int):
    """[e0, e1): rank's contiguous block of experts (sizes differ by at most 1)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return rank * num_experts // world, (rank + 1) * num_experts // world


def _rank_world(group):
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return 0, 1
    return dist.get_rank(group), dist.get_world_size(group)


def ep_sum(partial, num_experts: int, group=None):
    """partial(e0, e1, with_shared) -> this rank's fp32 partial sum (a
    tensor); returns the sum over all ranks (every rank gets it)."""
    import torch.distributed as dist
    rank, world = _rank_world(group)
    e0, e1 = expert_range(rank, world, num_experts)
    y = partial(e0, e1, rank == 0)
    if world > 1:
        dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    return y


def moe_forward_ep(layer, x, logits, top_k: int, group=None, residual=None, path: int = 0,
                   stream=None):
    """One MoE layer with its experts split over the group's ranks; every
    rank returns the whole layer output [T, H] in x's dtype."""
    from .api import round_output
    y = ep_sum(lambda e0, e1, sh: layer.forward_experts(x, logits, top_k, e0, e1, with_shared=sh,
                                                         path=path, stream=stream),
               layer.n_coded, group)
    return round_output(y, x.dtype, residual=residual, stream=stream)
