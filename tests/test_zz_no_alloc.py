"""exl3_moe_route_static, the routing entry point that allocates nothing.

Some callers cannot allocate device memory: a plugin whose host framework
owns every device allocation and passes in only the call's tensors, or a
loop that must not call cudaMalloc because it can synchronise the device.
exl3_moe_route_static serves them by keeping its routing scratch in a
library-owned device array.  This test calls it through the C ABI twice in a
row, in both orders of a large (multi-chunk) and a small case, so that each
second call starts from the first call's leftovers, and requires every
result to equal, bit for bit, both the CPU oracle's routing and what
exl3_moe_route computes from the same logits with its own workspace (routing
is integer and index work plus an fp32 softmax in a fixed order, so the
tolerance of the routing tests is exact equality).

The file name sorts last so that a run stopping at its first failure has run
every other test before this one."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from trellis_quantized_moe_exl3_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

# (T, E, top_k, logit distribution): a multi-chunk case (scan + scatter
# kernels), then a smaller single-chunk one
CASES = [(2048, 288, 8, "zipf"), (77, 256, 8, "normal")]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(T, E, k):
    return (torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
            torch.full((T, k), -7.0, dtype=torch.float32, device="cuda"),
            torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((max(T * k, 1),), -7, dtype=torch.int32, device="cuda"))


def _route_with_workspace(logits, k):
    T, E = logits.shape
    ids, w, off, pairs = _outputs(T, E, k)
    n = int(_lib.lib().exl3_route_workspace_size(T, E, k))
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
    st = _lib.lib().exl3_moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(off),
                                   _ptr(pairs), _ptr(ws), ws.numel(), None)
    assert st == 0, _lib.status_string(st)
    return ids, w, off, pairs


@pytest.mark.parametrize("order", [(0, 1), (1, 0)], ids=["large_then_small", "small_then_large"])
def test_route_static_matches_oracle_and_workspace_route_twice(order):
    L = _lib.lib()
    cases = [CASES[i] for i in order]
    inputs = [synth.router_logits(90 + i, CASES[i][0], CASES[i][1], CASES[i][3]) for i in order]
    d_inputs = [torch.from_numpy(lg).cuda() for lg in inputs]
    results = []
    for (T, E, k, _), lg in zip(cases, d_inputs):  # back to back on one stream
        outs = _outputs(T, E, k)
        st = L.exl3_moe_route_static(_ptr(lg), T, E, k, *map(_ptr, outs), None)
        assert st == 0, _lib.status_string(st)
        results.append(outs)
    torch.cuda.synchronize()
    for (T, E, k, _), lg, d_lg, got in zip(cases, inputs, d_inputs, results):
        ref = oracle.route(lg, k)
        got_np = [t.cpu().numpy() for t in got]
        got_np[3] = got_np[3][:T * k]
        for g, r in zip(got_np, ref):
            assert np.array_equal(g.view(np.int32).ravel(), np.asarray(r).view(np.int32).ravel())
        want = _route_with_workspace(d_lg, k)
        torch.cuda.synchronize()
        for g, r in zip(got, want):
            assert torch.equal(g.view(torch.int32), r.view(torch.int32))


def test_route_static_rejects_oversize():
    """Sizes beyond the static array return EXL3_ERR_SHAPE before any launch
    and leave the outputs untouched."""
    L = _lib.lib()
    T, E, k = 8192, 1024, 16
    assert L.exl3_route_workspace_size(T, E, k) > 1 << 20
    logits = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    outs = _outputs(T, E, k)
    st = L.exl3_moe_route_static(_ptr(logits), T, E, k, *map(_ptr, outs), None)
    assert st == 2, _lib.status_string(st)
    torch.cuda.synchronize()
    assert bool((outs[2] == -7).all())
