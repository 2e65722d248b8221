"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs.  Decode and routing must match bit for bit; layer
outputs must meet max|gpu-oracle|/max|oracle| <= 2e-2 and relative Frobenius
error <= 5e-3."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from _helpers import HostLayer, act_to_f64, assert_layer_close, oracle_forward_parallel
from trellis_quantized_moe_exl3_gb300 import synth
from trellis_quantized_moe_exl3_gb300.api import device_status, rmsnorm, route

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _act(bits, act):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if act == "bf16" else torch.float16)


# ------------------------------------------------------------------ decode


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_dense_every_state(fp8):
    """65,536 tiles whose first word is the tile index: weight 0 of tile n has
    state n, so every trellis state is decoded; the whole 4096x4096 matrix
    must equal the oracle's bit for bit."""
    K = 2
    rng = np.random.default_rng(20)
    codes = rng.integers(0, 65536, size=(1, 256, 256, 16 * K), dtype=np.uint16)
    codes[0, :, :, 0] = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    spec = synth.LayerSpec(seed=0, num_experts=1, hidden=4096, inter=4096, K=(K, K, K),
                           fp8_round=fp8)
    hl = HostLayer(spec, codes=[codes, codes, codes])
    layer = hl.device()
    got = _u16(layer.decode_dense(0, 0))
    ref = oracle.decode_dense(codes[0], 4096, 4096, K, fp8_round=fp8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("K,fp8", [(3, False), (4, False), (3, True), (4, True), (2, True)])
def test_decode_dense_widths_and_side(K, fp8):
    spec = synth.LayerSpec(seed=30 + K, num_experts=3, hidden=256, inter=384, K=(K, K, K),
                           fp8_round=fp8)
    hl = HostLayer(spec)
    layer = hl.device(mult=0x2545F491)
    for e in range(3):
        for p in range(3):
            fin, fout = spec.dims(p)
            for side in (False, True):
                got = _u16(layer.decode_dense(e, p, apply_side=side))
                ref = oracle.decode_dense(hl.codes[p][e], fin, fout, K, mult=0x2545F491,
                                          fp8_round=fp8, suh=hl.suh[p][e] if side else None,
                                          svh=hl.svh[p][e] if side else None)
                assert np.array_equal(got, ref), (e, p, side)


def test_decode_dense_full_size_experts():
    wl = synth.WORKLOADS["prefill"]
    spec = wl.layers[0]
    codes = [np.stack([synth.expert_codes(spec, p, e) for e in (0, 287)]) for p in range(3)]
    small = synth.LayerSpec(seed=spec.seed, num_experts=2, K=spec.K, fp8_round=True)
    hl = HostLayer(small, codes=codes)
    layer = hl.device()
    for e in range(2):
        for p in range(3):
            fin, fout = small.dims(p)
            got = _u16(layer.decode_dense(e, p))
            ref = oracle.decode_dense(codes[p][e], fin, fout, spec.K[p], fp8_round=True)
            assert np.array_equal(got, ref), (e, p)


# ------------------------------------------------------------------ routing


def _route_cases():
    rng = np.random.default_rng(40)
    cases = []
    for name in ("tiny", "decode", "verify3", "prefill"):
        wl = synth.WORKLOADS[name]
        s = wl.layers[0]
        cases.append((name, synth.router_logits(s.seed, wl.T, s.num_experts, wl.routing), wl.top_k))
    wl = synth.WORKLOADS["long"]
    cases.append(("long", synth.router_logits(wl.layers[0].seed, wl.T, 288, "zipf"), 8))
    odd = rng.standard_normal((300, 40)).astype(np.float32)   # E not a multiple of 32, 3 chunks
    odd[1, 5] = odd[1, 30] = 50.0                               # tie
    odd[2, :] = 1.0                                             # all tied
    odd[3, 7] = np.nan
    odd[4, :] = -np.inf
    odd[5, :] = np.nan
    odd[6, :3] = np.inf
    odd[7, :] = 0.0
    odd[7, ::3] = -0.0                                          # +0 and -0 compare equal
    odd[8, :] = -1.0
    odd[8, 3], odd[8, 10] = 0.0, -0.0
    cases.append(("odd", odd, 5))
    zeros = rng.choice(np.array([0.0, -0.0, 1.0, -1.0], np.float32), (20, 288))
    cases.append(("signed_zeros", zeros, 8))                     # one chunk, many ties
    cases.append(("k1", rng.standard_normal((129, 288)).astype(np.float32), 1))
    cases.append(("k16", rng.standard_normal((77, 64)).astype(np.float32), 16))
    cases.append(("T1", rng.standard_normal((1, 288)).astype(np.float32), 8))
    cases.append(("E8k8", rng.standard_normal((33, 8)).astype(np.float32), 8))
    return cases


@pytest.mark.parametrize("case", _route_cases(), ids=lambda c: c[0])
def test_route_bit_exact(case):
    _, logits, k = case
    ids, w, off, pairs = route(torch.from_numpy(logits).cuda(), k)
    r_ids, r_w, r_off, r_pairs = oracle.route(logits, k)
    assert np.array_equal(ids.cpu().numpy(), r_ids)
    assert np.array_equal(w.cpu().numpy().view(np.int32), r_w.view(np.int32))
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(pairs.cpu().numpy(), r_pairs)


def test_route_empty():
    ids, w, off, pairs = route(torch.zeros((0, 288), dtype=torch.float32, device="cuda"), 8)
    assert (off.cpu().numpy() == 0).all()


# ------------------------------------------------------------------ layer


def _run_small(spec, T, top_k, act, path=0, residual=False, seed=50, routing="normal"):
    hl = HostLayer(spec)
    layer = hl.device()
    x = synth.activations(seed, T, spec.hidden, act)
    logits = synth.router_logits(seed, T, spec.num_experts, routing)
    xt = _act(x, act)
    res = _act(synth.activations(seed + 1, T, spec.hidden, act), act) if residual else None
    out = layer.forward(xt, torch.from_numpy(logits).cuda(), top_k, residual=res, path=path)
    torch.cuda.synchronize()
    ref = hl.oracle().forward(x, act == "bf16", logits, top_k)
    if residual:
        ref = ref + act_to_f64(res)
    return act_to_f64(out), ref, layer


@pytest.mark.parametrize("path", [0, 2], ids=["auto", "gemm"])
def test_forward_tiny_workload(path):
    wl = synth.WORKLOADS["tiny"]
    spec = wl.layers[0]
    hl = HostLayer(spec)
    layer = hl.device()
    x, logits = synth.workload_inputs(wl)
    out = layer.forward(_act(x, wl.act), torch.from_numpy(logits).cuda(), wl.top_k, path=path)
    torch.cuda.synchronize()
    ref = hl.oracle().forward(x, False, logits, wl.top_k)
    assert_layer_close(act_to_f64(out), ref)
    assert device_status(layer.workspace(wl.T, wl.top_k)) == 0


@pytest.mark.parametrize("K,fp8,shared,T,k,act", [
    ((2, 2, 3), False, False, 37, 4, "bf16"),
    ((3, 3, 4), False, True, 9, 3, "f16"),
    ((4, 4, 2), True, False, 20, 6, "bf16"),
    ((2, 2, 2), True, True, 1, 1, "bf16"),
    ((4, 4, 4), False, False, 64, 8, "bf16"),   # several token groups per expert
])
@pytest.mark.parametrize("path", [1, 2], ids=["gemv", "gemm"])
def test_forward_small_variants(K, fp8, shared, T, k, act, path):
    spec = synth.LayerSpec(seed=60 + sum(K), num_experts=10, hidden=384, inter=256, K=K,
                           fp8_round=fp8, shared=shared)
    out, ref, layer = _run_small(spec, T, k, act, path=path)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(T, k)) == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_forward_gemm_multi_tile(fp8):
    """Experts with more than 256 tokens (several tensor-core tiles, a ragged
    last tile), all three code widths, both paths."""
    spec = synth.LayerSpec(seed=75, num_experts=6, hidden=512, inter=384, K=(4, 4, 3), fp8_round=fp8)
    for path in (1, 2):
        out, ref, layer = _run_small(spec, 300, 4, "bf16", path=path)
        assert_layer_close(out, ref)
        assert device_status(layer.workspace(300, 4)) == 0


@pytest.mark.parametrize("T,k,routing,fp8", [
    (40, 4, "normal", False),    # every expert segment <= 64 tokens: small-tile kernel only
    (40, 4, "normal", True),
    (120, 4, "normal", False),   # segments of ~40-80 tokens: both small-tile widths (M 64, 128)
    (700, 4, "zipf", True),      # skewed: big tiles, ragged remainders, small tiles together
])
def test_forward_gemm_small_tiles(T, k, routing, fp8):
    """Tensor-core path on a shape whose H and I are multiples of 256, where
    segments (or their last tile) of <= 128 tokens take the swapped-operand
    small-tile kernel."""
    spec = synth.LayerSpec(seed=77, num_experts=8, hidden=512, inter=256, K=(3, 3, 4), fp8_round=fp8)
    out, ref, layer = _run_small(spec, T, k, "bf16", path=2, routing=routing)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(T, k)) == 0


def test_forward_residual():
    spec = synth.LayerSpec(seed=70, num_experts=6, hidden=256, inter=128, K=(3, 3, 3))
    out, ref, _ = _run_small(spec, 12, 2, "bf16", residual=True)
    assert_layer_close(out, ref)


def test_forward_zero_tokens():
    spec = synth.LayerSpec(seed=71, num_experts=4, hidden=128, inter=128, K=(2, 2, 2))
    layer = HostLayer(spec).device()
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    out = layer.forward(x, torch.zeros((0, 4), dtype=torch.float32, device="cuda"), 2)
    assert out.shape == (0, 128)


def test_rmsnorm_vs_oracle():
    x = synth.activations(80, 33, 512, "bf16")
    xt = _act(x, "bf16") * 7
    got = act_to_f64(rmsnorm(xt))
    xf = act_to_f64(xt)
    ref = np.stack([oracle.rmsnorm_row(r, 1e-6) for r in xf])
    assert np.abs(got - ref).max() <= 2 ** -7 * np.abs(ref).max()


def test_graph_capture_replays_same_output():
    spec = synth.LayerSpec(seed=72, num_experts=8, hidden=256, inter=128, K=(2, 2, 2), shared=True)
    hl = HostLayer(spec)
    layer = hl.device()
    T, k = 4, 2
    x = _act(synth.activations(72, T, 256, "bf16"), "bf16")
    lg = torch.from_numpy(synth.router_logits(72, T, 8, "normal")).cuda()
    ws = layer.workspace(T, k)
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(x, lg, k, out=out, ws=ws, stream=s)
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(x, lg, k, out=out, ws=ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)


# ------------------------------------------------------------------ format v2 (Hadamard)


@pytest.mark.parametrize("H,I,K,fp8,shared,T,k,routing,path", [
    (512, 256, (2, 2, 3), False, True, 37, 4, "normal", 1),   # GEMV, ragged token groups
    (384, 384, (4, 4, 4), True, False, 64, 8, "normal", 1),   # GEMV, odd block counts
    (512, 256, (3, 3, 4), False, False, 40, 4, "normal", 2),  # small-tile kernel, M 64
    (512, 256, (3, 3, 4), True, False, 120, 4, "normal", 2),  # both small-tile widths
    (512, 256, (4, 4, 3), False, True, 700, 4, "zipf", 2),    # big + small tiles
    (384, 384, (2, 2, 2), True, False, 300, 4, "normal", 2),  # big-tile kernel only
])
def test_forward_hadamard(H, I, K, fp8, shared, T, k, routing, path):
    """Format v2: the rotated input passes and the rotated epilogues of the
    GEMV and of both tensor-core kernels against the oracle, which rotates
    with the explicit 128x128 matrix."""
    spec = synth.LayerSpec(seed=90 + sum(K), num_experts=8, hidden=H, inter=I, K=K,
                           fp8_round=fp8, shared=shared, hadamard=True)
    out, ref, layer = _run_small(spec, T, k, "bf16", path=path, routing=routing)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(T, k)) == 0


# ------------------------------------------------------------------ coded shared expert


@pytest.mark.parametrize("E,H,I,K,fp8,had,T,k,routing,path", [
    (10, 384, 256, (2, 2, 3), False, False, 9, 3, "normal", 1),     # GEMV
    (8, 512, 256, (3, 3, 4), True, True, 40, 4, "normal", 1),       # GEMV, format v2
    (20, 256, 128, (2, 2, 2), False, False, 5, 16, "normal", 1),    # 17 pairs per token
    (8, 512, 256, (4, 4, 4), False, False, 120, 4, "normal", 2),    # shared segment: small tile
    (8, 512, 256, (3, 3, 2), False, True, 700, 4, "zipf", 2),       # shared segment: 2 big tiles
    (6, 256, 128, (2, 2, 2), False, False, 1, 1, "normal", 0),      # one token, top-1
])
def test_forward_shared_coded(E, H, I, K, fp8, had, T, k, routing, path):
    """A trellis-coded shared expert (the last expert of the arrays) routed
    as one more pair per token with weight 1, on both paths."""
    spec = synth.LayerSpec(seed=110 + sum(K), num_experts=E, hidden=H, inter=I, K=K,
                           fp8_round=fp8, hadamard=had, shared_coded=True)
    out, ref, layer = _run_small(spec, T, k, "bf16", path=path, routing=routing)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(T, k)) == 0


# ------------------------------------------------------------------ edge shapes


@pytest.mark.parametrize("E,H,I,K,had,T,k", [
    (1, 128, 128, (2, 2, 2), False, 5, 1),     # one expert, the smallest dimensions
    (6, 256, 128, (3, 3, 4), False, 10, 6),    # top_k = E: every expert for every token
    (4, 128, 128, (4, 4, 3), True, 7, 2),      # format v2 on single 128-blocks
])
@pytest.mark.parametrize("path", [1, 2], ids=["gemv", "gemm"])
def test_forward_edge_shapes(E, H, I, K, had, T, k, path):
    spec = synth.LayerSpec(seed=150 + E + k, num_experts=E, hidden=H, inter=I, K=K, hadamard=had)
    out, ref, layer = _run_small(spec, T, k, "bf16", path=path)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(T, k)) == 0


@pytest.mark.parametrize("path", [1, 2], ids=["gemv", "gemm"])
def test_forward_max_experts_and_top_k(path):
    """The largest expert count (1024: 32 logits per lane in the top-k, a
    thread per expert in the table scans) with the largest top_k (16)."""
    spec = synth.LayerSpec(seed=160, num_experts=1024, hidden=128, inter=128, K=(2, 2, 3))
    out, ref, layer = _run_small(spec, 40, 16, "bf16", path=path)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(40, 16)) == 0


# ------------------------------------------------------------------ mixed widths


@pytest.mark.parametrize("E,H,I,fp8,had,sc,T,k,routing,path", [
    (10, 384, 256, False, False, False, 37, 4, "normal", 1),   # GEMV
    (8, 512, 256, True, True, True, 40, 4, "normal", 1),       # GEMV, format v2, coded shared
    (8, 512, 256, False, False, False, 120, 4, "normal", 2),   # small tiles
    (8, 512, 256, True, False, True, 700, 4, "zipf", 2),       # big and small tiles
    (6, 384, 384, False, True, False, 300, 4, "normal", 2),    # big tiles only
])
def test_forward_mixed_widths(E, H, I, fp8, had, sc, T, k, routing, path):
    """A width per expert and projection (K2, K3 or K4; codes back to back):
    the expert kernels run once per width over device-built work lists."""
    seed = 130 + E + T
    spec = synth.LayerSpec(seed=seed, num_experts=E, hidden=H, inter=I, K=(2, 2, 2),
                           fp8_round=fp8, hadamard=had, shared_coded=sc,
                           expert_K=synth.mixed_widths(seed, E + int(sc), (2, 3, 4)))
    out, ref, layer = _run_small(spec, T, k, "bf16", path=path, routing=routing)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(T, k)) == 0
    hl = HostLayer(spec)
    for e in range(E + int(sc)):  # decode_dense at each expert's own width
        for p in range(3):
            fin, fout = spec.dims(p)
            o = sum(spec.code_words_per_expert(p, f) for f in range(e))
            words = hl.codes[p][o:o + spec.code_words_per_expert(p, e)]
            ref_d = oracle.decode_dense(words, fin, fout, spec.width(p, e), fp8_round=fp8)
            assert np.array_equal(_u16(layer.decode_dense(e, p)), ref_d)


@pytest.mark.parametrize("path", [1, 2], ids=["gemv", "gemm"])
def test_forward_gate_up_widths_differ(path):
    """Gate and up of different widths (K[0] != K[1]) without a table."""
    spec = synth.LayerSpec(seed=140, num_experts=8, hidden=512, inter=256, K=(3, 4, 2))
    out, ref, layer = _run_small(spec, 200 if path == 2 else 20, 4, "bf16", path=path)
    assert_layer_close(out, ref)


# ------------------------------------------------------------------ workloads


def _workload_parity(name, tokens_fn, path=0, **spec_changes):
    wl = synth.WORKLOADS[name]
    spec = dataclasses.replace(wl.layers[0], **spec_changes)
    hl = HostLayer(spec)
    layer = hl.device()
    x, logits = synth.workload_inputs(wl)
    out = layer.forward(_act(x, wl.act), torch.from_numpy(logits).cuda(), wl.top_k, path=path)
    torch.cuda.synchronize()
    assert device_status(layer.workspace(wl.T, wl.top_k)) == 0
    toks = tokens_fn(wl, logits)
    ref = oracle_forward_parallel(hl.oracle(), x, wl.act == "bf16", logits, wl.top_k, toks)
    got = act_to_f64(out)[toks]
    return assert_layer_close(got, ref)


def test_decode_workload_all_tokens():
    _workload_parity("decode", lambda wl, lg: list(range(wl.T)))


@pytest.mark.parametrize("name", ["verify3", "verify4"])
def test_verify_workloads_sampled(name):
    _workload_parity(name, lambda wl, lg: [0, 9, 22, 31])


def _prefill_tokens(wl, logits):
    ids, _, off, pairs = oracle.route(logits, wl.top_k)
    cnt = np.diff(off)
    e_small = int(np.argmin(np.where(cnt > 0, cnt, 1 << 30)))
    t_small = int(pairs[off[e_small]]) // wl.top_k
    e_big = int(np.argmax(cnt))
    t_big = int(pairs[off[e_big + 1] - 1]) // wl.top_k
    return sorted({0, wl.T - 1, t_small, t_big})


def test_prefill_workload_sampled():
    _workload_parity("prefill", _prefill_tokens)


def test_large_T_sampled():
    """131,072 tokens (1,048,576 pairs; the pages report their fused MoE
    failing at 98,304): workspace sizing and 64-bit indexing on the
    tensor-core path, sampled parity at both ends and the middle."""
    T, k = 131072, 8
    spec = synth.LayerSpec(seed=170, K=(2, 2, 2))
    hl = HostLayer(spec)
    layer = hl.device()
    x = synth.activations(171, T, spec.hidden, "bf16")
    logits = synth.router_logits(171, T, spec.num_experts, "zipf")
    out = layer.forward(_act(x, "bf16"), torch.from_numpy(logits).cuda(), k)
    torch.cuda.synchronize()
    assert device_status(layer.workspace(T, k)) == 0
    toks = [0, T // 2, T - 1]
    ref = oracle_forward_parallel(hl.oracle(), x, True, logits, k, toks)
    assert_layer_close(act_to_f64(out)[toks], ref)


def test_decode_workload_hadamard_all_tokens():
    """The decode workload's layer in format v2 (GEMV path, full size)."""
    _workload_parity("decode", lambda wl, lg: list(range(wl.T)), hadamard=True)


def test_verify_workload_mixed_widths_sampled():
    """The verify workload with every expert tensor K3 or K4 (the 3.5 bpw
    mixed recipe), full size, GEMV path."""
    wl = synth.WORKLOADS["verify3"]
    ek = synth.mixed_widths(wl.layers[0].seed, wl.layers[0].num_experts)
    _workload_parity("verify3", lambda wl, lg: [0, 9, 22, 31], expert_K=ek)


def test_decode_workload_shared_coded_all_tokens():
    """The decode workload with its shared expert trellis-coded as expert 288."""
    _workload_parity("decode", lambda wl, lg: list(range(wl.T)), shared=False, shared_coded=True)


def test_prefill_workload_hadamard_sampled():
    """The prefill workload's layer in format v2 (tensor-core path, full size)."""
    _workload_parity("prefill", _prefill_tokens, hadamard=True)


def test_long_workload_sampled():
    """Four stacked layers (K2, K3, K2, K4) with pre-RMSNorm and residual.

    The stated tolerance is a bound on each layer's output, so that is the
    acceptance: every layer is checked on the same input on both sides (the
    oracle takes the GPU's bf16 residual x_l for the sampled tokens and
    computes x_{l+1} = bf16(x_l + MoE(bf16(rmsnorm(x_l))))).  An independent
    4-layer oracle chain is not held to that bound: the difference a layer
    leaves is re-rounded to bf16, renormalised and pushed through the next
    roughly quadratic layer, so it grows by a factor that depends on the data
    and that no page fixes.  The chain is only required to stay finite."""
    wl = synth.WORKLOADS["long"]
    x0 = synth.activations(wl.seed, wl.T, 4096, "bf16")
    toks = [0, 5000, wl.T - 1]
    xt = _act(x0, "bf16")
    x_chain = x0[toks]
    for li, spec in enumerate(wl.layers):
        hl = HostLayer(spec)
        layer = hl.device()
        logits = synth.router_logits(spec.seed, wl.T, spec.num_experts, wl.routing)
        xn = rmsnorm(xt)
        nxt = layer.forward(xn, torch.from_numpy(logits).cuda(), wl.top_k, residual=xt)
        torch.cuda.synchronize()
        ol = hl.oracle()

        def oracle_layer(x_bits):
            xr = oracle.bf16_bits_to_f64(x_bits)
            xn_bits = np.stack([oracle.f64_to_bf16_bits(oracle.rmsnorm_row(r, 1e-6)) for r in xr])
            y = oracle_forward_parallel(ol, xn_bits, True, logits[toks], wl.top_k, range(len(toks)))
            return np.stack([oracle.f64_to_bf16_bits(r) for r in xr + y])

        x_in = xt.cpu().view(torch.int16).numpy().view(np.uint16)[toks]
        ref = oracle.bf16_bits_to_f64(oracle_layer(x_in))
        got = act_to_f64(nxt)[toks]
        assert_layer_close(got, ref)
        x_chain = oracle_layer(x_chain)
        xt = nxt
        del layer, hl
        torch.cuda.empty_cache()
    assert np.isfinite(act_to_f64(xt)[toks]).all()
    assert np.isfinite(oracle.bf16_bits_to_f64(x_chain)).all()


def test_forward_argument_errors_leave_output():
    """Argument errors of exl3_moe_forward_ex return their status before any
    launch and leave the output untouched."""
    import ctypes

    from trellis_quantized_moe_exl3_gb300 import _lib
    spec = synth.LayerSpec(seed=180, num_experts=6, hidden=256, inter=128, K=(2, 2, 2))
    hl = HostLayer(spec)
    layer = hl.device()
    T, k = 8, 2
    x = _act(synth.activations(181, T, spec.hidden, "bf16"), "bf16")
    lg = torch.from_numpy(synth.router_logits(181, T, spec.num_experts, "normal")).cuda()
    out = torch.full_like(x, 7.0)
    n = layer.workspace_size(T, k)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    L = _lib.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    bf = _lib.EXL3_BF16

    def call(x_=None, dt=bf, T_=T, k_=k, out_=None, path=0, ws_=ws, nbytes=n):
        xp = x_ if x_ is not None else p(x)
        op = out_ if out_ is not None else p(out)
        wp = p(ws_) if ws_ is not None else None
        return L.exl3_moe_forward_ex(layer.handle, xp, dt, p(lg), T_, k_, None, op, path, wp,
                                     nbytes, None)

    assert call(dt=7) == _lib.EXL3_ERR_ARG
    assert call(path=3) == _lib.EXL3_ERR_ARG
    assert call(T_=-1) == _lib.EXL3_ERR_SHAPE
    assert call(k_=0) == _lib.EXL3_ERR_ARG
    assert call(k_=spec.num_experts + 1) == _lib.EXL3_ERR_ARG
    assert call(out_=p(x)) == _lib.EXL3_ERR_ARG                       # out aliases x
    assert call(x_=ctypes.c_void_p(x.data_ptr() + 2)) == _lib.EXL3_ERR_ARG  # misaligned
    assert call(ws_=None) == _lib.EXL3_ERR_WORKSPACE
    assert call(nbytes=n - 1) == _lib.EXL3_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    assert call() == 0
    torch.cuda.synchronize()
    assert not bool((out == 7.0).all())


@pytest.mark.parametrize("scale", [1e-3, 1.0, 3e2])
@pytest.mark.parametrize("path,a8", [(2, False), (2, True), (1, False)], ids=["gemm", "gemm_fp8", "gemv"])
def test_forward_input_magnitudes(scale, path, a8):
    """Activations far from N(0, 1): the fp16 operand scales (per-row powers
    of two from the row maximum, and in the fused SwiGLU epilogue from the
    bound hb[e] |x|_1^2 on |h|) and the FP8 row scales must keep the layer
    within tolerance at any magnitude (|h| reaches ~1e9 at scale 300)."""
    spec = synth.LayerSpec(seed=250, num_experts=8, hidden=512, inter=256, K=(4, 4, 3),
                           fp8_round=True, act_fp8=a8)
    hl = HostLayer(spec)
    layer = hl.device()
    T, k = (300, 4) if path == 2 else (20, 4)
    x = synth.activations(251, T, spec.hidden, "bf16")
    xs = (oracle.bf16_bits_to_f64(x) * scale)
    x_bits = np.array([oracle.double_to_bf16(v) for v in xs.ravel()], np.uint16).reshape(xs.shape)
    logits = synth.router_logits(251, T, 8, "zipf")
    out = layer.forward(_act(x_bits, "bf16"), torch.from_numpy(logits).cuda(), k, path=path)
    torch.cuda.synchronize()
    ref = hl.oracle().forward(x_bits, True, logits, k)
    assert np.isfinite(act_to_f64(out)).all()
    assert_layer_close(act_to_f64(out), ref)
    assert device_status(layer.workspace(T, k)) == 0


# ------------------------------------------------------------------ FP8 x FP8 operands


@pytest.mark.parametrize("E,H,I,K,had,shared,sc,T,k,routing,path", [
    (10, 384, 256, (2, 2, 3), False, True, False, 37, 4, "normal", 1),   # GEMV
    (8, 512, 256, (4, 4, 4), True, False, True, 40, 4, "normal", 1),     # GEMV, v2, coded shared
    (8, 512, 256, (3, 3, 4), False, False, False, 40, 4, "normal", 2),   # small tiles, M 64
    (8, 512, 256, (4, 4, 2), False, True, False, 120, 4, "normal", 2),   # both small-tile widths
    (8, 512, 256, (4, 4, 3), False, False, True, 700, 4, "zipf", 2),     # big + small tiles
    (6, 384, 384, (2, 2, 2), False, False, False, 300, 4, "normal", 2),  # big tiles only
    (8, 512, 256, (4, 4, 4), True, False, False, 700, 4, "zipf", 2),     # v2, big + small
    (6, 512, 384, (3, 3, 4), True, False, False, 300, 4, "normal", 2),   # v2, big tiles only
])
def test_forward_act_fp8(E, H, I, K, had, shared, sc, T, k, routing, path):
    """FP8 x FP8 products (every routed projection's activation row
    quantised to E4M3 with an fp32 row scale): the tensor-core kernels on
    kind::f8f6f4 with E4M3 weights, and the GEMV with the same operand
    values, against the oracle in the same mode."""
    spec = synth.LayerSpec(seed=190 + sum(K), num_experts=E, hidden=H, inter=I, K=K,
                           fp8_round=True, hadamard=had, shared=shared, shared_coded=sc,
                           act_fp8=True)
    out, ref, layer = _run_small(spec, T, k, "bf16", path=path, routing=routing)
    assert_layer_close(out, ref)
    assert device_status(layer.workspace(T, k)) == 0


def _adversarial_rows(n=2048):
    """Rows whose quotients a / s land on E4M3 rounding boundaries, just
    beside them, and on E4M3 values, for exact and inexact row scales, plus
    plain N(0, 1) rows at several magnitudes and an all-zero row."""
    rng = np.random.default_rng(301)
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    vals = np.unique(np.abs(e4[np.isfinite(e4)]))
    mids = (vals[:-1] + vals[1:]) / 2.0                      # every rounding boundary
    rows = []
    for amax in (448.0, 1344.0, 1000.0, 0.37, 3.0e5):
        s = np.float32(np.float32(amax) / np.float32(448.0))
        targets = np.concatenate([mids, vals])
        a = (targets.astype(np.float64) * np.float64(s)).astype(np.float32)
        a = np.concatenate([a, np.nextafter(a, np.float32(np.inf)), np.nextafter(a, np.float32(0))])
        a = np.concatenate([a, -a])
        row = np.zeros(n, np.float32)
        row[:a.size] = a[:n - 1]
        row[n - 1] = np.float32(amax)                        # fixes the row's amax
        rows.append(row)
    for mag in (1e-3, 1.0, 7.0e4):
        rows.append((rng.standard_normal(n) * mag).astype(np.float32))
    rows.append(np.zeros(n, np.float32))
    return np.stack(rows)


def test_quantize_rows_e4m3_bit_exact():
    """The FP8 path's per-row activation quantisation (s = amax / 448 and
    q = E4M3(a / s), decided as IEEE fp32 divisions would) against the
    oracle's, bit for bit, on rows built to put quotients on and beside every
    E4M3 rounding boundary (where the kernel's reciprocal shortcut must fall
    back to the division)."""
    import ctypes

    from trellis_quantized_moe_exl3_gb300 import _lib
    a = _adversarial_rows()
    R, n = a.shape
    da = torch.from_numpy(a).cuda()
    q = torch.empty((R, n), dtype=torch.uint8, device="cuda")
    sc = torch.empty(R, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert _lib.lib().exl3_quantize_rows_e4m3(p(da), R, n, p(q), p(sc), None) == 0
    torch.cuda.synchronize()
    qv = q.cpu().view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    s_gpu = sc.cpu().numpy()
    for r in range(R):
        amax = np.float32(np.abs(a[r]).max())
        want_s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(0.0)
        assert s_gpu[r] == want_s, (r, s_gpu[r], want_s)
        got = qv[r] * np.float64(s_gpu[r])
        ref = oracle.quantize_row_e4m3(a[r].astype(np.float64))
        assert np.array_equal(got, ref), (r, int(np.sum(got != ref)))


def test_prefill_workload_act_fp8_sampled():
    """The prefill workload's layer (K4 with the E4M3 rule) with FP8 x FP8
    products, full size, against the oracle in the same mode."""
    _workload_parity("prefill", _prefill_tokens, act_fp8=True)


# ------------------------------------------------------------------ expert parallelism


@pytest.mark.parametrize("E,H,I,K,fp8,a8,shared,sc,T,k,routing,path", [
    (10, 384, 256, (2, 2, 3), False, False, True, False, 37, 4, "normal", 1),   # GEMV, dense shared
    (8, 512, 256, (3, 3, 4), False, False, False, True, 40, 4, "normal", 1),    # GEMV, coded shared
    (8, 512, 256, (4, 4, 3), False, False, True, False, 700, 4, "zipf", 2),     # big + small tiles
    (8, 512, 256, (4, 4, 4), True, True, False, True, 300, 4, "normal", 2),     # FP8, coded shared
])
def test_forward_experts_partition(E, H, I, K, fp8, a8, shared, sc, T, k, routing, path):
    """Expert-parallel shards on one GPU: forwards over a partition of the
    experts into three ranges (the dense shared expert in one of them), their
    fp32 partial sums added and rounded once, against the oracle's whole
    layer; an empty range gives zeros."""
    from trellis_quantized_moe_exl3_gb300.api import round_output
    from trellis_quantized_moe_exl3_gb300.ep import expert_range
    spec = synth.LayerSpec(seed=230 + sum(K), num_experts=E, hidden=H, inter=I, K=K,
                           fp8_round=fp8, act_fp8=a8, shared=shared, shared_coded=sc)
    hl = HostLayer(spec)
    layer = hl.device()
    x = synth.activations(231, T, H, "bf16")
    logits = synth.router_logits(231, T, E, routing)
    xt, lg = _act(x, "bf16"), torch.from_numpy(logits).cuda()
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    for r in range(3):
        e0, e1 = expert_range(r, 3, layer.n_coded)
        y += layer.forward_experts(xt, lg, k, e0, e1, with_shared=(r == 1), path=path)
    out = round_output(y, torch.bfloat16)
    torch.cuda.synchronize()
    assert_layer_close(act_to_f64(out), hl.oracle().forward(x, True, logits, k))
    assert device_status(layer.workspace(T, k)) == 0
    empty = layer.forward_experts(xt, lg, k, 2, 2, with_shared=False, path=path)
    torch.cuda.synchronize()
    assert bool((empty == 0).all())


def test_moe_forward_ep_single_rank():
    """moe_forward_ep without a process group (one rank: every expert) equals
    the plain forward's output within the layer tolerance, residual included."""
    from trellis_quantized_moe_exl3_gb300.ep import moe_forward_ep
    spec = synth.LayerSpec(seed=240, num_experts=8, hidden=256, inter=128, K=(2, 2, 2), shared=True)
    hl = HostLayer(spec)
    layer = hl.device()
    x = _act(synth.activations(241, 9, 256, "bf16"), "bf16")
    res = _act(synth.activations(242, 9, 256, "bf16"), "bf16")
    lg = torch.from_numpy(synth.router_logits(241, 9, 8, "normal")).cuda()
    a = moe_forward_ep(layer, x, lg, 2, residual=res)
    b = layer.forward(x, lg, 2, residual=res)
    torch.cuda.synchronize()
    assert_layer_close(act_to_f64(a), act_to_f64(b))


# ------------------------------------------------------------------ bounded waits


@pytest.mark.parametrize("kernel,T,routing", [(1, 700, "zipf"), (2, 40, "normal")],
                         ids=["big_tiles", "small_tiles"])
def test_bounded_wait_runs_out(kernel, T, routing):
    """A pipeline wait of a tensor-core kernel that nothing completes: the
    test hook makes the activation-load thread of one gate/up launch skip one
    K step (no copy is left in flight: the load is never issued), with a
    budget of 2,000,000 SM cycles (about 1 ms).  The forward must return,
    the device status must carry the timeout bit (4), and the next forward
    on the same workspace must be correct again."""
    from trellis_quantized_moe_exl3_gb300 import _lib
    spec = synth.LayerSpec(seed=77, num_experts=8, hidden=512, inter=256, K=(3, 3, 4))
    hl = HostLayer(spec)
    layer = hl.device()
    k = 4
    x = synth.activations(50, T, spec.hidden, "bf16")
    logits = synth.router_logits(50, T, spec.num_experts, routing)
    xt, lg = _act(x, "bf16"), torch.from_numpy(logits).cuda()
    ws = layer.workspace(T, k)
    L = _lib.lib()
    assert L.exl3_test_set_wait_fault(kernel, 3, 2_000_000) == 0
    try:
        layer.forward(xt, lg, k, ws=ws, path=2)
        status = device_status(ws)
    finally:
        assert L.exl3_test_set_wait_fault(0, 0, 0) == 0
    assert status & 4, f"status {status}: the wait did not report its timeout"
    out = layer.forward(xt, lg, k, ws=ws, path=2)
    torch.cuda.synchronize()
    assert device_status(ws) == 0
    assert_layer_close(act_to_f64(out), hl.oracle().forward(x, True, logits, k))
