"""Seeded synthetic inputs for the EXL3 MoE layer workloads.

This module only draws random numbers (numpy PCG64) and stores them in the
layer's storage formats; it holds none of the layer's arithmetic.  Both the
CUDA library's tests/benchmark and the CPU oracle consume exactly these arrays.

Each array has its own generator keyed by (seed, tag, ...), so a subset (one
expert's codes, say) can be regenerated without drawing everything before it.

Workloads (shapes of GLM-5.3-Flash's routed-expert MoE layer: 288 experts,
top-8, hidden 4096, expert intermediate 2048; pages "GLM-5.3-Flash · exlr8
(K2/K3/K4)" intro and Loading):
  tiny     8 experts, top-2, 256/128, K2, 16 fp16 tokens, seed 0
  decode   288 experts, top-8, K2, 4 bf16 tokens, + fp16 shared expert, seed 2
  verify3  same shape, K3, 32 tokens, logits N(0,1) + per-expert bias N(0,0.5), seed 3
  verify4  as verify3 with K4, seed 4
  prefill  K4 with the E4M3 rule, 7168 tokens, Zipf(1.1) popularity, seed 5
  long     4 layers K2,K3,K2,K4, 16384 tokens, Zipf popularity, seeds 6..9
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

TAG_CODES, TAG_SIDE, TAG_ACT, TAG_LOGITS, TAG_BIAS, TAG_PERM, TAG_GUMBEL, TAG_SHARED = range(1, 9)
TAG_WIDTHS = 9


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


@dataclass(frozen=True)
class LayerSpec:
    seed: int
    num_experts: int = 288
    hidden: int = 4096
    inter: int = 2048
    K: tuple = (2, 2, 2)
    fp8_round: bool = False
    shared: bool = False
    hadamard: bool = False  # format v2 (rotation on both sides); no effect on the draws
    shared_coded: bool = False  # one more coded expert (the shared one) after the routed ones
    expert_K: tuple | None = None  # per expert (gate, up, down) widths; codes then flat
    act_fp8: bool = False  # FP8 x FP8 products (E4M3 activation rows); no effect on the draws

    @property
    def n_coded(self) -> int:
        """Experts in the code and side-vector arrays."""
        return self.num_experts + int(self.shared_coded)

    def dims(self, proj: int):
        """(in_features, out_features) of projection 0=gate, 1=up, 2=down."""
        return (self.inter, self.hidden) if proj == 2 else (self.hidden, self.inter)

    def width(self, proj: int, expert: int) -> int:
        return self.expert_K[expert][proj] if self.expert_K else self.K[proj]

    def code_words_per_expert(self, proj: int, expert: int = 0) -> int:
        i, o = self.dims(proj)
        return (i // 16) * (o // 16) * 16 * self.width(proj, expert)


@dataclass(frozen=True)
class Workload:
    name: str
    layers: tuple
    T: int
    top_k: int
    act: str            # "f16" or "bf16"
    routing: str        # "normal", "normal_bias" or "zipf"
    seed: int
    residual: bool = False
    notes: str = field(default="")


def _spec(seed, **kw):
    return LayerSpec(seed=seed, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", (_spec(0, num_experts=8, hidden=256, inter=128, K=(2, 2, 2)),),
                     T=16, top_k=2, act="f16", routing="normal", seed=0),
    "decode": Workload("decode", (_spec(2, K=(2, 2, 2), shared=True),),
                       T=4, top_k=8, act="bf16", routing="normal", seed=2),
    "verify3": Workload("verify3", (_spec(3, K=(3, 3, 3)),),
                        T=32, top_k=8, act="bf16", routing="normal_bias", seed=3),
    "verify4": Workload("verify4", (_spec(4, K=(4, 4, 4)),),
                        T=32, top_k=8, act="bf16", routing="normal_bias", seed=4),
    "prefill": Workload("prefill", (_spec(5, K=(4, 4, 4), fp8_round=True),),
                        T=7168, top_k=8, act="bf16", routing="zipf", seed=5),
    "long": Workload("long", tuple(_spec(6 + l, K=(k, k, k)) for l, k in enumerate((2, 3, 2, 4))),
                     T=16384, top_k=8, act="bf16", routing="zipf", seed=6, residual=True),
}


# ---------------------------------------------------------------- weights
def expert_codes(spec: LayerSpec, proj: int, expert: int) -> np.ndarray:
    """Uniform-random uint16 code words [in/16][out/16][16K] of one expert."""
    i, o = spec.dims(proj)
    n = spec.code_words_per_expert(proj, expert)
    a = _rng(spec.seed, TAG_CODES, proj, expert).integers(0, 65536, size=n, dtype=np.uint16)
    return a.reshape(i // 16, o // 16, 16 * spec.width(proj, expert))


def mixed_widths(seed: int, n: int, choices=(3, 4)) -> tuple:
    """A width per expert and projection, drawn uniformly from `choices`
    (the 3.5 bpw mixed recipe: every routed tensor K3 or K4)."""
    w = _rng(seed, TAG_WIDTHS).choice(np.asarray(choices), size=(n, 3))
    return tuple(tuple(int(v) for v in row) for row in w)


def layer_codes(spec: LayerSpec, proj: int, out: np.ndarray | None = None) -> np.ndarray:
    """Code words of every expert, [E][in/16][out/16][16K]; with per-expert
    widths a flat array of the experts' codes back to back."""
    if spec.expert_K:
        return np.concatenate([expert_codes(spec, proj, e).reshape(-1) for e in range(spec.n_coded)])
    i, o = spec.dims(proj)
    shape = (spec.n_coded, i // 16, o // 16, 16 * spec.K[proj])
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    for e in range(spec.n_coded):
        out[e] = expert_codes(spec, proj, e)
    return out


def side_vectors(spec: LayerSpec, proj: int):
    """suh [E][in], svh [E][out]: fp16 bits of round(1 + 0.1 N(0,1))."""
    i, o = spec.dims(proj)
    g = _rng(spec.seed, TAG_SIDE, proj)
    suh = (1.0 + 0.1 * g.standard_normal((spec.n_coded, i))).astype(np.float16)
    svh = (1.0 + 0.1 * g.standard_normal((spec.n_coded, o))).astype(np.float16)
    return suh.view(np.uint16), svh.view(np.uint16)


def shared_weights(spec: LayerSpec):
    """Dense fp16 shared expert [in][out] per projection, N(0,1) entries."""
    ws = []
    for p in range(3):
        i, o = spec.dims(p)
        w = _rng(spec.seed, TAG_SHARED, p).standard_normal((i, o)).astype(np.float16)
        ws.append(w.view(np.uint16))
    return ws


# ---------------------------------------------------------------- activations
def _to_bf16_bits(a32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations(seed: int, T: int, H: int, dtype: str) -> np.ndarray:
    """N(0,1) activations as fp16 or bf16 bits [T][H]."""
    a = _rng(seed, TAG_ACT).standard_normal((T, H), dtype=np.float32)
    if dtype == "f16":
        return a.astype(np.float16).view(np.uint16)
    return _to_bf16_bits(a)


def router_logits(seed: int, T: int, E: int, kind: str) -> np.ndarray:
    """fp32 router logits [T][E].
    normal:      N(0,1)
    normal_bias: N(0,1) + bias_e, bias_e ~ N(0, 0.5) per expert
    zipf:        ln p_e + Gumbel(0,1), p_e proportional to rank_e^-1.1 with a
                 seeded rank permutation (Gumbel-top-k samples experts without
                 replacement in proportion to p)."""
    if kind == "normal":
        return _rng(seed, TAG_LOGITS).standard_normal((T, E), dtype=np.float32)
    if kind == "normal_bias":
        base = _rng(seed, TAG_LOGITS).standard_normal((T, E), dtype=np.float32)
        bias = _rng(seed, TAG_BIAS).normal(0.0, 0.5, size=E).astype(np.float32)
        return (base + bias[None, :]).astype(np.float32)
    if kind == "zipf":
        rank = _rng(seed, TAG_PERM).permutation(E) + 1
        logp = -1.1 * np.log(rank.astype(np.float64))
        logp -= np.log(np.exp(logp).sum())
        gum = _rng(seed, TAG_GUMBEL).gumbel(size=(T, E))
        return (logp[None, :] + gum).astype(np.float32)
    raise ValueError(kind)


def workload_inputs(wl: Workload, layer: int = 0):
    """(x bits [T][H] of the first layer, logits [T][E] of layer `layer`)."""
    spec = wl.layers[layer]
    x = activations(wl.seed, wl.T, spec.hidden, wl.act)
    logits = router_logits(spec.seed, wl.T, spec.num_experts, wl.routing)
    return x, logits
