"""Shared helpers of the GPU parity tests: build one layer from the seeded
generators both as device tensors (for the CUDA library) and as numpy arrays
(for the oracle), and compare outputs with the layer tolerance."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle
from trellis_quantized_moe_exl3_gb300 import synth

# Layer tolerance (fp32 accumulation): max|gpu - oracle| / max|oracle| and the
# relative Frobenius error.
MAX_REL = 2e-2
FRO_REL = 5e-3


class HostLayer:
    def __init__(self, spec: synth.LayerSpec, codes=None):
        self.spec = spec
        self.codes = codes if codes is not None else [synth.layer_codes(spec, p) for p in range(3)]
        sides = [synth.side_vectors(spec, p) for p in range(3)]
        self.suh = [s[0] for s in sides]
        self.svh = [s[1] for s in sides]
        self.shared = synth.shared_weights(spec) if spec.shared else None

    def oracle(self) -> oracle.Layer:
        s = self.spec
        return oracle.Layer(s.num_experts, s.hidden, s.inter, s.K, self.codes, self.suh, self.svh,
                            fp8_round=s.fp8_round, shared_w=self.shared, hadamard=s.hadamard,
                            shared_coded=s.shared_coded,
                            expert_K=np.array(s.expert_K, np.uint8) if s.expert_K else None,
                            act_fp8=s.act_fp8)

    def device(self, mult: int = 0):
        import torch
        from trellis_quantized_moe_exl3_gb300.api import Layer
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
        self.dev = dict(codes=[t(c) for c in self.codes], suh=[t(a).view(torch.float16) for a in self.suh],
                        svh=[t(a).view(torch.float16) for a in self.svh],
                        shared=[t(a).view(torch.float16) for a in self.shared] if self.shared else None)
        return Layer(self.dev["codes"], self.dev["suh"], self.dev["svh"], self.spec.K,
                     fp8_round=self.spec.fp8_round, mcg_mult=mult, shared=self.dev["shared"],
                     hadamard=self.spec.hadamard, shared_coded=self.spec.shared_coded,
                     expert_K=self.spec.expert_K, act_fp8=self.spec.act_fp8)


def oracle_forward_parallel(olayer: oracle.Layer, x_bits, is_bf16, logits, top_k, tokens,
                            workers=None):
    """Oracle rows for `tokens`, one token per thread (the C oracle releases the
    GIL; tokens are independent)."""
    tokens = list(tokens)
    workers = workers or min(len(tokens), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        rows = list(ex.map(lambda t: olayer.forward(x_bits, is_bf16, logits, top_k, tokens=[t])[0],
                           tokens))
    return np.stack(rows)


def act_to_f64(t):
    import torch
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_layer_close(gpu: np.ndarray, ref: np.ndarray, max_rel=MAX_REL, fro_rel=FRO_REL):
    d = gpu - ref
    m = np.abs(ref).max()
    fro = np.linalg.norm(d) / np.linalg.norm(ref)
    mx = np.abs(d).max() / m
    assert np.isfinite(gpu).all(), "non-finite output"
    assert mx <= max_rel, f"max rel error {mx:.3e} > {max_rel}"
    assert fro <= fro_rel, f"Frobenius rel error {fro:.3e} > {fro_rel}"
    return mx, fro
