"""Python API over the C ABI.  PyTorch supplies device memory and streams only.

    layer = Layer(codes, suh, svh, K=(2, 2, 2))            # device tensors
    out = layer.forward(x, logits, top_k=8)                # one MoE layer
    ids, w, seg_offsets, seg_pairs = route(logits, top_k)  # routing tables
    dense = layer.decode_dense(expert, proj)               # fp16 [in][out]
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import check


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return _lib.EXL3_BF16
    if dt == torch.float16:
        return _lib.EXL3_F16
    raise TypeError(f"activations must be fp16 or bf16, not {dt}")


def _req(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")


class Layer:
    """One routed-expert MoE layer with EXL3 trellis-coded experts.

    codes[p]: uint16-bit tensors (torch.int16 or uint16 view) of shape
    [E, in/16, out/16, 16*K[p]]; suh[p]: fp16 [E, in]; svh[p]: fp16 [E, out];
    shared (optional): three fp16 dense [in, out] matrices.  p = 0 gate,
    1 up, 2 down.  hadamard: format v2 (the 128-point Hadamard rotation on
    both sides of every routed projection).  shared_coded: the last expert of
    the arrays is a trellis-coded shared expert (weight 1 for every token);
    the router then has E - 1 columns.  expert_K ([E][3] ints): a width per
    expert and projection; codes[p] is then a flat tensor of the experts'
    codes back to back (K is ignored).  act_fp8: FP8 x FP8 products (every
    routed projection's activation row quantised to E4M3 with an fp32 row
    scale; requires fp8_round).  The tensors must stay alive as long as the
    layer.
    """

    def __init__(self, codes, suh, svh, K, fp8_round=False, mcg_mult=0, shared=None,
                 hadamard=False, shared_coded=False, expert_K=None, act_fp8=False):
        E, H = suh[0].shape
        I = svh[0].shape[1]
        E -= int(bool(shared_coded))  # routed experts
        self.E, self.H, self.I = E, H, I
        self.K = tuple(int(k) for k in K)
        self._ek = None
        if expert_K is not None:
            import numpy as np
            self._ek = np.ascontiguousarray(np.asarray(expert_K, dtype=np.uint8))
            if self._ek.shape != (E + int(bool(shared_coded)), 3):
                raise ValueError(f"expert_K must be [{E + int(bool(shared_coded))}][3], "
                                 f"not {list(self._ek.shape)}")
        self._keep = [*codes, *suh, *svh] + (list(shared) if shared is not None else [])
        for t in self._keep:
            _req(t, "layer tensor")
        d = _lib.LayerDesc()
        d.num_experts, d.hidden, d.inter = E, H, I
        for p in range(3):
            d.K[p] = self.K[p]
            d.codes[p] = codes[p].data_ptr()
            d.suh[p] = suh[p].data_ptr()
            d.svh[p] = svh[p].data_ptr()
            d.shared_w[p] = shared[p].data_ptr() if shared is not None else None
        d.fp8_round = int(bool(fp8_round))
        d.mcg_mult = int(mcg_mult)
        d.hadamard = int(bool(hadamard))
        d.shared_coded = int(bool(shared_coded))
        d.expert_K = self._ek.ctypes.data if self._ek is not None else None
        d.act_fp8 = int(bool(act_fp8))
        h = ctypes.c_void_p()
        check(_lib.lib().exl3_layer_create(ctypes.byref(d), ctypes.byref(h)), "exl3_layer_create")
        self._h = h
        self._ws = None
        self._sc = bool(shared_coded)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.lib().exl3_layer_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def workspace_size(self, T: int, top_k: int) -> int:
        return int(_lib.lib().exl3_moe_workspace_size(self._h, T, top_k))

    def workspace(self, T: int, top_k: int, device=None) -> torch.Tensor:
        n = self.workspace_size(T, top_k)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8,
                                   device=device or self._keep[0].device)
        return self._ws

    def decode_dense(self, expert: int, proj: int, apply_side: bool = False, out=None,
                     stream=None) -> torch.Tensor:
        fin, fout = (self.I, self.H) if proj == 2 else (self.H, self.I)
        if out is None:
            out = torch.empty((fin, fout), dtype=torch.float16, device=self._keep[0].device)
        _req(out, "out", torch.float16)
        check(_lib.lib().exl3_decode_dense(self._h, expert, proj, int(apply_side), _ptr(out),
                                           _stream(stream)), "exl3_decode_dense")
        return out

    def forward(self, x, logits, top_k: int, out=None, residual=None, path: int = 0, ws=None,
                stream=None) -> torch.Tensor:
        _req(x, "x", (torch.float16, torch.bfloat16))
        _req(logits, "logits", torch.float32)
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        if ws is None:
            ws = self.workspace(T, top_k, x.device)
        st = _lib.lib().exl3_moe_forward_ex(self._h, _ptr(x), _dtype_code(x.dtype), _ptr(logits),
                                            T, top_k, _ptr(residual), _ptr(out), int(path),
                                            _ptr(ws), ws.numel(), _stream(stream))
        check(st, "exl3_moe_forward_ex")
        return out


    @property
    def n_coded(self) -> int:
        """Experts in the code arrays (routed, plus a coded shared expert)."""
        return self.E + int(self._sc)

    def forward_experts(self, x, logits, top_k: int, expert_begin: int, expert_end: int,
                        with_shared: bool = True, out=None, path: int = 0, ws=None,
                        stream=None) -> torch.Tensor:
        """fp32 [T, H] sum of the pairs whose expert is in [expert_begin,
        expert_end) (+ the dense shared expert when with_shared), unrounded."""
        _req(x, "x", (torch.float16, torch.bfloat16))
        _req(logits, "logits", torch.float32)
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.float32, device=x.device)
        _req(out, "out", torch.float32)
        if ws is None:
            ws = self.workspace(T, top_k, x.device)
        st = _lib.lib().exl3_moe_forward_experts(
            self._h, _ptr(x), _dtype_code(x.dtype), _ptr(logits), T, top_k, int(expert_begin),
            int(expert_end), int(bool(with_shared)), _ptr(out), int(path), _ptr(ws), ws.numel(),
            _stream(stream))
        check(st, "exl3_moe_forward_experts")
        return out


def round_output(y, dtype, residual=None, out=None, stream=None):
    """round(y + residual) to dtype (fp16 or bf16); y fp32 [T, H]."""
    _req(y, "y", torch.float32)
    if out is None:
        out = torch.empty(y.shape, dtype=dtype, device=y.device)
    T, H = y.shape
    check(_lib.lib().exl3_round_output(_ptr(y), T, H, _ptr(residual), _dtype_code(dtype), _ptr(out),
                                       _stream(stream)), "exl3_round_output")
    return out


def route(logits, top_k: int, ws=None, stream=None):
    """(ids [T,k] int32, w [T,k] fp32, seg_offsets [E+1] int32, seg_pairs [T*k] int32)."""
    _req(logits, "logits", torch.float32)
    T, E = logits.shape
    dev = logits.device
    ids = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    w = torch.empty((T, top_k), dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    pairs = torch.empty(max(T * top_k, 1), dtype=torch.int32, device=dev)
    n = int(_lib.lib().exl3_route_workspace_size(T, E, top_k))
    if ws is None:
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    check(_lib.lib().exl3_moe_route(_ptr(logits), T, E, top_k, _ptr(ids), _ptr(w), _ptr(off),
                                    _ptr(pairs), _ptr(ws), ws.numel(), _stream(stream)),
          "exl3_moe_route")
    return ids, w, off, pairs[:T * top_k]


def rmsnorm(x, eps: float = 1e-6, out=None, stream=None):
    _req(x, "x", (torch.float16, torch.bfloat16))
    if out is None:
        out = torch.empty_like(x)
    T, H = x.shape
    check(_lib.lib().exl3_rmsnorm(_ptr(x), _dtype_code(x.dtype), T, H, float(eps), _ptr(out),
                                  _stream(stream)), "exl3_rmsnorm")
    return out


def device_status(ws, stream=None) -> int:
    s = ctypes.c_int32(0)
    _lib.lib().exl3_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(s))
    return int(s.value)
