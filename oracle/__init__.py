"""CPU oracle for the EXL3 trellis-quantized routed-expert MoE layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``trellis_quantized_moe_exl3_gb300``) and never imports
it; the two meet only at the seeded input generators.

The arithmetic lives in ``exl3_oracle.c`` (plain C, fp64, single thread).  This
module compiles it with gcc and exposes it through ctypes with numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exl3_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DEFAULT_MCG_MULT = 0x9E3779B1


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, no SIMD flags, no contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLayer(ctypes.Structure):
    _fields_ = [
        ("num_experts", ctypes.c_int), ("hidden", ctypes.c_int), ("inter", ctypes.c_int),
        ("K", ctypes.c_int * 3), ("fp8_round", ctypes.c_int), ("mult", ctypes.c_uint32),
        ("codes", ctypes.c_void_p * 3), ("suh", ctypes.c_void_p * 3),
        ("svh", ctypes.c_void_p * 3), ("shared_w", ctypes.c_void_p * 3),
        ("hadamard", ctypes.c_int), ("shared_coded", ctypes.c_int),
        ("expert_K", ctypes.c_void_p), ("act_fp8", ctypes.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u16p = ctypes.c_void_p
            L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_double.restype = ctypes.c_double
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_double_to_f16.argtypes = [ctypes.c_double]
            L.oracle_double_to_f16.restype = ctypes.c_uint16
            L.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            L.oracle_double_to_bf16.restype = ctypes.c_uint16
            L.oracle_e4m3_rne_sat.argtypes = [ctypes.c_double]
            L.oracle_e4m3_rne_sat.restype = ctypes.c_double
            L.oracle_tile_state.argtypes = [u16p, ctypes.c_int, ctypes.c_int]
            L.oracle_tile_state.restype = ctypes.c_uint32
            L.oracle_codebook_f16.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
            L.oracle_codebook_f16.restype = ctypes.c_uint16
            L.oracle_weight_f16.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int]
            L.oracle_weight_f16.restype = ctypes.c_uint16
            L.oracle_tile_position.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                               ctypes.POINTER(ctypes.c_int)]
            L.oracle_tile_position.restype = None
            L.oracle_decode_tile.argtypes = [u16p, ctypes.c_int, ctypes.c_uint32, ctypes.c_int, u16p]
            L.oracle_decode_tile.restype = None
            L.oracle_decode_dense.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_uint32, ctypes.c_int, u16p, u16p,
                                              ctypes.c_int, u16p]
            L.oracle_decode_dense.restype = None
            L.oracle_exp_route.argtypes = [ctypes.c_float]
            L.oracle_exp_route.restype = ctypes.c_float
            L.oracle_route_token.argtypes = [u16p, ctypes.c_int, ctypes.c_int, u16p, u16p]
            L.oracle_route_token.restype = None
            L.oracle_route.argtypes = [u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       u16p, u16p, u16p, u16p]
            L.oracle_route.restype = None
            L.oracle_moe_forward.argtypes = [ctypes.POINTER(OracleLayer), u16p, ctypes.c_int,
                                             u16p, ctypes.c_int, ctypes.c_int, u16p,
                                             ctypes.c_int, u16p]
            L.oracle_moe_forward.restype = ctypes.c_int
            L.oracle_expert_pair.argtypes = [ctypes.POINTER(OracleLayer), u16p, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_float, u16p]
            L.oracle_expert_pair.restype = ctypes.c_int
            L.oracle_shared_row.argtypes = [ctypes.POINTER(OracleLayer), u16p, ctypes.c_int, u16p]
            L.oracle_shared_row.restype = None
            L.oracle_rmsnorm_row.argtypes = [u16p, ctypes.c_int, ctypes.c_double, u16p]
            L.oracle_rmsnorm_row.restype = None
            L.oracle_hadamard128_entry.argtypes = [ctypes.c_int, ctypes.c_int]
            L.oracle_hadamard128_entry.restype = ctypes.c_double
            L.oracle_hadamard_blocks.argtypes = [u16p, ctypes.c_int]
            L.oracle_hadamard_blocks.restype = None
            L.oracle_quantize_row_e4m3.argtypes = [u16p, ctypes.c_int, u16p]
            L.oracle_quantize_row_e4m3.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------- scalars
def f16_to_double(h: int) -> float:
    return lib().oracle_f16_to_double(int(h))


def bf16_to_double(h: int) -> float:
    return lib().oracle_bf16_to_double(int(h))


def double_to_f16(v: float) -> int:
    return lib().oracle_double_to_f16(float(v))


def double_to_bf16(v: float) -> int:
    return lib().oracle_double_to_bf16(float(v))


def e4m3(v: float) -> float:
    return lib().oracle_e4m3_rne_sat(float(v))


def exp_route(x: float) -> float:
    return lib().oracle_exp_route(float(x))


# ---------------------------------------------------------------- format
def tile_state(words: np.ndarray, K: int, t: int) -> int:
    words = np.ascontiguousarray(words, dtype=np.uint16)
    assert words.size == 16 * K
    return lib().oracle_tile_state(_ptr(words), K, t)


def codebook_f16(s: int, mult: int = DEFAULT_MCG_MULT) -> int:
    return lib().oracle_codebook_f16(s, mult)


def weight_f16(s: int, mult: int = DEFAULT_MCG_MULT, fp8_round: bool = False) -> int:
    return lib().oracle_weight_f16(s, mult, int(fp8_round))


def tile_position(t: int):
    r, q = ctypes.c_int(), ctypes.c_int()
    lib().oracle_tile_position(t, ctypes.byref(r), ctypes.byref(q))
    return r.value, q.value


def decode_tile(words: np.ndarray, K: int, mult: int = DEFAULT_MCG_MULT,
                fp8_round: bool = False) -> np.ndarray:
    """fp16 bits [16 inputs][16 outputs] of one tile."""
    words = np.ascontiguousarray(words, dtype=np.uint16)
    assert words.size == 16 * K
    out = np.zeros((16, 16), dtype=np.uint16)
    lib().oracle_decode_tile(_ptr(words), K, mult, int(fp8_round), _ptr(out))
    return out


def decode_dense(codes: np.ndarray, in_f: int, out_f: int, K: int,
                 mult: int = DEFAULT_MCG_MULT, fp8_round: bool = False,
                 suh: np.ndarray | None = None, svh: np.ndarray | None = None) -> np.ndarray:
    """fp16 bits [in][out] of one projection of one expert."""
    codes = np.ascontiguousarray(codes, dtype=np.uint16)
    assert codes.size == (in_f // 16) * (out_f // 16) * 16 * K
    out = np.zeros((in_f, out_f), dtype=np.uint16)
    apply_side = suh is not None
    if apply_side:
        suh = np.ascontiguousarray(suh, dtype=np.uint16)
        svh = np.ascontiguousarray(svh, dtype=np.uint16)
        lib().oracle_decode_dense(_ptr(codes), in_f, out_f, K, mult, int(fp8_round),
                                  _ptr(suh), _ptr(svh), 1, _ptr(out))
    else:
        lib().oracle_decode_dense(_ptr(codes), in_f, out_f, K, mult, int(fp8_round),
                                  None, None, 0, _ptr(out))
    return out


# ---------------------------------------------------------------- rotation
def hadamard128_entry(i: int, j: int) -> float:
    return lib().oracle_hadamard128_entry(int(i), int(j))


def hadamard_blocks(v: np.ndarray) -> np.ndarray:
    """v . Hb for a vector whose length is a multiple of 128 (a copy)."""
    v = np.array(v, dtype=np.float64, copy=True)
    assert v.ndim == 1 and v.size % 128 == 0
    lib().oracle_hadamard_blocks(_ptr(v), v.size)
    return v


def quantize_row_e4m3(a: np.ndarray) -> np.ndarray:
    """The row as the FP8 x FP8 product's activation operand: q_i * s."""
    a = np.array(a, dtype=np.float64, copy=True)
    out = np.zeros_like(a)
    lib().oracle_quantize_row_e4m3(_ptr(a), a.size, _ptr(out))
    return out


# ---------------------------------------------------------------- routing
def route(logits: np.ndarray, top_k: int):
    """ids [T,k] int32, w [T,k] f32, seg_offsets [E+1] int32, seg_pairs [T*k] int32."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.zeros((T, top_k), np.int32)
    w = np.zeros((T, top_k), np.float32)
    off = np.zeros(E + 1, np.int32)
    pairs = np.zeros(T * top_k, np.int32)
    lib().oracle_route(_ptr(logits), T, E, top_k, _ptr(ids), _ptr(w), _ptr(off), _ptr(pairs))
    return ids, w, off, pairs


# ---------------------------------------------------------------- layer
class Layer:
    """Holds numpy arrays of one layer (host copies) and its oracle view."""

    def __init__(self, num_experts, hidden, inter, K, codes, suh, svh, fp8_round=False,
                 mult=DEFAULT_MCG_MULT, shared_w=None, hadamard=False, shared_coded=False,
                 expert_K=None, act_fp8=False):
        """num_experts routed experts; with shared_coded the code and side
        arrays hold num_experts + 1 experts, the last one the shared expert.
        expert_K ([experts][3] widths) gives every expert and projection its
        own width; codes[p] is then a flat array of the experts' codes back to
        back (K is ignored)."""
        self.arrays = []
        st = OracleLayer()
        st.num_experts, st.hidden, st.inter = num_experts, hidden, inter
        for p in range(3):
            st.K[p] = int(K[p])
        st.fp8_round = int(bool(fp8_round))
        st.mult = mult
        st.hadamard = int(bool(hadamard))
        st.shared_coded = int(bool(shared_coded))
        st.act_fp8 = int(bool(act_fp8))
        if expert_K is not None:
            ek = np.ascontiguousarray(expert_K, dtype=np.uint8)
            self.arrays.append(ek)
            st.expert_K = ek.ctypes.data
        else:
            st.expert_K = None
        for p in range(3):
            c = np.ascontiguousarray(codes[p], dtype=np.uint16)
            a = np.ascontiguousarray(suh[p], dtype=np.uint16)
            b = np.ascontiguousarray(svh[p], dtype=np.uint16)
            self.arrays += [c, a, b]
            st.codes[p] = c.ctypes.data
            st.suh[p] = a.ctypes.data
            st.svh[p] = b.ctypes.data
            if shared_w is not None:
                s = np.ascontiguousarray(shared_w[p], dtype=np.uint16)
                self.arrays.append(s)
                st.shared_w[p] = s.ctypes.data
            else:
                st.shared_w[p] = None
        self.st = st
        self.hidden = hidden

    def forward(self, x_bits: np.ndarray, x_is_bf16: bool, logits: np.ndarray, top_k: int,
                tokens=None) -> np.ndarray:
        """fp64 output rows [len(tokens)][H] (all tokens by default)."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T = x_bits.shape[0]
        if tokens is None:
            tokens = np.arange(T, dtype=np.int32)
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        y = np.zeros((tokens.size, self.hidden), np.float64)
        rc = lib().oracle_moe_forward(ctypes.byref(self.st), _ptr(x_bits), int(bool(x_is_bf16)),
                                      _ptr(logits), T, top_k, _ptr(tokens), tokens.size, _ptr(y))
        if rc != 0:
            raise MemoryError("oracle_moe_forward failed to allocate")
        return y


    def expert_pair(self, x_row_bits: np.ndarray, x_is_bf16: bool, expert: int,
                    weight: float) -> np.ndarray:
        """weight * expert(x_row) in fp64 (one (token, expert) pair)."""
        x_row_bits = np.ascontiguousarray(x_row_bits, dtype=np.uint16)
        r = np.zeros(self.hidden, np.float64)
        if lib().oracle_expert_pair(ctypes.byref(self.st), _ptr(x_row_bits), int(bool(x_is_bf16)),
                                    int(expert), float(weight), _ptr(r)) != 0:
            raise MemoryError("oracle_expert_pair failed to allocate")
        return r

    def shared_row(self, x_row_bits: np.ndarray, x_is_bf16: bool) -> np.ndarray:
        x_row_bits = np.ascontiguousarray(x_row_bits, dtype=np.uint16)
        y = np.zeros(self.hidden, np.float64)
        lib().oracle_shared_row(ctypes.byref(self.st), _ptr(x_row_bits), int(bool(x_is_bf16)), _ptr(y))
        return y


def rmsnorm_row(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    lib().oracle_rmsnorm_row(_ptr(x), x.size, eps, _ptr(out))
    return out


def f16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Vectorised exact fp16 -> double through the oracle's scalar rule table."""
    table = np.array([f16_to_double(h) for h in range(65536)], dtype=np.float64) \
        if not hasattr(f16_bits_to_f64, "_t") else f16_bits_to_f64._t
    f16_bits_to_f64._t = table
    return table[np.asarray(a, dtype=np.uint16)]


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    table = np.array([bf16_to_double(h) for h in range(65536)], dtype=np.float64) \
        if not hasattr(bf16_bits_to_f64, "_t") else bf16_bits_to_f64._t
    bf16_bits_to_f64._t = table
    return table[np.asarray(a, dtype=np.uint16)]


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return np.array([double_to_bf16(v) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)
