"""ctypes binding to libexl3_gb300.so (the C ABI of include/exl3.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  There is no fallback: if the library is missing, importing the API
raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import LIB_PATH

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "exl3.h")

EXL3_OK, EXL3_ERR_ARG, EXL3_ERR_SHAPE, EXL3_ERR_K, EXL3_ERR_WORKSPACE, EXL3_ERR_CUDA, \
    EXL3_ERR_DEVICE = range(7)
EXL3_F16, EXL3_BF16 = 0, 1
EXL3_PATH_AUTO, EXL3_PATH_GEMV, EXL3_PATH_GEMM = 0, 1, 2
EXL3_NUM_STAGE_EVENTS = 8
STAGE_NAMES = ("route", "gather", "gate_up", "down_prep", "down", "shared", "combine")


class LayerDesc(ctypes.Structure):
    _fields_ = [
        ("num_experts", ctypes.c_int), ("hidden", ctypes.c_int), ("inter", ctypes.c_int),
        ("K", ctypes.c_int * 3), ("fp8_round", ctypes.c_int), ("mcg_mult", ctypes.c_uint32),
        ("codes", ctypes.c_void_p * 3), ("suh", ctypes.c_void_p * 3),
        ("svh", ctypes.c_void_p * 3), ("shared_w", ctypes.c_void_p * 3),
        ("hadamard", ctypes.c_int), ("shared_coded", ctypes.c_int),
        ("expert_K", ctypes.c_void_p), ("act_fp8", ctypes.c_int),
    ]


class Exl3Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def declared_functions():
    """Names of the functions include/exl3.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(exl3_[a-z_0-9]+)\s*\(", src)))


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "trellis_quantized_moe_exl3_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.exl3_layer_create.argtypes = [ctypes.POINTER(LayerDesc), ctypes.POINTER(vp)]
    L.exl3_layer_create.restype = i
    L.exl3_layer_destroy.argtypes = [vp]
    L.exl3_layer_destroy.restype = None
    L.exl3_decode_dense.argtypes = [vp, i, i, i, vp, vp]
    L.exl3_decode_dense.restype = i
    L.exl3_route_workspace_size.argtypes = [i, i, i]
    L.exl3_route_workspace_size.restype = sz
    L.exl3_moe_route.argtypes = [vp, i, i, i, vp, vp, vp, vp, vp, sz, vp]
    L.exl3_moe_route.restype = i
    L.exl3_moe_route_static.argtypes = [vp, i, i, i, vp, vp, vp, vp, vp]
    L.exl3_moe_route_static.restype = i
    L.exl3_moe_workspace_size.argtypes = [vp, i, i]
    L.exl3_moe_workspace_size.restype = sz
    L.exl3_moe_forward.argtypes = [vp, vp, i, vp, i, i, vp, vp, sz, vp]
    L.exl3_moe_forward.restype = i
    L.exl3_moe_forward_ex.argtypes = [vp, vp, i, vp, i, i, vp, vp, i, vp, sz, vp]
    L.exl3_moe_forward_ex.restype = i
    L.exl3_moe_forward_experts.argtypes = [vp, vp, i, vp, i, i, i, i, i, vp, i, vp, sz, vp]
    L.exl3_moe_forward_experts.restype = i
    L.exl3_round_output.argtypes = [vp, i, i, vp, i, vp, vp]
    L.exl3_round_output.restype = i
    L.exl3_rmsnorm.argtypes = [vp, i, i, i, ctypes.c_float, vp, vp]
    L.exl3_rmsnorm.restype = i
    L.exl3_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    L.exl3_get_device_status.restype = i
    L.exl3_layer_set_stage_events.argtypes = [vp, vp, i]
    L.exl3_layer_set_stage_events.restype = i
    L.exl3_launch_count.argtypes = []
    L.exl3_launch_count.restype = ctypes.c_uint64
    L.exl3_quantize_rows_e4m3.argtypes = [vp, i, i, vp, vp, vp]
    L.exl3_quantize_rows_e4m3.restype = i
    L.exl3_test_set_wait_fault.argtypes = [i, i, ctypes.c_longlong]
    L.exl3_test_set_wait_fault.restype = i
    L.exl3_status_string.argtypes = [i]
    L.exl3_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def status_string(s: int) -> str:
    return lib().exl3_status_string(int(s)).decode()


def check(status: int, what: str):
    if status != EXL3_OK:
        raise Exl3Error(status, what)
