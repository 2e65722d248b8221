"""The C-ABI library loads, exports every symbol include/exl3.h declares, and
rejects bad arguments on the host before touching the GPU.  No compute calls:
these run without a GPU."""
import ctypes

import pytest

from trellis_quantized_moe_exl3_gb300 import _lib, build


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.lib()


def test_every_declared_symbol_is_exported(L):
    names = _lib.declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), f"{n} declared in exl3.h but not exported"


def test_status_strings(L):
    for s in range(7):
        assert len(_lib.status_string(s)) > 0
    assert _lib.status_string(99) == "unknown status"


def _desc(E=8, H=256, I=128, K=(2, 2, 2)):
    d = _lib.LayerDesc()
    d.num_experts, d.hidden, d.inter = E, H, I
    for p in range(3):
        d.K[p] = K[p]
        d.codes[p] = 4096 * (p + 1)   # never dereferenced by create
        d.suh[p] = 4096 * (p + 4)
        d.svh[p] = 4096 * (p + 7)
        d.shared_w[p] = None
    return d


def _create(L, d):
    h = ctypes.c_void_p()
    return L.exl3_layer_create(ctypes.byref(d), ctypes.byref(h)), h


def test_layer_create_validation(L):
    assert L.exl3_layer_create(None, None) == _lib.EXL3_ERR_ARG
    assert _create(L, _desc(E=0))[0] == _lib.EXL3_ERR_SHAPE
    assert _create(L, _desc(E=2000))[0] == _lib.EXL3_ERR_SHAPE
    assert _create(L, _desc(H=200))[0] == _lib.EXL3_ERR_SHAPE
    assert _create(L, _desc(I=64))[0] == _lib.EXL3_ERR_SHAPE
    assert _create(L, _desc(K=(1, 1, 2)))[0] == _lib.EXL3_ERR_K
    assert _create(L, _desc(K=(2, 2, 5)))[0] == _lib.EXL3_ERR_K
    ek = (ctypes.c_uint8 * 24)(*([3, 4, 2] * 7 + [3, 5, 2]))       # a width table entry of 5
    d = _desc()
    d.expert_K = ctypes.cast(ek, ctypes.c_void_p)
    assert _create(L, d)[0] == _lib.EXL3_ERR_K
    d = _desc()
    d.mcg_mult = 2                                              # multiplier must be odd
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc()
    d.codes[1] = None
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc()
    d.codes[0] = 4096 + 2                                       # 16-byte alignment
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc()
    d.shared_w[0] = 8192                                        # all three or none
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    for field in ("suh", "svh"):                                 # side vectors aligned too
        d = _desc()
        getattr(d, field)[2] += 8
        assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc()
    d.hadamard = 2                                              # 0 (format v1) or 1 (v2)
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc()
    d.shared_coded = 2                                          # 0 or 1
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc()
    d.shared_coded = 1                                          # dense or coded, not both
    for p in range(3):
        d.shared_w[p] = 8192 * (p + 1)
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc(E=1024)
    d.shared_coded = 1                                          # 1025 experts in the tables
    assert _create(L, d)[0] == _lib.EXL3_ERR_SHAPE
    d = _desc()
    d.act_fp8 = 2                                               # 0 or 1
    d.fp8_round = 1
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG
    d = _desc()
    d.act_fp8 = 1                                               # FP8 operands need the E4M3 rule
    assert _create(L, d)[0] == _lib.EXL3_ERR_ARG


def test_route_validation_and_sizes(L):
    vp = ctypes.c_void_p
    n = L.exl3_route_workspace_size(100, 288, 8)
    assert n > 0 and L.exl3_route_workspace_size(100, 288, 8) == n
    assert L.exl3_route_workspace_size(1000, 288, 8) > n
    assert L.exl3_route_workspace_size(-1, 288, 8) == 0
    dummy = vp(4096)
    # top_k out of range
    assert L.exl3_moe_route(dummy, 4, 288, 0, dummy, dummy, dummy, dummy, dummy, 1 << 20,
                            None) == _lib.EXL3_ERR_ARG
    assert L.exl3_moe_route(dummy, 4, 8, 9, dummy, dummy, dummy, dummy, dummy, 1 << 20,
                            None) == _lib.EXL3_ERR_ARG
    assert L.exl3_moe_route(dummy, 4, 288, 17, dummy, dummy, dummy, dummy, dummy, 1 << 20,
                            None) == _lib.EXL3_ERR_ARG
    # bad shapes, missing workspace, too small workspace
    assert L.exl3_moe_route(dummy, -1, 288, 8, dummy, dummy, dummy, dummy, dummy, 1 << 20,
                            None) == _lib.EXL3_ERR_SHAPE
    assert L.exl3_moe_route(dummy, 4, 2000, 8, dummy, dummy, dummy, dummy, dummy, 1 << 20,
                            None) == _lib.EXL3_ERR_SHAPE
    assert L.exl3_moe_route(dummy, 1 << 27, 288, 8, dummy, dummy, dummy, dummy, dummy, 1 << 20,
                            None) == _lib.EXL3_ERR_SHAPE              # 2^30 pairs > 2^29
    assert L.exl3_moe_route(dummy, 4, 288, 8, dummy, dummy, dummy, dummy, None, 1 << 20,
                            None) == _lib.EXL3_ERR_WORKSPACE
    assert L.exl3_moe_route(dummy, 4, 288, 8, dummy, dummy, dummy, dummy, dummy, 16,
                            None) == _lib.EXL3_ERR_WORKSPACE


def test_forward_validation_without_layer(L):
    vp = ctypes.c_void_p
    assert L.exl3_moe_forward(None, vp(4096), 1, vp(4096), 4, 8, vp(8192), vp(4096), 1 << 20,
                              None) == _lib.EXL3_ERR_ARG
    assert L.exl3_moe_workspace_size(None, 4, 8) == 0
    assert L.exl3_rmsnorm(vp(4096), 7, 4, 256, 1e-6, vp(4096), None) == _lib.EXL3_ERR_ARG
    assert L.exl3_rmsnorm(vp(4096), 1, 4, 250, 1e-6, vp(4096), None) == _lib.EXL3_ERR_SHAPE
    s = ctypes.c_int32()
    assert L.exl3_get_device_status(None, None, ctypes.byref(s)) == _lib.EXL3_ERR_ARG


def test_expert_range_and_round_validation(L):
    vp = ctypes.c_void_p
    assert L.exl3_moe_forward_experts(None, vp(4096), 1, vp(4096), 4, 8, 0, 8, 1, vp(8192), 0,
                                      vp(4096), 1 << 20, None) == _lib.EXL3_ERR_ARG
    assert L.exl3_round_output(vp(4096), 4, 250, None, 1, vp(8192), None) == _lib.EXL3_ERR_SHAPE
    assert L.exl3_round_output(vp(4096), 4, 256, None, 7, vp(8192), None) == _lib.EXL3_ERR_ARG
    assert L.exl3_round_output(None, 4, 256, None, 1, vp(8192), None) == _lib.EXL3_ERR_ARG
    assert L.exl3_round_output(None, 0, 256, None, 1, None, None) == _lib.EXL3_OK


def test_quantize_rows_validation(L):
    vp = ctypes.c_void_p
    assert L.exl3_quantize_rows_e4m3(vp(4096), -1, 16, vp(4096), vp(4096), None) == _lib.EXL3_ERR_SHAPE
    assert L.exl3_quantize_rows_e4m3(None, 2, 16, vp(4096), vp(4096), None) == _lib.EXL3_ERR_ARG
    assert L.exl3_quantize_rows_e4m3(None, 0, 16, None, None, None) == _lib.EXL3_OK


def test_wait_fault_hook_validation(L):
    """The bounded-wait test hook checks its arguments on the host (and
    kernel 0 always clears it)."""
    assert L.exl3_test_set_wait_fault(3, 1, 1000000) == _lib.EXL3_ERR_ARG
    assert L.exl3_test_set_wait_fault(1, -1, 1000000) == _lib.EXL3_ERR_ARG
    assert L.exl3_test_set_wait_fault(1, 1, 10) == _lib.EXL3_ERR_ARG
    assert L.exl3_test_set_wait_fault(2, 1, 1 << 40) == _lib.EXL3_ERR_ARG
    assert L.exl3_test_set_wait_fault(1, 2, 2000000) == _lib.EXL3_OK
    assert L.exl3_test_set_wait_fault(0, 0, 0) == _lib.EXL3_OK
