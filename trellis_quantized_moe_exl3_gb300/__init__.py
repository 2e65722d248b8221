"""GB300-native (sm_103a) EXL3 trellis-quantized routed-expert MoE layer.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/exl3.h``); this package only binds it.  ``synth`` holds the seeded
synthetic workloads.
"""
from . import synth  # noqa: F401


def _api():
    from . import api
    return api


def __getattr__(name):
    if name in ("Layer", "route", "rmsnorm", "device_status"):
        return getattr(_api(), name)
    raise AttributeError(name)
