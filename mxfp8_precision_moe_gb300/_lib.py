"""ctypes loader for libmxfp8moe.so (the sm_103a C ABI in include/mxfp8moe.h).

There is no fallback: if the library is missing or the device is not sm_103,
every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxfp8moe.so")

MXFP8_OK = 0
STATUS_NAMES = {
    0: "MXFP8_OK", 1: "MXFP8_ERR_NULL", 2: "MXFP8_ERR_SHAPE", 3: "MXFP8_ERR_ALIGN", 4: "MXFP8_ERR_LAYOUT",
    5: "MXFP8_ERR_ARCH", 6: "MXFP8_ERR_LAUNCH", 7: "MXFP8_ERR_OFFSETS", 8: "MXFP8_ERR_TIMEOUT",
    9: "MXFP8_ERR_DRIVER",
}
ROW, COL, BLOCK32X32 = 1, 2, 4
OPT_STOCHASTIC, OPT_HADAMARD_ROW, OPT_HADAMARD_COL = 1, 2, 4
SCALES_COMPACT, SCALES_BLOCKED = 0, 1
MAX_GROUPS = 1024

_lib = None


class Mxfp8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({describe(status)})")


def load():
    """Load the library (building it with nvcc first if it is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        from . import build as _build

        _build.build()
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I32, U32, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint, ctypes.c_int
    S = ctypes.c_int
    L.mxfp8_quantize_2d.argtypes = [P, I64, I64, U32, INT, P, I32, P, P, P, P, P, P]
    L.mxfp8_quantize_2d.restype = S
    L.mxfp8_quantize_2d_opts.argtypes = [P, I64, I64, U32, INT, P, I32, U32, ctypes.c_uint64, P, P, P, P, P, P]
    L.mxfp8_quantize_2d_opts.restype = S
    L.mxfp8_quantize_3d_experts.argtypes = [P, I32, I64, I64, U32, INT, P, P, P, P, P, P]
    L.mxfp8_quantize_3d_experts.restype = S
    for name in ("mxfp8_grouped_mm_fwd", "mxfp8_grouped_mm_dgrad", "mxfp8_grouped_mm_wgrad"):
        f = getattr(L, name)
        f.argtypes = [P, P, P, P, P, I32, I64, I64, I64, P, P, P]
        f.restype = S
    L.mxfp8_grouped_mm_swiglu_fwd.argtypes = [P, P, P, P, P, P, P, I32, I64, I64, I64, P, P, P, P, P, P, P, P]
    L.mxfp8_grouped_mm_swiglu_fwd.restype = S
    L.mxfp8_swiglu_bwd_quantize.argtypes = [P, P, P, I64, I64, P, I32, P, P, P, P, P, P, P, P, P, P]
    L.mxfp8_swiglu_bwd_quantize.restype = S
    L.mxfp8_grouped_mm_dgrad2.argtypes = [P, P, P, P, P, P, P, P, P, I32, I64, I64, I64, P, P, P]
    L.mxfp8_grouped_mm_dgrad2.restype = S
    L.mxfp8_scale_bytes.argtypes = [I64, I64, I32, INT]
    L.mxfp8_scale_bytes.restype = ctypes.c_size_t
    L.mxfp8_scale_bytes_colgroups.argtypes = [I64, I64, I32]
    L.mxfp8_scale_bytes_colgroups.restype = ctypes.c_size_t
    L.mxfp8_check_offsets.argtypes = [P, I32, I64, I32, P, P]
    L.mxfp8_check_offsets.restype = S
    L.mxfp8_status_string.argtypes = [S]
    L.mxfp8_status_string.restype = ctypes.c_char_p
    L.mxfp8_debug_wait_timeout.argtypes = [P, ctypes.c_uint64, P]
    L.mxfp8_debug_wait_timeout.restype = S
    _lib = L
    return L


def describe(status: int) -> str:
    try:
        return load().mxfp8_status_string(int(status)).decode()
    except OSError:
        return "library not loaded"


def check(status: int, where: str) -> None:
    if status != MXFP8_OK:
        raise Mxfp8Error(status, where)
