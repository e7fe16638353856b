"""ctypes view of ``libgdn_qdq.so`` (the C ABI in ``include/gdn_qdq.h``).

Loading never falls back to anything: if the library is missing the import
of a compute entry point raises, naming the build step.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn_qdq.so")

QDQ_MODES = {"none": 0, "e4m3": 1, "int8": 2}
DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2}

STATUS = {
    0: "GDN_OK", -1: "GDN_ERR_INVALID_ARG", -2: "GDN_ERR_UNSUPPORTED_DTYPE",
    -3: "GDN_ERR_UNSUPPORTED_SHAPE", -4: "GDN_ERR_UNSUPPORTED_MODE",
    -5: "GDN_ERR_WORKSPACE_TOO_SMALL", -6: "GDN_ERR_CUDA", -7: "GDN_ERR_MISALIGNED",
}

# Every symbol the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


class GdnProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("T", ctypes.c_int64),
        ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
        ("N", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p), ("scale", ctypes.c_float),
        ("state_mode", ctypes.c_int32), ("w_mode", ctypes.c_int32), ("block_v", ctypes.c_int32),
        ("chunk", ctypes.c_int32), ("dtype", ctypes.c_int32), ("solve", ctypes.c_int32),
        ("solve_degree", ctypes.c_int32), ("save_ctx", ctypes.c_int32),
    ]


_PP = ctypes.POINTER(GdnProblem)

READOUTS = {"pre": 0, "post": 1}


class GdnDecodeProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("T", ctypes.c_int64),
        ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
        ("scale", ctypes.c_float), ("state_mode", ctypes.c_int32), ("block_v", ctypes.c_int32),
        ("readout", ctypes.c_int32), ("dtype", ctypes.c_int32),
    ]


_DP = ctypes.POINTER(GdnDecodeProblem)


class GdnTwoPrecisionProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("T", ctypes.c_int64),
        ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32), ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
        ("N", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p), ("scale", ctypes.c_float),
        ("read_mode", ctypes.c_int32), ("flush", ctypes.c_int32), ("dtype", ctypes.c_int32),
    ]


_TP = ctypes.POINTER(GdnTwoPrecisionProblem)
SIGNATURES = {
    "gdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gdn_abi_version": (ctypes.c_int, []),
    "gdn_device_error": (ctypes.c_int, [ctypes.c_int]),
    "gdn_validate": (ctypes.c_int, [_PP]),
    "gdn_num_chunk_slots": (ctypes.c_int64, [_PP]),
    "gdn_ctx_bytes": (_SZ, [_PP]),
    "gdn_ctx_offset": (_I64, [_PP, ctypes.c_int]),
    "gdn_chunk_fwd_qdq": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_bwd_workspace_bytes": (_SZ, [_PP]),
    "gdn_chunk_bwd_ste": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                         _P, _P, _P, _SZ, _P]),
    "gdn_chunk_bwd_ste_noalloc": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                 _P, _P, _P, _P]),
    "fake_qdq_e4m3": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "fake_qdq_int8": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "kda_recurrent_fwd_qdq": (ctypes.c_int, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_decode_validate": (ctypes.c_int, [_DP]),
    "gdn_decode_qdq": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_two_precision_validate": (ctypes.c_int, [_TP]),
    "gdn_two_precision_anchor_bytes": (_SZ, [_TP]),
    "gdn_two_precision_fwd": (ctypes.c_int, [_TP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gdn_two_precision_bwd_workspace_bytes": (_SZ, [_TP]),
    "gdn_two_precision_bwd": (ctypes.c_int, [_TP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                             _P, _P, _P, _SZ, _P]),
}

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s returned %d (%s)" % (fn, status, STATUS.get(status, "unknown")))


def load():
    """Load the library (building it first if absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            from . import build as _build
            if not os.path.exists(LIB_PATH) or _build._stale():
                try:
                    _build.build()
                except Exception as exc:  # no silent fallback: the CUDA library is required
                    raise RuntimeError(
                        "libgdn_qdq.so is missing and could not be built "
                        "(python -m gated_delta_rule_54_gb300.build): %s" % exc) from exc
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def check(fn: str, status: int):
    if status != 0:
        raise GdnError(fn, status)
