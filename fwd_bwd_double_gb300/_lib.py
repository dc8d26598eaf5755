"""ctypes loading of libfbd.so and the C-ABI prototypes (mirrors include/fbd.h)."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfbd.so")

ATTN_F32 = 0
ATTN_BF16 = 1
ATTN_ROW_PASS = 1
ATTN_COL_PASS = 2

STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_ALIGNMENT",
    4: "ATTN_ERR_WORKSPACE", 5: "ATTN_ERR_LAUNCH", 6: "ATTN_ERR_TIMEOUT", 7: "ATTN_ERR_DEVICE",
}


def status_name(code: int) -> str:
    return STATUS_NAMES.get(int(code), f"status {code}")


class FbdError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = int(status)
        super().__init__(f"{status_name(status)}: {detail}")


class AttnDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64), ("d", ctypes.c_int64),
                ("scale", ctypes.c_float), ("causal", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("group", ctypes.c_int32), ("window", ctypes.c_int32), ("seg_lo", ctypes.c_void_p),
                ("seg_hi", ctypes.c_void_p)]


_P = ctypes.c_void_p
_D = ctypes.POINTER(AttnDesc)
PROTOTYPES = {
    "attn_fwd": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P]),
    "attn_bwd_workspace_bytes": (ctypes.c_size_t, [_D, ctypes.c_int]),
    "attn_bwd": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "attn_bob_workspace_bytes": (ctypes.c_size_t, [_D, ctypes.c_int]),
    "attn_bob": (ctypes.c_int, [_D] + [_P] * 13 + [ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "attn_bwd_passes": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_size_t,
                                        ctypes.c_int, _P]),
    "attn_bob_passes": (ctypes.c_int, [_D] + [_P] * 13 + [ctypes.c_int, _P, ctypes.c_size_t, ctypes.c_int, _P]),
    "attn_bob_static": (ctypes.c_int, [_D] + [_P] * 13 + [_P]),
    "attn_bwd_projected_dS": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P]),
    "attn_segment_bounds": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P]),
    "attn_device_status": (ctypes.c_int, [_P]),
    "attn_check_wait_timeout": (ctypes.c_int, [_P]),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_version": (ctypes.c_char_p, []),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libfbd.so not built ({path}); run `python -c 'import __graft_entry__ as g; g.build()'`")
    dll = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(dll, name)
        fn.restype = res
        fn.argtypes = args
    return dll


lib = load()
