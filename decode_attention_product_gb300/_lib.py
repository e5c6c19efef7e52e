"""ctypes binding of libaqpq.so (the C ABI in include/aqpq.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  The library is loaded on first use; if it is missing or fails to
load, the call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libaqpq.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "_build_debug", "libaqpq.so")   # AQ_DEBUG_CHECKS build

AQ_OK = 0
STATUS_NAMES = {0: "AQ_OK", 1: "AQ_ERR_INVALID_ARGUMENT", 2: "AQ_ERR_UNSUPPORTED",
                3: "AQ_ERR_WORKSPACE_TOO_SMALL", 4: "AQ_ERR_CUDA"}
DEV_BAD_PAGE, DEV_BAD_LENGTH, DEV_BAD_SET, DEV_TIMEOUT, DEV_INVARIANT = 1, 2, 4, 8, 16
STEP_OVERLAP = 1
STEP_E4M3 = 2

# every symbol include/aqpq.h declares, with its ctypes signature
P = ctypes.c_void_p
i32, i64, sz, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "aq_status_string": ([i32], ctypes.c_char_p),
    "aq_last_error_message": ([], ctypes.c_char_p),
    "aq_version": ([], ctypes.c_char_p),
    "aq_set_wait_limit_ns": ([ctypes.c_uint64], ctypes.c_uint64),
    "aq_fit_codebooks": ([P, i64, i32, i32, P, P, P, P], i32),
    "aq_kmeans_step": ([P, i64, i32, P, P, P, P, P], i32),
    "aq_refine_codebooks": ([P, i64, i32, i32, P, P, P, P], i32),
    "aq_codebooks_to_e4m3": ([i64, P, P, P], i32),
    "aq_codebooks_from_e4m3": ([i64, P, P, P], i32),
    "aq_encode_append": ([P, i32, i32, P, P, P, P, i64, P, i64, P, P], i32),
    "aq_decode_plan": ([P, i32, i32, i32, i32, i32, i32, P, P, P], i32),
    "aq_decode_attention": ([P, i32, i32, i32, P, P, i64, P, i64, P, P, i32, P, i32, f32, i32,
                             P, P, sz, P, P], i32),
    "aq_decode_attention_fp16": ([P, i32, i32, i32, P, P, i64, P, i32, P, i32, f32, i32, P, P, sz,
                                  P, P], i32),
    "aq_decode_step": ([P, i32, i32, i32, P, P, P, i64, P, i64, P, P, i32, P, i32, f32, i32, i32,
                        P, P, sz, P, P], i32),
    "aq_decode_step_host_staging": ([i32, i32, i32], sz),
    "aq_decode_step_host": ([P, i32, i32, i32, P, P, P, i64, P, i64, P, P, i32, P, i32, f32, i32, i32, P, P, sz, P,
                             sz, P, P], i32),
    "aq_decode_step_mixed": ([P, i32, i32, i32, i32, P, P, P, i64, P, i64, P, i64, P, P, i32, P, i32, f32,
                              i32, P, P, sz, P, P], i32),
    "aq_decode_step_mixed_workspace": ([P, i32, i32, i32, i32, i32, P], i32),
    "aq_decode_attention_noalloc": ([P, i32, i32, i32, P, P, i64, P, i64, P, P, i32, P, i32, f32,
                                     i32, P, P, P], i32),
}


class PQConfig(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("num_subspaces", ctypes.c_int32),
                ("num_codewords", ctypes.c_int32), ("page_size", ctypes.c_int32)]


class AQError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load libaqpq.so (once).  Raises if it is missing.  The environment
    variable AQPQ_LIB names another build of the library to load instead;
    AQPQ_DEBUG_CHECKS=1 selects the AQ_DEBUG_CHECKS build."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or os.environ.get("AQPQ_LIB") or (
            DEBUG_LIB_PATH if os.environ.get("AQPQ_DEBUG_CHECKS") == "1" else LIB_PATH)
        if not os.path.exists(p):
            raise RuntimeError(
                f"libaqpq.so not found at {p}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def check(status: int, where: str) -> None:
    if status != AQ_OK:
        detail = ""
        if status == 4:
            detail = load().aq_last_error_message().decode()
        raise AQError(status, where, detail)


def config(num_subspaces: int, head_dim: int = 128, num_codewords: int = 256,
           page_size: int = 16) -> PQConfig:
    return PQConfig(head_dim, num_subspaces, num_codewords, page_size)
