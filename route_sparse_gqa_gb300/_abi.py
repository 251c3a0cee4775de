"""ctypes view of libqsa's C ABI (include/qsa.h, include/qsa_route.h).  Marshalling only: every step
of the attention runs in the library's CUDA kernels; nothing here computes."""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libqsa.so")

QSA_OK = 0
STATUS_NAMES = {
    0: "QSA_OK",
    1: "QSA_ERR_INVALID_ARGUMENT",
    2: "QSA_ERR_UNSUPPORTED",
    3: "QSA_ERR_WORKSPACE_TOO_SMALL",
    4: "QSA_ERR_CUDA",
    5: "QSA_ERR_TIMEOUT",
    6: "QSA_ERR_DEVICE_CHECK",
}

# Every symbol include/qsa.h and include/qsa_route.h declare (checked by the tests
# against the built library).
EXPORTS = (
    "qsa_check_problem",
    "qsa_workspace_bytes",
    "qsa_preprocess",
    "qsa_forward",
    "qsa_backward",
    "qsa_backward_deterministic",
    "qsa_copy_route_sets",
    "qsa_forward_no_alloc",
    "qsa_read_no_alloc_status",
    "qsa_read_device_status",
    "qsa_status_string",
    "qsa_last_error",
    "qsa_route_check_problem",
    "qsa_route_width",
    "qsa_route_workspace_bytes",
    "qsa_index_scores",
    "qsa_select_from_scores",
    "qsa_select_token_ids",
)


class QSAError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{self.status_name}: {message}")


class Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("S_q", ctypes.c_int64), ("S_kv", ctypes.c_int64), ("Hq", ctypes.c_int64),
        ("Hkv", ctypes.c_int64), ("D", ctypes.c_int64), ("K", ctypes.c_int64),
        ("route_bits", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
        ("q_stride", ctypes.c_int64 * 4), ("k_stride", ctypes.c_int64 * 4), ("v_stride", ctypes.c_int64 * 4),
        ("r_stride", ctypes.c_int64 * 3), ("flags", ctypes.c_uint32),
    ]


ROUTES_SORTED = 1  # Problem.flags: rows already sorted and unique, invalid slots last
DETERMINISTIC_FORWARD = 2  # Problem.flags: bitwise reproducible forward (the tile kernels)


class RouteProblem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("S_q", ctypes.c_int64), ("H_index", ctypes.c_int64), ("D_index", ctypes.c_int64),
        ("n_blocks", ctypes.c_int64), ("token_budget", ctypes.c_int64), ("compress_ratio", ctypes.c_int64),
        ("query_position_offset", ctypes.c_int64),
        ("q_stride", ctypes.c_int64 * 4), ("k_stride", ctypes.c_int64 * 3),
    ]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Loads the in-tree libqsa.so.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libqsa.so is not built ({LIB_PATH}); run route_sparse_gqa_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(Problem)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        lib.qsa_check_problem.argtypes = [P]
        lib.qsa_workspace_bytes.argtypes = [P]
        lib.qsa_workspace_bytes.restype = sz
        lib.qsa_preprocess.argtypes = [P, vp, vp, sz, vp]
        lib.qsa_forward.argtypes = [P, vp, sz, vp, vp, vp, vp, vp, vp]
        lib.qsa_backward.argtypes = [P, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.qsa_backward_deterministic.argtypes = [P, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.qsa_copy_route_sets.argtypes = [P, vp, sz, vp, vp, vp]
        lib.qsa_forward_no_alloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp]
        lib.qsa_read_device_status.argtypes = [vp, vp]
        lib.qsa_read_no_alloc_status.argtypes = [vp]
        lib.qsa_status_string.argtypes = [ctypes.c_int]
        lib.qsa_status_string.restype = ctypes.c_char_p
        lib.qsa_last_error.argtypes = []
        lib.qsa_last_error.restype = ctypes.c_char_p
        R = ctypes.POINTER(RouteProblem)
        lib.qsa_route_check_problem.argtypes = [R]
        lib.qsa_route_width.argtypes = [R]
        lib.qsa_route_width.restype = ctypes.c_int64
        lib.qsa_route_workspace_bytes.argtypes = [R]
        lib.qsa_route_workspace_bytes.restype = sz
        lib.qsa_index_scores.argtypes = [R, vp, vp, vp, vp, sz, vp, vp]
        lib.qsa_select_from_scores.argtypes = [R, vp, vp, vp, sz, vp, vp]
        lib.qsa_select_token_ids.argtypes = [R, vp, vp, vp, vp, sz, vp, vp]
        for name in ("qsa_check_problem", "qsa_preprocess", "qsa_forward", "qsa_backward",
                     "qsa_backward_deterministic", "qsa_copy_route_sets",
                     "qsa_forward_no_alloc", "qsa_read_no_alloc_status", "qsa_read_device_status",
                     "qsa_route_check_problem",
                     "qsa_index_scores", "qsa_select_from_scores", "qsa_select_token_ids"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != QSA_OK:
        msg = load().qsa_last_error().decode(errors="replace")
        raise QSAError(status, msg)
