"""ctypes loader of the in-tree CUDA library ``libfkl.so`` (C ABI in include/fkl.h).

There is no fallback: if the library is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

LIB_PATH = Path(__file__).resolve().with_name("libfkl.so")

STATUS = {
    0: "FKL_OK",
    1: "FKL_ERR_INVALID_ARG",
    2: "FKL_ERR_ALIGNMENT",
    3: "FKL_ERR_UNSUPPORTED",
    4: "FKL_ERR_WORKSPACE",
    5: "FKL_ERR_CUDA",
    6: "FKL_ERR_BAD_TOPK_ID",
    7: "FKL_ERR_BAD_TOPK_ROW",
    8: "FKL_ERR_TIMEOUT",
    9: "FKL_ERR_BAD_SEQ_ID",
    10: "FKL_ERR_TOPK_OVERFLOW",
    11: "FKL_ERR_BAD_COUNT",
}
FKL_OK = 0

class FklOptions(ctypes.Structure):
    """fkl_options of include/fkl.h."""

    _fields_ = [("normalization", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("seq_ids", ctypes.c_void_p), ("accumulate", ctypes.c_int32), ("divergence", ctypes.c_int32),
                ("div_param", ctypes.c_float), ("reserved", ctypes.c_int32),
                ("student_topk_logits", ctypes.c_void_p), ("global_count", ctypes.c_void_p)]


FKL_NORM_TOKENS, FKL_NORM_SEQUENCES = 0, 1
FKL_ACCUMULATE_DH, FKL_ACCUMULATE_DW = 1, 2
# fkl_options.divergence, by the names the binding accepts
DIVERGENCES = {"kl": 0, "jsd": 1, "skew_kl": 2, "skew_rkl": 3, "tv": 4}

# Every symbol declared in include/*.h, with (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGNATURES = {
    "fkl_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, _I64, _I64]),
    "fkl_backward_slabs": (ctypes.c_int64, [_I64, _I64, _I64, _I64, _I64]),
    "fkl_forward": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float, _I64,
                                   _P, _P, _P, ctypes.c_size_t, _P]),
    "fkl_backward": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                    _I64, _P, _P, _P, ctypes.c_size_t, _P]),
    "fkl_forward_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                           _P, _P, _P]),
    "fkl_trace_start": (ctypes.c_int, [ctypes.c_int32]),
    "fkl_trace_stop": (ctypes.c_int, []),
    "fkl_trace_read": (ctypes.c_int32, [_P, _P, _P, ctypes.c_int32]),
    "fkl_forward_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float, _I64,
                                      ctypes.POINTER(FklOptions), _P, _P, _P, ctypes.c_size_t, _P]),
    "fkl_backward_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                       _I64, ctypes.POINTER(FklOptions), _P, _P, _P, ctypes.c_size_t, _P]),
    "fkl_backward_bf16": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_float,
                                       _I64, ctypes.POINTER(FklOptions), _P, _P, _P, ctypes.c_size_t, _P]),
    "fkl_backward_bf16_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, _I64, _I64]),
    "fkl_teacher_topk_workspace_size": (ctypes.c_size_t, [_I64, _I64, _I64, _I64]),
    "fkl_teacher_topk": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, ctypes.c_size_t, _P]),
    "fkl_test_backward_plan": (ctypes.c_int, [_I64, _I64, _I64, _I64, _I64, ctypes.c_int32, _P]),
    "fkl_teacher_topk_ex": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, ctypes.c_int32, _P, _P, _P,
                                           ctypes.c_size_t, _P]),
    "fkl_read_status": (ctypes.c_int, [_P, _P]),
    "fkl_local_count": (ctypes.c_int, [_P, _I64, ctypes.POINTER(FklOptions), _P, _P, ctypes.c_size_t, _P]),
    "fkl_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fkl_last_error": (ctypes.c_char_p, []),
    "fkl_test_gemm": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "fkl_test_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, _P, ctypes.c_size_t, _P]),
}

_lib = None
_lock = threading.Lock()


class FklError(RuntimeError):
    """A non-zero fkl_status from the library."""

    def __init__(self, status: int, where: str, message: str = ""):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        super().__init__(f"{where}: {name}" + (f" ({message})" if message else ""))


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not LIB_PATH.exists():
                    raise RuntimeError(
                        f"{LIB_PATH} is not built; run `python -m lm_head_top_tcgen05_gb300.build` "
                        "or __graft_entry__.build() first")
                L = ctypes.CDLL(str(LIB_PATH))
                for name, (res, args) in _SIGNATURES.items():
                    f = getattr(L, name)
                    f.restype = res
                    f.argtypes = args
                _lib = L
    return _lib


def check(status: int, where: str) -> None:
    if status != FKL_OK:
        msg = lib().fkl_last_error() or b""
        raise FklError(status, where, msg.decode(errors="replace"))
