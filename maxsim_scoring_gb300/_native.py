"""ctypes loader for libmaxsim.so (the C ABI in include/maxsim.h).

The library is built in-tree by ``maxsim_scoring_gb300.build``. There is no
fallback: if the shared library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmaxsim.so")

_lock = threading.Lock()
_lib = None

STATUS = {
    0: "MAXSIM_OK",
    1: "MAXSIM_ERR_INVALID_ARG",
    2: "MAXSIM_ERR_UNSUPPORTED",
    3: "MAXSIM_ERR_CUDA",
    4: "MAXSIM_ERR_TIMEOUT",
    5: "MAXSIM_ERR_WORKSPACE",
    6: "MAXSIM_ERR_DEVICE_INPUT",
}

OP_FWD, OP_FWD_VARLEN, OP_BWD, OP_FWD_INT8, OP_SCORE_PAIRS = 0, 1, 2, 3, 4
OP_CHAMFER_FWD, OP_CHAMFER_BWD, OP_TWO_STAGE, OP_FWD_STREAMED, OP_BWD_VARLEN = 5, 6, 7, 8, 9
OP_FWD_VARLEN_STREAMED = 10
F16, BF16 = 0, 1

# Every symbol the header declares, with its ctypes signature.
_I64, _VP, _SZ, _I = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
SIGNATURES = {
    "maxsim_fwd": (_I, [_VP, _VP, _I, _I64, _I64, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "maxsim_fwd_varlen": (_I, [_VP, _VP, _I64, _VP, _VP, _I64, _I, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _SZ,
                               _VP]),
    "maxsim_bwd": (_I, [_VP, _VP, _I, _I64, _I64, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                        _VP]),
    "maxsim_fwd_int8": (_I, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                             _VP]),
    "maxsim_fwd_varlen_noalloc": (_I, [_VP, _VP, _I64, _VP, _VP, _I64, _I, _I64, _I64, _I64, _VP, _VP, _VP, _VP,
                                       _VP]),
    "maxsim_score_pairs_packed": (_I, [_VP, _VP, _I64, _VP, _VP, _I64, _I, _I64, _I64, _I64, _VP, _VP, _VP, _I64,
                                       _VP, _VP, _VP, _SZ, _VP]),
    "maxsim_chamfer_fwd": (_I, [_VP, _VP, _I64, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "maxsim_chamfer_bwd": (_I, [_VP, _VP, _I64, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "maxsim_topk": (_I, [_VP, _I64, _I64, _I64, _VP, _VP, _VP]),
    "maxsim_bwd_varlen": (_I, [_VP, _VP, _I64, _VP, _VP, _I64, _I64, _I, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP,
                               _VP, _VP, _VP, _SZ, _VP]),
    "maxsim_fwd_streamed": (_I, [_VP, _VP, _I, _I64, _I64, _I64, _I64, _I64, _I64, _VP, _VP, _VP, _SZ, _VP]),
    "maxsim_fwd_varlen_streamed": (_I, [_VP, _VP, _I64, _VP, _VP, _I64, _I, _I64, _I64, _I64, _VP, _I64, _I64, _VP,
                                        _VP, _SZ, _VP]),
    "maxsim_two_stage_topk": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _VP,
                                   _VP, _VP, _VP, _VP, _SZ, _VP]),
    "maxsim_workspace_size": (_SZ, [_I, _I64, _I64, _I64, _I64, _I64]),
    "maxsim_status_string": (ctypes.c_char_p, [_I]),
    "maxsim_device_status": (_I, [_VP]),
    "maxsim_last_device_status": (_I, [_VP]),
    "maxsim_debug_inject_wait_timeout": (_I, [ctypes.c_uint64]),
    "maxsim_version": (_I, []),
}


class MaxSimError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code)})")


def lib():
    """The loaded library; raises if it was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with maxsim_scoring_gb300.build.build()")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def status_string(code: int) -> str:
    s = lib().maxsim_status_string(code)
    return s.decode() if s else "?"


def check(code: int, where: str) -> None:
    if code != 0:
        raise MaxSimError(code, where)
