"""ctypes binding of libmuonbank.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module only turns
torch tensors into device pointers and shapes, passes the current CUDA
stream, and raises on a non-zero status.  There is no fallback: if the
library is missing the call fails.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmuonbank.so")

c_int, c_float, c_void_p, c_size_t, c_uint = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint

MB_OK = 0
MB_ERR_NULL = -1
MB_ERR_SHAPE = -2
MB_ERR_ALIGN = -3
MB_ERR_NS_STEPS = -4
MB_ERR_WORKSPACE = -5
MB_ERR_CUDA = -6
MB_ERR_TIMEOUT = -7
MB_ERR_ARG = -8
MB_ERR_UNSUPPORTED = -9
MB_ERR_TOO_MANY = -10
MB_ERR_SCRATCH_LIMIT = -11
MB_ERR_DEVICE = -12
MB_NOALLOC_SCRATCH_BYTES = 32 << 20
MB_MAX_BANKS = 8
MB_STEP_FUSE_UPDATE = 1
MB_STEP_FUSE_ROWSTATS = 2


class MbShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("rows", ctypes.c_int32), ("cols", ctypes.c_int32)]


class MbBankDesc(ctypes.Structure):
    _fields_ = [("bank", c_void_p), ("grad", c_void_p), ("momentum", c_void_p), ("mantissa", c_void_p),
                ("row_state", c_void_p), ("shape", MbShape), ("bank_copy", c_void_p)]


_P = c_void_p
_SIGNATURES = {
    "mb_workspace_bytes": (c_int, [MbShape, c_int, ctypes.POINTER(c_size_t)]),
    "muon_bank_step": (c_int, [_P, _P, _P, _P, MbShape, c_float, c_float, c_float, c_int, _P, c_size_t, _P]),
    "normuon_bank_step": (c_int, [_P, _P, _P, _P, _P, MbShape, c_float, c_float, c_float, c_float, c_int, _P,
                                  c_size_t, _P]),
    "mb_multi_workspace_bytes": (c_int, [ctypes.POINTER(MbBankDesc), c_int, c_int, ctypes.POINTER(c_size_t)]),
    "muon_multi_step": (c_int, [ctypes.POINTER(MbBankDesc), c_int, c_float, c_float, c_float, c_int, c_float,
                                c_int, _P, c_size_t, _P]),
    "muon_multi_step_ex": (c_int, [ctypes.POINTER(MbBankDesc), c_int, c_float, c_float, c_float, c_int, c_float,
                                   c_int, c_uint, _P, c_size_t, _P]),
    "muon_multi_step_dev": (c_int, [ctypes.POINTER(MbBankDesc), c_int, _P, c_int, c_int, _P, c_size_t, _P]),
    "mb_momentum": (c_int, [_P, _P, _P, MbShape, c_float, _P]),
    "mb_newton_schulz": (c_int, [_P, _P, MbShape, c_int, _P, c_size_t, _P]),
    "mb_newton_schulz_coeffs": (c_int, [_P, _P, MbShape, c_int, ctypes.POINTER(c_float), _P, c_size_t, _P]),
    "mb_newton_schulz_noalloc": (c_int, [_P, _P, MbShape, c_int, _P]),
    "mb_update": (c_int, [_P, _P, _P, MbShape, c_float, c_float, _P]),
    "mb_normuon_update": (c_int, [_P, _P, _P, _P, MbShape, c_float, c_float, c_float, _P, c_size_t, _P]),
    "mb_workspace_views": (c_int, [MbShape, c_int, c_int, ctypes.POINTER(c_size_t), ctypes.POINTER(c_size_t),
                                   ctypes.POINTER(c_size_t)]),
    "mb_sync_status": (c_int, [_P]),
    "mb_selftest_timeout": (c_int, [c_uint, _P]),
    "mb_status_string": (ctypes.c_char_p, [c_int]),
    "mb_last_cuda_error": (ctypes.c_char_p, []),
    "mb_version": (c_int, []),
    "mb_launch_count": (ctypes.c_uint64, []),
    "mb_timing_begin": (c_int, [c_int]),
    "mb_timing_end": (c_int, [c_int, ctypes.POINTER(c_int), ctypes.POINTER(c_float), ctypes.POINTER(c_int)]),
}

MARK_NAMES = {0: "begin", 1: "momentum", 2: "scale", 3: "small_ns", 4: "ns_gemm", 5: "ns0", 6: "rowstats",
              7: "update"}

_lib = None


def load():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() or "
                               "python -m newton_schulz_stacked_gb300.build")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class MuonBankError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = load()
        msg = lib.mb_status_string(status).decode()
        if status == MB_ERR_CUDA:
            msg += ": " + lib.mb_last_cuda_error().decode()
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != MB_OK:
        raise MuonBankError(fn, status)


def shape_of(batch: int, rows: int, cols: int) -> MbShape:
    return MbShape(batch, rows, cols)
