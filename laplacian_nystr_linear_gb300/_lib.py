"""ctypes binding of liblapnys.so (argument marshalling only).

The names and argument orders mirror include/lapnys.h one to one.  The library
is loaded from this package directory; if it is missing, every call raises:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblapnys.so")

(LAPNYS_OK, LAPNYS_EINVAL, LAPNYS_ECUDA, LAPNYS_ETIMEOUT, LAPNYS_ENOSPC, LAPNYS_ENOTSUP,
 LAPNYS_ESCRATCH) = range(7)
LAPNYS_F32, LAPNYS_BF16 = 0, 1
LAPNYS_NORM, LAPNYS_GAUSS, LAPNYS_NORM_BATCH = 1, 2, 4

# every symbol include/lapnys.h declares
EXPORTS = (
    "lapnys_ctx_bytes", "lapnys_workspace_bytes", "lapnys_fwd", "lapnys_bwd",
    "lapnys_ctx_offsets", "lapnys_pool", "lapnys_strerror", "lapnys_launch_count",
    "lapnys_profile_enable", "lapnys_profile_read", "lapnys_fwd_static", "lapnys_matmul",
    "lapnys_device_status", "lapnys_block_ctx_bytes", "lapnys_block_workspace_bytes",
    "lapnys_block_fwd", "lapnys_block_bwd", "lapnys_wait_selftest",
    "lapnys_fma_probe",
)


class CtxLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("L", "Llo", "A", "alpha", "X", "Y", "W", "What", "stats", "idx", "P", "C",
                 "total")]


_lib = None

P, I, F, U, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint, ctypes.c_size_t


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
            " (nvcc, sm_103a); there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    lib.lapnys_ctx_bytes.argtypes = [I, I, I, I, I, I, U]
    lib.lapnys_ctx_bytes.restype = S
    lib.lapnys_workspace_bytes.argtypes = [I, I, I, I, I, I, U]
    lib.lapnys_workspace_bytes.restype = S
    lib.lapnys_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, F, I, I, P, I, U, P, S, P, S]
    lib.lapnys_fwd.restype = I
    lib.lapnys_fwd_static.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, F, I, I, P, I, U]
    lib.lapnys_fwd_static.restype = I
    LL = ctypes.c_longlong
    lib.lapnys_matmul.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, I, I, LL, LL, LL, LL, F, F,
                                  I, P]
    lib.lapnys_matmul.restype = I
    lib.lapnys_block_ctx_bytes.argtypes = [I, I, I, I, I, I, I, I, I, U]
    lib.lapnys_block_ctx_bytes.restype = S
    lib.lapnys_block_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I, U]
    lib.lapnys_block_workspace_bytes.restype = S
    lib.lapnys_block_fwd.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, F, I, I, P, I, U,
                                     P, S, P, S]
    lib.lapnys_block_fwd.restype = I
    lib.lapnys_block_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, F, I,
                                     I, P, I, U, P, S]
    lib.lapnys_block_bwd.restype = I
    lib.lapnys_fma_probe.argtypes = [I, I, P, ctypes.POINTER(ctypes.c_ulonglong), P]
    lib.lapnys_fma_probe.restype = I
    lib.lapnys_wait_selftest.argtypes = [I, P]
    lib.lapnys_wait_selftest.restype = I
    lib.lapnys_device_status.argtypes = [I]
    lib.lapnys_device_status.restype = I
    lib.lapnys_bwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, F, I, I, P, I, U, P, S]
    lib.lapnys_bwd.restype = I
    lib.lapnys_ctx_offsets.argtypes = [I, I, I, I, I, I, U, ctypes.POINTER(CtxLayout)]
    lib.lapnys_ctx_offsets.restype = I
    lib.lapnys_pool.argtypes = [P, P, P, I, I, I, I, I, I, I, I, P]
    lib.lapnys_pool.restype = I
    lib.lapnys_strerror.argtypes = [I]
    lib.lapnys_strerror.restype = ctypes.c_char_p
    lib.lapnys_launch_count.argtypes = []
    lib.lapnys_launch_count.restype = ctypes.c_uint64
    lib.lapnys_profile_enable.argtypes = [I]
    lib.lapnys_profile_enable.restype = I
    lib.lapnys_profile_read.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(I),
                                        ctypes.POINTER(ctypes.c_double), I]
    lib.lapnys_profile_read.restype = I
    _lib = lib
    return lib


class LapnysError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = load().lapnys_strerror(code).decode()
        super().__init__(f"{where}: lapnys status {code} ({msg})")
        self.code = code


def check(code: int, where: str) -> None:
    if code != LAPNYS_OK:
        raise LapnysError(code, where)
