"""ctypes binding of libkda.so (argument marshalling only).

Every function here forwards to the C entry point of the same name declared
in include/kda.h. Nothing is computed in Python. If the shared library is
missing the import fails loudly: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK = 0
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED",
                3: "KDA_ERR_WORKSPACE", 4: "KDA_ERR_CUDA", 5: "KDA_ERR_DEVICE_TIMEOUT"}
DTYPES = {"bf16": 0, "fp32": 1}
GATES = {"none": 0, "scalar": 1, "channel": 2}


class KdaProblem(ctypes.Structure):
    """Mirror of ``kda_problem`` in include/kda.h."""

    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("K", ctypes.c_int), ("V", ctypes.c_int),
        ("N", ctypes.c_int),
        ("cu_seqlens", ctypes.c_void_p),
        ("io", ctypes.c_int),
        ("gate", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("g", ctypes.c_void_p),
        ("h0", ctypes.c_void_p),
        ("save_policy", ctypes.c_int),
        ("schedule", ctypes.c_int),
        ("A_log", ctypes.c_void_p),
        ("dt_bias", ctypes.c_void_p),
        ("lower_bound", ctypes.c_float),
        ("qk_l2norm", ctypes.c_int),
        ("l2norm_eps", ctypes.c_float),
        ("erase", ctypes.c_void_p),
        ("write", ctypes.c_void_p),
        ("HV", ctypes.c_int),
    ]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libkda.so is not built (run `python -m chunkwise_delta_rule_gb300.build`); "
            "this package has no non-CUDA implementation")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(KdaProblem)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.kda_workspace_size.argtypes = [P, ctypes.c_int]
    lib.kda_workspace_size.restype = sz
    lib.kda_saved_size.argtypes = [P]
    lib.kda_saved_size.restype = sz
    lib.kda_chunk_fwd.argtypes = [P, vp, vp, vp, vp, sz, vp]
    lib.kda_chunk_fwd.restype = ctypes.c_int
    lib.kda_chunk_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.kda_chunk_bwd.restype = ctypes.c_int
    lib.kda_device_status.argtypes = [P, vp, sz, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.kda_device_status.restype = ctypes.c_int
    lib.kda_last_error.argtypes = []
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_recurrent_fwd.argtypes = [P, vp, vp, vp, vp]
    lib.kda_recurrent_fwd.restype = ctypes.c_int
    lib.kda_abi_version.argtypes = []
    lib.kda_abi_version.restype = ctypes.c_int
    _lib = lib
    return lib


def last_error() -> str:
    return load().kda_last_error().decode()


def check(status: int, where: str) -> None:
    if status != KDA_OK:
        raise KdaError(status, where, last_error())
