"""ctypes binding of libnvfp4fc2.so (argument marshalling only).

Every function here has the name of the C entry point it calls; PyTorch only
supplies device memory and the current CUDA stream.  There is no fallback:
if the library cannot be loaded, or a call returns a non-zero status, a
RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libnvfp4fc2.so")

NVFP4_OK = 0
NVFP4_EINVAL = 1
NVFP4_EUNSUPPORTED = 2
NVFP4_EALIGN = 3
NVFP4_ENONFINITE = 4
NVFP4_ETIMEOUT = 5
NVFP4_ECUDA = 6
STATUS_NAMES = {0: "NVFP4_OK", 1: "NVFP4_EINVAL", 2: "NVFP4_EUNSUPPORTED", 3: "NVFP4_EALIGN",
                4: "NVFP4_ENONFINITE", 5: "NVFP4_ETIMEOUT", 6: "NVFP4_ECUDA"}

# every symbol the headers in include/ declare
EXPORTED = ["nvfp4_padded_rows", "nvfp4_qdata_bytes", "nvfp4_scale_bytes", "nvfp4_scale_offset",
            "nvfp4_quantize_weight", "swiglu_nvfp4_quantize", "nvfp4_fc2_gemm", "nvfp4_last_error",
            "nvfp4_version", "nvfp4_diag_silu_all", "nvfp4_diag_swiglu", "nvfp4_diag_code_transitions",
            "nvfp4_diag_wait_timeout", "nvfp4_diag_mma_peak", "nvfp4_diag_mma_peak_pairs",
            "nvfp4_diag_quotient_codes", "nvfp4_fc1_swiglu", "nvfp4_quantize_with_amax",
            "nvfp4_diag_silu_epilogue", "nvfp4_diag_block_scale_codes", "nvfp4_diag_tc_e2m1_read", "nvfp4_fc2_host",
            "nvfp4_fc2_host_noalloc", "nvfp4_diag_fc2_gemm_clock"]

_lock = threading.Lock()
_lib = None


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (building it in-tree first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            from . import build as _build
            p = _build.build()
        L = ctypes.CDLL(p)
        i64, u32, vp = ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p
        st = ctypes.c_int
        L.nvfp4_padded_rows.restype = i64
        L.nvfp4_padded_rows.argtypes = [i64]
        L.nvfp4_qdata_bytes.restype = i64
        L.nvfp4_qdata_bytes.argtypes = [i64, i64]
        L.nvfp4_scale_bytes.restype = i64
        L.nvfp4_scale_bytes.argtypes = [i64, i64]
        L.nvfp4_scale_offset.restype = i64
        L.nvfp4_scale_offset.argtypes = [i64, i64, i64]
        L.nvfp4_quantize_weight.restype = st
        L.nvfp4_quantize_weight.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        L.swiglu_nvfp4_quantize.restype = st
        L.swiglu_nvfp4_quantize.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        L.nvfp4_fc2_gemm.restype = st
        L.nvfp4_fc2_gemm.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, vp]
        L.nvfp4_last_error.restype = ctypes.c_char_p
        L.nvfp4_last_error.argtypes = []
        L.nvfp4_version.restype = u32
        L.nvfp4_version.argtypes = []
        L.nvfp4_diag_silu_all.restype = st
        L.nvfp4_diag_silu_all.argtypes = [vp, vp]
        L.nvfp4_diag_swiglu.restype = st
        L.nvfp4_diag_swiglu.argtypes = [vp, vp, vp, i64, vp]
        L.nvfp4_diag_code_transitions.restype = st
        L.nvfp4_diag_code_transitions.argtypes = [ctypes.c_int, vp, u32, vp, vp, vp]
        L.nvfp4_diag_wait_timeout.restype = st
        L.nvfp4_diag_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp]
        L.nvfp4_diag_mma_peak.restype = st
        L.nvfp4_diag_mma_peak.argtypes = [i64, vp, vp, vp]
        L.nvfp4_diag_fc2_gemm_clock.restype = st
        L.nvfp4_diag_fc2_gemm_clock.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, vp, vp]
        L.nvfp4_diag_mma_peak_pairs.restype = i64
        L.nvfp4_diag_mma_peak_pairs.argtypes = []
        L.nvfp4_diag_quotient_codes.restype = st
        L.nvfp4_diag_quotient_codes.argtypes = [u32, u32, vp, vp]
        L.nvfp4_fc1_swiglu.restype = st
        L.nvfp4_fc1_swiglu.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, vp, vp]
        L.nvfp4_quantize_with_amax.restype = st
        L.nvfp4_quantize_with_amax.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        L.nvfp4_diag_silu_epilogue.restype = st
        L.nvfp4_diag_silu_epilogue.argtypes = [vp, vp]
        L.nvfp4_diag_block_scale_codes.restype = st
        L.nvfp4_diag_block_scale_codes.argtypes = [u32, u32, vp, vp]
        L.nvfp4_diag_tc_e2m1_read.restype = st
        L.nvfp4_fc2_host.restype = st
        L.nvfp4_fc2_host.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp]
        L.nvfp4_fc2_host_noalloc.restype = st
        L.nvfp4_fc2_host_noalloc.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64, vp, vp, vp]
        L.nvfp4_diag_tc_e2m1_read.argtypes = [vp, vp, vp, vp]
        _lib = L
        return _lib


def check(status: int, where: str) -> None:
    if status != NVFP4_OK:
        msg = load().nvfp4_last_error().decode(errors="replace")
        raise NVFP4Error(status, where, msg)


def last_error() -> str:
    return load().nvfp4_last_error().decode(errors="replace")
