"""NVFP4 FC2 oracle (CPU, plain C behind ctypes).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library (``diffusion_transformer_mlp_gb300``) never imports it and
shares no code, header, table or constant generator with it.

What it computes follows "FC2 NVFP4 Scheduling Results" (Canonical Operation)
and "GB10 component-2 nsys summary" (nvfp4, native_pack_validation,
other_boundaries); each C function cites its passage in ``nvfp4_oracle.c``.

Pinned on the CPU by tests/test_oracle_pins.py.  The byte conventions no
page prints are pinned on the GPU against readers outside this repository
(tests/test_gpu_pins.py): the nibble order by the tensor core's own reading
of the oracle's QDATA, the tiled scale layout by cuBLASLt's block-scaled
NVFP4 matmul on the oracle's bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_nvfp4.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ENONFINITE = 0, 1, 4


class ScaleRec(ctypes.Structure):
    _fields_ = [("global_scale", ctypes.c_float), ("amax_bits", ctypes.c_uint32),
                ("status", ctypes.c_uint32), ("pad", ctypes.c_uint32)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            i64 = ctypes.c_int64
            f64p = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_bf16_to_f32.restype = ctypes.c_float
            L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_f32_to_bf16.restype = ctypes.c_uint16
            L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            L.oracle_e2m1_value.restype = ctypes.c_double
            L.oracle_e2m1_value.argtypes = [ctypes.c_int]
            L.oracle_e2m1_encode.restype = ctypes.c_int
            L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_e4m3_value.argtypes = [ctypes.c_int]
            L.oracle_e4m3_encode.restype = ctypes.c_int
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_silu_bf16.restype = ctypes.c_uint16
            L.oracle_silu_bf16.argtypes = [ctypes.c_uint16]
            L.oracle_silu_table.restype = ctypes.c_int
            L.oracle_silu_table.argtypes = [u16p]
            L.oracle_swiglu_bf16.restype = ctypes.c_uint16
            L.oracle_swiglu_bf16.argtypes = [ctypes.c_uint16, ctypes.c_uint16, u16p]
            L.oracle_swiglu_rows.restype = ctypes.c_int
            L.oracle_swiglu_rows.argtypes = [u16p, i64, i64, i64, u16p]
            L.oracle_padded_rows.restype = i64
            L.oracle_padded_rows.argtypes = [i64]
            L.oracle_scale_cols_padded.restype = i64
            L.oracle_scale_cols_padded.argtypes = [i64]
            L.oracle_scale_offset.restype = i64
            L.oracle_scale_offset.argtypes = [i64, i64, i64]
            L.oracle_quantize.restype = ctypes.c_int
            L.oracle_quantize.argtypes = [u16p, i64, i64, i64, ctypes.c_int, u8p, u8p,
                                          ctypes.POINTER(ScaleRec)]
            L.oracle_dequantize_rows.restype = None
            L.oracle_dequantize_rows.argtypes = [u8p, u8p, ctypes.c_float, i64, i64p, i64, f64p]
            L.oracle_gemm_rows.restype = ctypes.c_int
            L.oracle_gemm_rows.argtypes = [u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float,
                                           i64, i64, i64p, i64, f64p]
            L.oracle_epilogue_bf16.restype = None
            L.oracle_epilogue_bf16.argtypes = [f64p, i64, ctypes.c_float, u16p]
            _lib = L
    return _lib


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(t))


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# ---- scalar codecs ---------------------------------------------------------

def e2m1_value(code: int) -> float:
    return float(lib().oracle_e2m1_value(int(code)))


def e2m1_encode(q: float) -> int:
    return int(lib().oracle_e2m1_encode(float(np.float32(q))))


def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_value(int(code)))


def e4m3_encode(r: float) -> int:
    return int(lib().oracle_e4m3_encode(float(np.float32(r))))


def f32_to_bf16(f: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(np.float32(f))))


def silu_table() -> tuple[np.ndarray, int]:
    """(65536 BF16 bit patterns of correctly rounded silu, unresolved ties)."""
    out = np.zeros(65536, dtype=np.uint16)
    unresolved = lib().oracle_silu_table(_p(out, ctypes.c_uint16))
    return out, int(unresolved)


def swiglu_bf16(g: int, u: int) -> int:
    return int(lib().oracle_swiglu_bf16(g, u, None))


def swiglu_rows(x: np.ndarray, cols: int) -> np.ndarray:
    """SwiGLU of a gate|up BF16 matrix (uint16 bits [rows, ld >= 2 cols]):
    h [rows, cols] as BF16 bits, the tensor the activation producer
    quantises."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows, ld = x.shape
    h = np.empty((rows, cols), dtype=np.uint16)
    st = lib().oracle_swiglu_rows(_p(x, ctypes.c_uint16), rows, cols, ld, _p(h, ctypes.c_uint16))
    if st != OK:
        raise ValueError(f"oracle_swiglu_rows rejected its arguments (status {st})")
    return h


# ---- sizes and layout ------------------------------------------------------

def padded_rows(rows: int) -> int:
    return int(lib().oracle_padded_rows(rows))


def scale_cols_padded(cols: int) -> int:
    return int(lib().oracle_scale_cols_padded(cols))


def scale_offset(r: int, c: int, cols: int) -> int:
    return int(lib().oracle_scale_offset(r, c, cols))


def qdata_bytes(rows: int, cols: int) -> int:
    return padded_rows(rows) * cols // 2


def scale_bytes(rows: int, cols: int) -> int:
    return padded_rows(rows) * scale_cols_padded(cols)


# ---- tensors ---------------------------------------------------------------

def quantize(x: np.ndarray, cols: int, swiglu: bool):
    """Two-pass NVFP4 quantisation of a BF16 tensor given as uint16 bits.

    x: [rows, ld] uint16; with swiglu the first 2*cols columns are gate|up.
    Returns (qdata uint8 [padded_rows, cols/2], scales uint8 [scale_bytes],
    rec dict).
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rows, ld = x.shape
    q = np.empty((padded_rows(rows), cols // 2), dtype=np.uint8)
    s = np.empty(scale_bytes(rows, cols), dtype=np.uint8)
    rec = ScaleRec()
    st = lib().oracle_quantize(_p(x, ctypes.c_uint16), rows, cols, ld, 1 if swiglu else 0,
                               _p(q, ctypes.c_uint8), _p(s, ctypes.c_uint8), ctypes.byref(rec))
    if st != OK:
        raise ValueError(f"oracle_quantize rejected its arguments (status {st})")
    return q, s, {"global_scale": np.float32(rec.global_scale), "amax_bits": int(rec.amax_bits),
                  "status": int(rec.status)}


def dequantize_rows(qdata: np.ndarray, scales: np.ndarray, global_scale: float, cols: int,
                    rows: np.ndarray) -> np.ndarray:
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, cols), dtype=np.float64)
    qdata = np.ascontiguousarray(qdata, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    lib().oracle_dequantize_rows(_p(qdata, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                                 float(global_scale), cols, _p(rows, ctypes.c_int64), rows.size,
                                 _p(out, ctypes.c_double))
    return out


def gemm_rows(a_q, a_s, ga, w_q, w_s, gw, n: int, k: int, rows: np.ndarray) -> np.ndarray:
    """Unrounded FP64 reference out[i, :] for activation rows ``rows``."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, n), dtype=np.float64)
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (a_q, a_s, w_q, w_s)]
    st = lib().oracle_gemm_rows(_p(arrs[0], ctypes.c_uint8), _p(arrs[1], ctypes.c_uint8), float(ga),
                                _p(arrs[2], ctypes.c_uint8), _p(arrs[3], ctypes.c_uint8), float(gw),
                                n, k, _p(rows, ctypes.c_int64), rows.size, _p(out, ctypes.c_double))
    if st != OK:
        raise ValueError(f"oracle_gemm_rows rejected its arguments (status {st})")
    return out


def epilogue_bf16(ref: np.ndarray, alpha: float) -> np.ndarray:
    """BF16 bits RNE(RN_f32(float32(ref) * alpha)): the GPU output for inputs
    whose FP32 accumulation is exact (every partial sum a binary32 value)."""
    ref = np.ascontiguousarray(ref, dtype=np.float64)
    out = np.empty(ref.shape, dtype=np.uint16)
    lib().oracle_epilogue_bf16(_p(ref, ctypes.c_double), ref.size, float(np.float32(alpha)), _p(out, ctypes.c_uint16))
    return out


def check_gemm_tolerance(gpu: np.ndarray, ref: np.ndarray) -> tuple[bool, float]:
    """|gpu - ref| <= 1e-2*|ref| + 1e-3*rms(ref), elementwise; returns
    (ok, worst ratio of |gpu-ref| to the bound)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = 1e-2 * np.abs(ref) + 1e-3 * rms
    err = np.abs(gpu - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    worst = float(ratio.max()) if ratio.size else 0.0
    return bool(np.all(err <= bound)), worst
