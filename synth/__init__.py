"""Seeded synthetic FC2 inputs (BF16 bit patterns as numpy uint16).

Shared by the tests, the benchmark and the oracle checks; it holds none of
the NVFP4 method's arithmetic.  The recipe (splitmix64 counter stream,
Box-Muller, 0.1% x20 outliers, RNE to BF16) is documented in synth.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_ACTIVATION = 0
STREAM_WEIGHT = 1


def build(force: bool = False) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.synth_normal_bf16.restype = None
            L.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                            ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                            ctypes.c_double, ctypes.POINTER(ctypes.c_uint16)]
            _lib = L
    return _lib


def normal_bf16(shape, seed: int, stream: int, sigma: float = 1.0, outlier_p: float = 0.0,
                outlier_scale: float = 20.0, first: int = 0, out: np.ndarray | None = None):
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"] and out.size == n
    _get().synth_normal_bf16(seed, stream, first, n, float(sigma), float(outlier_p),
                             float(outlier_scale), out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))
    return out


def activation(m: int, k: int, seed: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """gate|up BF16 [m, 2k]: N(0,1) with 0.1% of entries x20."""
    return normal_bf16((m, 2 * k), seed, STREAM_ACTIVATION, 1.0, 1e-3, 20.0, out=out)


def quant_input(m: int, f: int, seed: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """BF16 [m, f] activations for the quantise-only workload (same law)."""
    return normal_bf16((m, f), seed, STREAM_ACTIVATION, 1.0, 1e-3, 20.0, out=out)


def weight(n: int, k: int, seed: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """BF16 [n, k]: N(0, sigma = k^-1/2), no outliers."""
    return normal_bf16((n, k), seed, STREAM_WEIGHT, float(k) ** -0.5, 0.0, 1.0, out=out)


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.uint32) << 16).view(np.float32)
