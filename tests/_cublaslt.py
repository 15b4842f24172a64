"""Block-scaled NVFP4 matmul through cuBLASLt (ctypes).

An NVFP4 consumer written by someone else: the GPU tests hand it the
oracle's QDATA and tiled scale bytes to check that those bytes mean what a
library reading NVFP4 takes them to mean.  cuBLASLt's vector-16 UE4M3 mode
reads the block scales in its own documented 128-row by 4-column tiled
layout, so a wrong scale offset in the oracle gives a wrong product here.

out[i, j] = sum_k A[i, k] W[j, k] (FP32), A = E2M1(a_q) * UE4M3(a_s) and
W likewise; no global scales (alpha = 1).  In cuBLASLt's column-major terms
this is D[N, M] = op(W)^T op(A) with TRANSA = T and TRANSB = N (the "TN"
form block-scaled FP4 requires); the row-major [M, N] result is D.
"""
from __future__ import annotations

import ctypes

import torch

CUBLAS_COMPUTE_32F = 68
CUDA_R_32F = 0
CUDA_R_4F_E2M1 = 33
CUBLAS_OP_N, CUBLAS_OP_T = 0, 1
DESC_TRANSA, DESC_TRANSB = 3, 4
DESC_A_SCALE_POINTER, DESC_B_SCALE_POINTER = 17, 18
DESC_A_SCALE_MODE, DESC_B_SCALE_MODE = 31, 32
SCALE_VEC16_UE4M3 = 1
PREF_MAX_WORKSPACE_BYTES = 1
WORKSPACE = 64 << 20


class _Heuristic(ctypes.Structure):
    _fields_ = [("algo", ctypes.c_uint64 * 8), ("workspace_size", ctypes.c_size_t), ("state", ctypes.c_int),
                ("waves", ctypes.c_float), ("reserved", ctypes.c_int * 4)]


_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        err = None
        for name in ("libcublasLt.so.13", "/usr/local/cuda/lib64/libcublasLt.so.13", "libcublasLt.so"):
            try:
                _lib = ctypes.CDLL(name)
                break
            except OSError as e:  # try the next location
                err = e
        if _lib is None:
            raise OSError(f"cuBLASLt not found: {err}")
    return _lib


def _ok(st: int, what: str) -> None:
    if st != 0:
        raise RuntimeError(f"cuBLASLt {what} returned status {st}")


def nvfp4_matmul(a_q: torch.Tensor, a_s: torch.Tensor, w_q: torch.Tensor, w_s: torch.Tensor,
                 m: int, n: int, k: int) -> torch.Tensor:
    """FP32 [m, n] = (A W^T) of device NVFP4 bytes: a_q [>= m, k/2] and w_q
    [n, k/2] uint8 row-major, a_s and w_s the tiled UE4M3 scales."""
    L = load()
    vp = ctypes.c_void_p
    handle, desc, pref = vp(), vp(), vp()
    lay_w, lay_a, lay_d = vp(), vp(), vp()
    _ok(L.cublasLtCreate(ctypes.byref(handle)), "create")
    try:
        _ok(L.cublasLtMatmulDescCreate(ctypes.byref(desc), CUBLAS_COMPUTE_32F, CUDA_R_32F), "desc")

        def set_i32(attr, v):
            x = ctypes.c_int32(v)
            _ok(L.cublasLtMatmulDescSetAttribute(desc, attr, ctypes.byref(x), ctypes.sizeof(x)), f"attr {attr}")

        def set_ptr(attr, t):
            x = ctypes.c_void_p(t.data_ptr())
            _ok(L.cublasLtMatmulDescSetAttribute(desc, attr, ctypes.byref(x), ctypes.sizeof(x)), f"attr {attr}")

        set_i32(DESC_TRANSA, CUBLAS_OP_T)
        set_i32(DESC_TRANSB, CUBLAS_OP_N)
        set_i32(DESC_A_SCALE_MODE, SCALE_VEC16_UE4M3)
        set_i32(DESC_B_SCALE_MODE, SCALE_VEC16_UE4M3)
        set_ptr(DESC_A_SCALE_POINTER, w_s)  # cuBLASLt's A is the weight
        set_ptr(DESC_B_SCALE_POINTER, a_s)
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        _ok(L.cublasLtMatrixLayoutCreate(ctypes.byref(lay_w), CUDA_R_4F_E2M1, u64(k), u64(n), i64(k)), "layout W")
        _ok(L.cublasLtMatrixLayoutCreate(ctypes.byref(lay_a), CUDA_R_4F_E2M1, u64(k), u64(m), i64(k)), "layout A")
        _ok(L.cublasLtMatrixLayoutCreate(ctypes.byref(lay_d), CUDA_R_32F, u64(n), u64(m), i64(n)), "layout D")
        _ok(L.cublasLtMatmulPreferenceCreate(ctypes.byref(pref)), "preference")
        ws = ctypes.c_uint64(WORKSPACE)
        _ok(L.cublasLtMatmulPreferenceSetAttribute(pref, PREF_MAX_WORKSPACE_BYTES, ctypes.byref(ws),
                                                     ctypes.sizeof(ws)), "workspace preference")
        heur = _Heuristic()
        found = ctypes.c_int(0)
        _ok(L.cublasLtMatmulAlgoGetHeuristic(handle, desc, lay_w, lay_a, lay_d, lay_d, pref, 1,
                                             ctypes.byref(heur), ctypes.byref(found)), "heuristic")
        if found.value < 1:
            raise RuntimeError("cuBLASLt found no algorithm for the block-scaled NVFP4 matmul")
        out = torch.zeros(m, n, dtype=torch.float32, device=a_q.device)
        work = torch.empty(WORKSPACE, dtype=torch.uint8, device=a_q.device)
        alpha, beta = ctypes.c_float(1.0), ctypes.c_float(0.0)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        _ok(L.cublasLtMatmul(handle, desc, ctypes.byref(alpha), vp(w_q.data_ptr()), lay_w, vp(a_q.data_ptr()),
                             lay_a, ctypes.byref(beta), vp(out.data_ptr()), lay_d, vp(out.data_ptr()), lay_d,
                             ctypes.byref(heur.algo), vp(work.data_ptr()), ctypes.c_size_t(WORKSPACE), stream),
            "matmul")
        torch.cuda.synchronize()
        return out
    finally:
        for h, fn in ((pref, "cublasLtMatmulPreferenceDestroy"), (lay_d, "cublasLtMatrixLayoutDestroy"),
                      (lay_a, "cublasLtMatrixLayoutDestroy"), (lay_w, "cublasLtMatrixLayoutDestroy"),
                      (desc, "cublasLtMatmulDescDestroy")):
            if h.value:
                getattr(L, fn)(h)
        if handle.value:
            L.cublasLtDestroy(handle)
