"""NVFP4 FC2 step of a video diffusion transformer MLP on GB300 (sm_103a).

Python face of libnvfp4fc2.so.  Each function forwards to the C entry point
of the same name; PyTorch provides device memory and the current stream.

    w_q  = nvfp4_quantize_weight(w_bf16)                 # once per weight
    a_q  = swiglu_nvfp4_quantize(gate_up_bf16)           # per step
    out  = nvfp4_fc2_gemm(a_q, w_q)                      # per step
    out  = fc2(gate_up_bf16, w_q)                        # both per-step calls
    out  = fc2_host(gate_up_host, w_q)                   # host in, host out

Sources: "FC2 NVFP4 Scheduling Results" (Canonical Operation; Production
Integration: forward_swiglu = accepted producer, then the FC2 GEMM) and
"GB10 component-2 nsys summary" (nvfp4; native_pack_validation).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import NVFP4Error, load  # noqa: F401

__all__ = ["NVFP4Tensor", "NVFP4Error", "load", "padded_rows", "qdata_bytes", "scale_bytes", "scale_offset",
           "nvfp4_quantize_weight", "swiglu_nvfp4_quantize", "nvfp4_fc2_gemm", "nvfp4_fc1_swiglu", "fc2", "fc2_host",
           "empty_nvfp4", "read_rec"]


def padded_rows(rows: int) -> int:
    return int(load().nvfp4_padded_rows(rows))


def qdata_bytes(rows: int, cols: int) -> int:
    return int(load().nvfp4_qdata_bytes(rows, cols))


def scale_bytes(rows: int, cols: int) -> int:
    return int(load().nvfp4_scale_bytes(rows, cols))


def scale_offset(r: int, c: int, cols: int) -> int:
    return int(load().nvfp4_scale_offset(r, c, cols))


@dataclass
class NVFP4Tensor:
    """Device NVFP4 tensor: QDATA [padded_rows, cols/2] uint8, tiled scales,
    and the 16-byte global-scale record (float32 g, u32 amax bits, u32
    status, reserved), all on one CUDA device."""
    qdata: torch.Tensor
    scales: torch.Tensor
    rec: torch.Tensor
    rows: int
    cols: int

    @property
    def device(self) -> torch.device:
        return self.qdata.device


def empty_nvfp4(rows: int, cols: int, device="cuda") -> NVFP4Tensor:
    q = torch.empty(qdata_bytes(rows, cols), dtype=torch.uint8, device=device).view(padded_rows(rows), cols // 2)
    s = torch.empty(scale_bytes(rows, cols), dtype=torch.uint8, device=device)
    rec = torch.empty(16, dtype=torch.uint8, device=device)
    return NVFP4Tensor(q, s, rec, rows, cols)


def read_rec(t: NVFP4Tensor) -> dict:
    """Copy the record to the host (synchronises)."""
    r = t.rec.cpu()
    return {"global_scale": float(r[0:4].view(torch.float32)[0]),
            "amax_bits": int(r[4:8].view(torch.int32)[0]) & 0xFFFFFFFF,
            "status": int(r[8:12].view(torch.int32)[0])}


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _check_dev(*ts: torch.Tensor) -> torch.device:
    dev = ts[0].device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for t in ts:
        if t.device != dev:
            raise ValueError("tensors must be on one CUDA device")
    return dev


def _check_nvfp4(t: NVFP4Tensor, rows: int, cols: int, name: str) -> NVFP4Tensor:
    """The buffers of `t` can hold an NVFP4 [rows, cols] tensor: the shape it
    records is (rows, cols), and QDATA, scales and record are contiguous
    uint8 buffers of at least the bytes the kernels read or write."""
    if t.rows != rows or t.cols != cols:
        raise ValueError(f"{name} holds a [{t.rows}, {t.cols}] NVFP4 tensor, [{rows}, {cols}] is needed")
    need = {"qdata": qdata_bytes(rows, cols), "scales": scale_bytes(rows, cols), "rec": 16}
    for field, n in need.items():
        b = getattr(t, field)
        if b.dtype != torch.uint8 or not b.is_contiguous():
            raise ValueError(f"{name}.{field} must be a contiguous uint8 tensor")
        if b.numel() < n:
            raise ValueError(f"{name}.{field} has {b.numel()} bytes, {n} are needed")
    return t


def _bf16_matrix(x: torch.Tensor, name: str) -> torch.Tensor:
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError(f"{name} must be a 2-D bfloat16 tensor")
    if x.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its rows")
    return x


def nvfp4_quantize_weight(w: torch.Tensor, out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    _bf16_matrix(w, "w")
    rows, cols = w.shape
    out = _check_nvfp4(out, rows, cols, "out") if out is not None else empty_nvfp4(rows, cols, w.device)
    dev = _check_dev(w, out.qdata, out.scales, out.rec)
    with torch.cuda.device(dev):
        _lib.check(load().nvfp4_quantize_weight(_ptr(w), rows, cols, w.stride(0), _ptr(out.qdata), _ptr(out.scales),
                                                _ptr(out.rec), _stream(stream)), "nvfp4_quantize_weight")
    return out


def swiglu_nvfp4_quantize(gate_up: torch.Tensor, out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    _bf16_matrix(gate_up, "gate_up")
    m, two_k = gate_up.shape
    if two_k % 2:
        raise ValueError("gate_up must have an even number of columns (gate | up)")
    k = two_k // 2
    out = _check_nvfp4(out, m, k, "out") if out is not None else empty_nvfp4(m, k, gate_up.device)
    dev = _check_dev(gate_up, out.qdata, out.scales, out.rec)
    with torch.cuda.device(dev):
        _lib.check(load().swiglu_nvfp4_quantize(_ptr(gate_up), m, k, gate_up.stride(0), _ptr(out.qdata),
                                                _ptr(out.scales), _ptr(out.rec), _stream(stream)),
                   "swiglu_nvfp4_quantize")
    return out


def nvfp4_fc2_gemm(a: NVFP4Tensor, w: NVFP4Tensor, out: torch.Tensor | None = None,
                   status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if a.cols != w.cols:
        raise ValueError("activation and weight K differ")
    m, n, k = a.rows, w.rows, a.cols
    _check_nvfp4(a, m, k, "a")
    _check_nvfp4(w, n, k, "w")
    if out is None:
        out = torch.empty(m, n, dtype=torch.bfloat16, device=a.device)
    if out.dtype != torch.bfloat16 or out.dim() != 2 or out.shape[0] < m or out.shape[1] < n or out.stride(1) != 1:
        raise ValueError("out must be a bfloat16 [>=m, >=n] tensor with unit column stride")
    dev = _check_dev(a.qdata, a.scales, a.rec, w.qdata, w.scales, w.rec, out)
    st_ptr = ctypes.c_void_p(status.data_ptr()) if status is not None else ctypes.c_void_p(0)
    with torch.cuda.device(dev):
        _lib.check(load().nvfp4_fc2_gemm(_ptr(a.qdata), _ptr(a.scales), _ptr(a.rec), _ptr(w.qdata), _ptr(w.scales),
                                         _ptr(w.rec), m, n, k, _ptr(out), out.stride(0), st_ptr, _stream(stream)),
                   "nvfp4_fc2_gemm")
    return out


def nvfp4_fc1_swiglu(a: NVFP4Tensor, w1: NVFP4Tensor, h: torch.Tensor | None = None,
                     act: NVFP4Tensor | None = None, status: torch.Tensor | None = None,
                     stream=None) -> tuple[torch.Tensor, NVFP4Tensor]:
    """FC1 with the SwiGLU producer's first pass in its epilogue, then the
    quantise pass on h: returns (h [m, f] BF16, the NVFP4 activation of FC2).
    w1 holds the gate rows then the up rows (2f rows).  The bytes equal
    swiglu_nvfp4_quantize applied to nvfp4_fc2_gemm(a, w1)."""
    if a.cols != w1.cols:
        raise ValueError("activation and weight K differ")
    if w1.rows % 2:
        raise ValueError("w1 must hold gate and up rows (an even row count)")
    m, f, k = a.rows, w1.rows // 2, a.cols
    _check_nvfp4(a, m, k, "a")
    _check_nvfp4(w1, 2 * f, k, "w1")
    if h is None:
        h = torch.empty(m, f, dtype=torch.bfloat16, device=a.device)
    if h.dtype != torch.bfloat16 or h.dim() != 2 or h.shape[0] < m or h.shape[1] < f or h.stride(1) != 1:
        raise ValueError("h must be a bfloat16 [>=m, >=f] tensor with unit column stride")
    act = _check_nvfp4(act, m, f, "act") if act is not None else empty_nvfp4(m, f, a.device)
    dev = _check_dev(a.qdata, a.scales, a.rec, w1.qdata, w1.scales, w1.rec, h, act.qdata, act.scales, act.rec)
    st_ptr = ctypes.c_void_p(status.data_ptr()) if status is not None else ctypes.c_void_p(0)
    with torch.cuda.device(dev):
        L = load()
        _lib.check(L.nvfp4_fc1_swiglu(_ptr(a.qdata), _ptr(a.scales), _ptr(a.rec), _ptr(w1.qdata), _ptr(w1.scales),
                                      _ptr(w1.rec), m, f, k, _ptr(h), h.stride(0), _ptr(act.rec), st_ptr,
                                      _stream(stream)), "nvfp4_fc1_swiglu")
        _lib.check(L.nvfp4_quantize_with_amax(_ptr(h), m, f, h.stride(0), _ptr(act.qdata), _ptr(act.scales),
                                              _ptr(act.rec), _stream(stream)), "nvfp4_quantize_with_amax")
    return h, act


def fc2(gate_up: torch.Tensor, w: NVFP4Tensor, act: NVFP4Tensor | None = None, out: torch.Tensor | None = None,
        stream=None) -> torch.Tensor:
    """One FC2 step on device tensors: SwiGLU + NVFP4 quantise, then GEMM."""
    act = swiglu_nvfp4_quantize(gate_up, act, stream)
    return nvfp4_fc2_gemm(act, w, out, None, stream)


def fc2_host(gate_up_host: torch.Tensor, w: NVFP4Tensor, workspace: dict | None = None, stream=None,
             out_host: torch.Tensor | None = None, sync: bool = True):
    """FC2 from host memory to host memory through nvfp4_fc2_host: the C call
    copies gate|up to the device, runs the step and copies the BF16 output
    back, all on `stream`.  Pinned host tensors make the copies
    asynchronous; `workspace` (a dict) keeps the device buffers between
    calls.

    With ``sync=False`` the call returns ``(out_host, event)`` as soon as the
    work is queued on `stream`; `out_host` is valid, and `workspace` and
    `gate_up_host` may be reused, once `event` has completed.  Two workspaces
    on two streams let one step's copies overlap another step's kernels."""
    _bf16_matrix(gate_up_host, "gate_up_host")
    if gate_up_host.device.type != "cpu":
        raise ValueError("gate_up_host must be a host tensor")
    m, two_k = gate_up_host.shape
    k = two_k // 2
    n = w.rows
    _check_nvfp4(w, n, k, "w")
    ws = workspace if workspace is not None else {}
    dev = w.device
    key = (m, k, n)
    if ws.get("key") != key:
        ws.clear()
        ws["key"] = key
        ws["x"] = torch.empty(m, two_k, dtype=torch.bfloat16, device=dev)
        ws["act"] = empty_nvfp4(m, k, dev)
        ws["out"] = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
    if out_host is None:
        out_host = torch.empty(m, n, dtype=torch.bfloat16, pin_memory=True)
    if (out_host.dtype != torch.bfloat16 or out_host.device.type != "cpu" or tuple(out_host.shape) != (m, n)
            or not out_host.is_contiguous()):
        raise ValueError("out_host must be a contiguous host bfloat16 [m, n] tensor")
    s = torch.cuda.current_stream(dev) if stream is None else stream
    act = ws["act"]
    with torch.cuda.device(dev):
        _lib.check(load().nvfp4_fc2_host(_ptr(gate_up_host), m, k, gate_up_host.stride(0), _ptr(w.qdata),
                                         _ptr(w.scales), _ptr(w.rec), n, _ptr(ws["x"]), _ptr(act.qdata),
                                         _ptr(act.scales), _ptr(act.rec), _ptr(ws["out"]), _ptr(out_host),
                                         ctypes.c_void_p(0), ctypes.c_void_p(s.cuda_stream)), "nvfp4_fc2_host")
    if sync:
        s.synchronize()
        return out_host
    ev = torch.cuda.Event()
    ev.record(s)
    return out_host, ev
