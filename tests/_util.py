"""Helpers shared by the GPU parity tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def to_dev_bf16(x: np.ndarray) -> torch.Tensor:
    """uint16 BF16 bit patterns (host) -> bf16 CUDA tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rec_tuple(rec: dict):
    g = np.float32(rec["global_scale"])
    return (int(g.view(np.uint32)) if not np.isnan(g) else "nan", rec["amax_bits"], rec["status"])


def compare_quant(dev, q_ref, s_ref, rec_ref, rows, cols):
    """Bytes of the device NVFP4 tensor equal the oracle's (QDATA, scales,
    record); returns a short description of the first difference or None."""
    import diffusion_transformer_mlp_gb300 as fc2
    q = dev.qdata.cpu().numpy()
    s = dev.scales.cpu().numpy()
    rec = fc2.read_rec(dev)
    if rec["status"] != rec_ref["status"]:
        return f"status {rec['status']} != {rec_ref['status']}"
    if rec_ref["status"] == 0:
        if rec["amax_bits"] != rec_ref["amax_bits"]:
            return f"amax bits {rec['amax_bits']:#x} != {rec_ref['amax_bits']:#x}"
        if np.float32(rec["global_scale"]).view(np.uint32) != np.float32(rec_ref["global_scale"]).view(np.uint32):
            return f"global scale {rec['global_scale']} != {rec_ref['global_scale']}"
    else:
        if not np.isnan(rec["global_scale"]) or rec["amax_bits"] < 0x7F800000:
            return "non-finite record not flagged"
    if q.shape != q_ref.shape or s.shape != s_ref.shape:
        return f"shape {q.shape}/{s.shape} vs {q_ref.shape}/{s_ref.shape}"
    dq = np.nonzero(q != q_ref)
    if dq[0].size:
        r, c = dq[0][0], dq[1][0]
        return f"{dq[0].size} QDATA bytes differ; first at row {r} byte {c}: {q[r, c]:#x} vs {q_ref[r, c]:#x}"
    ds = np.nonzero(s != s_ref)[0]
    if ds.size:
        return f"{ds.size} scale bytes differ; first at offset {ds[0]}: {s[ds[0]]:#x} vs {s_ref[ds[0]]:#x}"
    return None


def sample_rows(m: int, count: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    if count >= m:
        return np.arange(m)
    rows = np.sort(rng.choice(m, size=count, replace=False))
    # always include the first and the last rows (tile edges / ragged tail)
    return np.unique(np.concatenate([[0, m - 1], rows]))


def gemm_check(out: torch.Tensor, a_ref, w_ref, rows: np.ndarray, n: int, k: int):
    """Compare device BF16 output rows with the oracle's FP64 reference under
    |gpu - ref| <= 1e-2|ref| + 1e-3 rms(ref)."""
    aq, as_, ar = a_ref
    wq, ws, wr = w_ref
    ref = oracle.gemm_rows(aq, as_, ar["global_scale"], wq, ws, wr["global_scale"], n, k, rows)
    got = out[torch.from_numpy(rows).to(out.device)].float().cpu().numpy().astype(np.float64)
    return oracle.check_gemm_tolerance(got, ref), ref, got
