"""Producer parity on the GPU: QDATA, scale bytes and the global-scale record
of both quantisers are bit-exact against the oracle, for small shapes that
span several tiles and a ragged tail, the hand-worked blocks, inputs built
to reach every UE4M3 block-scale code and the recipe's ties and zeros, the
quantise-only workload at feature widths 5376 / 7168 / 14336 (M = 37,810,
padded), and the canonical SwiGLU producer (M = 37,810, K = 14,336)."""
import json
import os

import numpy as np
import pytest
import torch

import diffusion_transformer_mlp_gb300 as fc2
import oracle
import synth
from _edge import E4M3, edge_matrix, swiglu_input
from _util import compare_quant, to_dev_bf16

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_weight(x: np.ndarray, cols: int):
    dev = fc2.nvfp4_quantize_weight(to_dev_bf16(x)[:, :cols])
    torch.cuda.synchronize()
    return dev


def run_swiglu(x: np.ndarray, k: int):
    dev = fc2.swiglu_nvfp4_quantize(to_dev_bf16(x)[:, : 2 * k])
    torch.cuda.synchronize()
    return dev


# Widths for each walk of the plain quantiser's second pass: whole 1024-element
# units (1024, 7168), multiples of 64 from 1024 up that are not (1088, 1344,
# 3136, 5376: the grid read as one sequence of units, which crosses row ends),
# and the rest (16, 272, 1040: one block a lane along each row).
@pytest.mark.parametrize("rows,cols", [(256, 1024), (1, 16), (300, 1040), (129, 272), (37, 5376), (513, 7168),
                                       (129, 1088), (1, 1344), (300, 3136), (640, 1344)])
def test_weight_quantizer_bit_exact_small(rows, cols):
    x = synth.quant_input(rows, cols, seed=rows + cols)
    q, s, rec = oracle.quantize(x, cols, swiglu=False)
    err = compare_quant(run_weight(x, cols), q, s, rec, rows, cols)
    assert err is None, err


def test_weight_quantizer_strided_rows_across_row_ends():
    """The sequence-of-units walk on rows longer than cols (ld > cols): only
    the first cols columns of each row are read, codes and scales exact."""
    rows, cols, ld = 200, 1344, 1344 + 192
    full = synth.quant_input(rows, ld, seed=17)
    q, s, rec = oracle.quantize(full[:, :cols].copy(), cols, swiglu=False)
    dev = fc2.nvfp4_quantize_weight(to_dev_bf16(full)[:, :cols])
    torch.cuda.synchronize()
    assert compare_quant(dev, q, s, rec, rows, cols) is None


@pytest.mark.parametrize("rows,k", [(256, 1024), (1, 16), (300, 1040), (131, 4096), (64, 48)])
def test_swiglu_producer_bit_exact_small(rows, k):
    x = synth.activation(rows, k, seed=rows * 3 + k)
    q, s, rec = oracle.quantize(x, k, swiglu=True)
    err = compare_quant(run_swiglu(x, k), q, s, rec, rows, k)
    assert err is None, err


def test_strided_input_rows():
    """ld larger than the row: only the first cols (2k) columns are read."""
    rows, k, ld = 70, 256, 2 * 256 + 64
    full = synth.normal_bf16((rows, ld), 9, 0, 1.0, 1e-3)
    q, s, rec = oracle.quantize(full, k, swiglu=True)
    dev = fc2.swiglu_nvfp4_quantize(to_dev_bf16(full)[:, : 2 * k])
    torch.cuda.synchronize()
    assert compare_quant(dev, q, s, rec, rows, k) is None


def test_hand_worked_blocks_on_device():
    fx = json.load(open(os.path.join(ROOT, "tests", "golden", "hand_blocks.json")))
    cols = fx["cols"]
    row = fx["rows"][0]
    x = torch.tensor(row["values"], dtype=torch.float32).to(torch.bfloat16).view(1, cols)
    dev = fc2.nvfp4_quantize_weight(x.cuda())
    torch.cuda.synchronize()
    assert list(dev.qdata[0].cpu().numpy()) == row["qdata"]
    sc = dev.scales.cpu().numpy()
    assert [int(sc[fc2.scale_offset(0, c, cols)]) for c in range(3)] == row["scale_codes"]
    rec = fc2.read_rec(dev)
    assert rec["global_scale"] == row["global_scale"] and rec["status"] == 0
    assert not dev.qdata[1:].any() and int(dev.scales.sum()) == sum(row["scale_codes"])


@pytest.mark.parametrize("rows,cols", [(300, 16), (300, 48), (300, 272), (257, 1024)])
def test_edge_blocks_bit_exact(rows, cols):
    """Every UE4M3 scale code 0x00..0x7E (subnormals included), ratios half
    way between two codes, ratios that round to 0, all-zero and all -0
    blocks inside a non-zero tensor, negatives that encode as E2M1 -0, and
    element values on E2M1 rounding midpoints; both quantisers (the SwiGLU
    one through gate = 8, up = h / 8, whose SwiGLU is h)."""
    x = edge_matrix(rows, cols, seed=rows + cols)
    q, s, rec = oracle.quantize(x, cols, swiglu=False)
    assert rec["global_scale"] == np.float32(1.0)
    codes = {int(s[oracle.scale_offset(r, b, cols)]) for r in range(rows) for b in range(cols // 16)}
    assert codes == set(range(len(E4M3)))
    err = compare_quant(run_weight(x, cols), q, s, rec, rows, cols)
    assert err is None, err
    gu = swiglu_input(x)
    qs, ss, recs = oracle.quantize(gu, cols, swiglu=True)
    assert np.array_equal(qs, q) and np.array_equal(ss, s)
    err = compare_quant(run_swiglu(gu, cols), qs, ss, recs, rows, cols)
    assert err is None, err


@pytest.mark.parametrize("factor", [0.3701171875, 1.0009765625e-30, 3.0e30])
def test_edge_blocks_other_global_scales(factor):
    """The same blocks scaled by a BF16 factor (truncated toward zero), so the
    global scale is no longer 1 and reaches the tiny and huge ends of
    binary32."""
    rows, cols = 300, 272
    xf = (edge_matrix(rows, cols, seed=7).astype(np.uint32) << 16).view(np.float32) * np.float32(factor)
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)
    q, s, rec = oracle.quantize(x, cols, swiglu=False)
    err = compare_quant(run_weight(x, cols), q, s, rec, rows, cols)
    assert err is None, err


@pytest.mark.parametrize("cols", [64, 1024, 1344])  # one block a lane, two along rows, two across row ends
def test_zero_input_and_nonfinite_status(cols):
    x = np.zeros((200, cols), dtype=np.uint16)
    dev = run_weight(x, cols)
    r = fc2.read_rec(dev)
    assert r["status"] == 0 and r["global_scale"] == 0.0 and not dev.qdata.any() and not dev.scales.any()
    x[150, 17] = 0x7FC0  # NaN
    dev = run_weight(x, cols)
    r = fc2.read_rec(dev)
    assert r["status"] == fc2._lib.NVFP4_ENONFINITE and np.isnan(r["global_scale"])
    assert not dev.qdata.any() and not dev.scales.any()
    g = np.zeros((3, 64), dtype=np.uint16)
    g[1, 0] = 0xFF80  # gate -inf
    dev = run_swiglu(g, 32)
    assert fc2.read_rec(dev)["status"] == fc2._lib.NVFP4_ENONFINITE


def test_outputs_fully_overwritten():
    """Stale bytes in reused buffers (pad rows, pad scale columns) are
    overwritten: run into buffers pre-filled with 0xAB."""
    rows, k = 130, 48   # 3 scale columns -> 1 pad column; 126 pad rows
    x = synth.activation(rows, k, seed=2)
    q, s, rec = oracle.quantize(x, k, swiglu=True)
    out = fc2.empty_nvfp4(rows, k)
    out.qdata.fill_(0xAB)
    out.scales.fill_(0xAB)
    out.rec.fill_(0xAB)
    fc2.swiglu_nvfp4_quantize(to_dev_bf16(x), out)
    torch.cuda.synchronize()
    assert compare_quant(out, q, s, rec, rows, k) is None


@pytest.mark.parametrize("cols", [48, 1024, 1344])
def test_plain_outputs_fully_overwritten(cols):
    """The plain quantiser on each walk writes every QDATA and scale byte of
    the padded grid (126 pad rows; 48 columns also leave a pad scale column)
    into buffers pre-filled with 0xAB."""
    rows = 130
    x = synth.quant_input(rows, cols, seed=cols)
    q, s, rec = oracle.quantize(x, cols, swiglu=False)
    out = fc2.empty_nvfp4(rows, cols)
    out.qdata.fill_(0xAB)
    out.scales.fill_(0xAB)
    out.rec.fill_(0xAB)
    fc2.nvfp4_quantize_weight(to_dev_bf16(x), out)
    torch.cuda.synchronize()
    assert compare_quant(out, q, s, rec, rows, cols) is None


@pytest.mark.parametrize("f", [5376, 7168, 14336])
def test_quantize_only_full_size_bit_exact(f):
    """Quantise-only workload: BF16 [37810, F], N(0,1) with 0.1% x20, two-pass
    absmax + pack + 128x4 swizzle, M padded to 37,888 with zero rows."""
    m = 37810
    x = synth.quant_input(m, f, seed=0)
    q, s, rec = oracle.quantize(x, f, swiglu=False)
    err = compare_quant(run_weight(x, f), q, s, rec, m, f)
    assert err is None, err


def test_canonical_swiglu_producer_bit_exact():
    """Canonical producer: gate|up BF16 [37810, 2*14336] -> NVFP4 [37888, 14336]."""
    m, k = 37810, 14336
    x = synth.activation(m, k, seed=0)
    q, s, rec = oracle.quantize(x, k, swiglu=True)
    err = compare_quant(run_swiglu(x, k), q, s, rec, m, k)
    assert err is None, err
