"""GEMM parity on the GPU: BF16 output against the oracle's unrounded FP64
reference, |gpu - ref| <= 1e-2|ref| + 1e-3 rms(ref) elementwise -- on all
rows for the tiny and mid FC2 workloads and small shapes that span several
tiles and a ragged M tail, on 1024 seeded rows (seed + 7) for the canonical
and ragged-M workloads; plus row invariance across M, run-to-run
determinism, untouched bytes outside [m, n], and the status word."""
import numpy as np
import pytest
import torch

import diffusion_transformer_mlp_gb300 as fc2
import oracle
import synth
from _edge import grid_matrix
from _util import compare_quant, gemm_check, sample_rows, to_dev_bf16

pytestmark = pytest.mark.gpu


def build_case(m, n, k, seed):
    x = synth.activation(m, k, seed=seed)
    w = synth.weight(n, k, seed=seed)
    a_ref = oracle.quantize(x, k, swiglu=True)
    w_ref = oracle.quantize(w, k, swiglu=False)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    w_dev = fc2.nvfp4_quantize_weight(wd)
    a_dev = fc2.swiglu_nvfp4_quantize(xd)
    return a_ref, w_ref, a_dev, w_dev, xd


@pytest.mark.parametrize("m,n,k", [(256, 512, 1024), (128, 128, 256), (200, 256, 512), (1, 128, 256),
                                   (1000, 384, 2048), (333, 640, 768)])
def test_gemm_all_rows_small(m, n, k):
    a_ref, w_ref, a_dev, w_dev, _ = build_case(m, n, k, seed=m + n + k)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    (ok, worst), ref, got = gemm_check(out, a_ref, w_ref, np.arange(m), n, k)
    assert ok, f"worst error / bound = {worst}"


def test_gemm_mid_all_rows():
    """Mid FC2: M=4096, K=14336, N=5376, full-output check."""
    m, n, k = 4096, 5376, 14336
    a_ref, w_ref, a_dev, w_dev, _ = build_case(m, n, k, seed=0)
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    (ok, worst), _, _ = gemm_check(out, a_ref, w_ref, np.arange(m), n, k)
    assert ok, f"worst error / bound = {worst}"


def test_gemm_clock_record_same_output():
    """nvfp4_diag_fc2_gemm_clock runs the same kernel: its output equals
    nvfp4_fc2_gemm's bit for bit, and its clock record is consistent (end
    after start on both clocks, an SM clock between 0.3 and 2.5 GHz)."""
    import ctypes

    from diffusion_transformer_mlp_gb300 import _lib
    m, n, k = 1000, 384, 2048
    _, _, a_dev, w_dev, _ = build_case(m, n, k, seed=11)
    ref = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    out = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    clk = torch.zeros(4, dtype=torch.int64, device="cuda")
    vp = ctypes.c_void_p
    L = _lib.load()
    _lib.check(L.nvfp4_diag_fc2_gemm_clock(vp(a_dev.qdata.data_ptr()), vp(a_dev.scales.data_ptr()),
                                           vp(a_dev.rec.data_ptr()), vp(w_dev.qdata.data_ptr()),
                                           vp(w_dev.scales.data_ptr()), vp(w_dev.rec.data_ptr()), m, n, k,
                                           vp(out.data_ptr()), n, vp(st.data_ptr()), vp(clk.data_ptr()),
                                           vp(torch.cuda.current_stream().cuda_stream)), "gemm clock")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    t0, t1, c0, c1 = (int(v) for v in clk.cpu())
    assert t1 > t0 and c1 > c0
    assert 300 < 1e3 * (c1 - c0) / (t1 - t0) < 2500


def test_gemm_output_bounds_untouched():
    """Rows >= m and columns >= n of a wider output buffer keep their bytes."""
    m, n, k = 130, 256, 512
    _, _, a_dev, w_dev, _ = build_case(m, n, k, seed=4)
    big = torch.full((m + 7, n + 40), 3.0, dtype=torch.bfloat16, device="cuda")
    fc2.nvfp4_fc2_gemm(a_dev, w_dev, out=big[:, : n + 40])
    torch.cuda.synchronize()
    assert torch.all(big[m:] == 3.0) and torch.all(big[:m, n:] == 3.0)
    assert not torch.all(big[:m, :n] == 3.0)


def test_gemm_output_view_at_column_offset():
    """The output as a view that starts 8 columns (16 bytes) into a wider
    buffer, rows 304 columns apart: the TMA-store epilogue writes the same
    bytes as into a packed buffer, and nothing outside the view."""
    m, n, k = 300, 384, 1024
    _, _, a_dev, w_dev, _ = build_case(m, n, k, seed=21)
    ref = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    big = torch.full((m, n + 304 - n % 8), 7.0, dtype=torch.bfloat16, device="cuda")
    view = big[:, 8: 8 + n]
    assert view.data_ptr() % 32 == 16
    fc2.nvfp4_fc2_gemm(a_dev, w_dev, out=view)
    torch.cuda.synchronize()
    assert torch.equal(view.view(torch.int16), ref.view(torch.int16))
    assert torch.all(big[:, :8] == 7.0) and torch.all(big[:, 8 + n:] == 7.0)


def test_gemm_nonfinite_record_propagates_nan():
    m, n, k = 64, 128, 256
    _, _, a_dev, w_dev, xd = build_case(m, n, k, seed=5)
    xd[3, 7] = float("inf")
    a_dev = fc2.swiglu_nvfp4_quantize(xd)
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    assert fc2.read_rec(a_dev)["status"] == fc2._lib.NVFP4_ENONFINITE
    assert torch.isnan(out.float()).all()


@pytest.fixture(scope="module")
def canonical():
    m, n, k = 37810, 5376, 14336
    return (m, n, k) + build_case(m, n, k, seed=0)


def test_gemm_canonical_sampled_rows(canonical):
    m, n, k, a_ref, w_ref, a_dev, w_dev, _ = canonical
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    rows = sample_rows(m, 1024, seed=0 + 7)
    (ok, worst), _, _ = gemm_check(out, a_ref, w_ref, rows, n, k)
    assert ok, f"worst error / bound = {worst}"


RAGGED = [37711, 37725, 37742, 37774, 37809, 37838, 37966, 38222]


@pytest.mark.parametrize("m", RAGGED)
def test_gemm_ragged_m(m):
    """Ragged-M sweep: producer bytes exact, output rows within tolerance on
    1024 sampled rows (always including the last row), 50 back-to-back runs
    with identical bytes."""
    n, k = 5376, 14336
    a_ref, w_ref, a_dev, w_dev, xd = build_case(m, n, k, seed=0)
    assert compare_quant(a_dev, *a_ref, m, k) is None
    out0 = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    rows = sample_rows(m, 1024, seed=0 + 7)
    (ok, worst), _, _ = gemm_check(out0, a_ref, w_ref, rows, n, k)
    assert ok, f"M={m}: worst error / bound = {worst}"
    # 50 whole steps (producer into the same activation buffers, then the
    # GEMM) queued back to back on one stream, each into its own output,
    # with one synchronisation at the end
    outs = [torch.empty_like(out0) for _ in range(50)]
    for out in outs:
        fc2.fc2(xd, w_dev, a_dev, out)
    torch.cuda.synchronize()
    for i, out in enumerate(outs):
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16)), f"run {i}"
    assert compare_quant(a_dev, *a_ref, m, k) is None


def test_gemm_row_invariance_across_m(canonical):
    """Output row r is bit-identical for every M of the ragged sweep (r < M):
    the K reduction order does not depend on M.  The same NVFP4 activation
    bytes are passed with each M (a row-major prefix of QDATA and whole
    128-row scale panels)."""
    m0, n, k, _, _, a_dev, w_dev, _ = canonical
    base = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    for m in [37711, 37725, 37742, 37774, 37809, 1, 128, 129]:
        a_m = fc2.NVFP4Tensor(a_dev.qdata, a_dev.scales, a_dev.rec, m, k)
        out = fc2.nvfp4_fc2_gemm(a_m, w_dev)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), base[:m].view(torch.int16)), m


def test_fc2_host_matches_device_step():
    """fc2_host (pinned host gate|up in, host BF16 out), synchronous and
    queued on two streams with two workspaces, gives the bytes of the
    device-side step."""
    m, n, k = 300, 256, 1024
    x = synth.activation(m, k, seed=11)
    w = synth.weight(n, k, seed=11)
    wq = fc2.nvfp4_quantize_weight(to_dev_bf16(w))
    ref = fc2.fc2(to_dev_bf16(x), wq)
    torch.cuda.synchronize()
    x_host = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    got = fc2.fc2_host(x_host, wq)
    assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16))
    # queued steps on two streams (their host-to-device copies ordered across
    # the streams by the library), three inputs in turn: every step's output
    # is checked when its slot comes round again
    x3 = [x_host] + [torch.from_numpy(synth.activation(m, k, seed=12 + i).view(np.int16)).view(torch.bfloat16)
                     .pin_memory() for i in range(2)]
    ref3 = [ref.cpu()] + [fc2.fc2(xi.to("cuda"), wq).cpu() for xi in x3[1:]]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [{}, {}]
    outs = [torch.empty(m, n, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    evs, last = [None, None], [None, None]
    for i in range(9):
        j = i % 2
        if evs[j] is not None:
            evs[j].synchronize()
            assert torch.equal(outs[j].view(torch.int16), ref3[last[j]].view(torch.int16)), (i, j)
        _, evs[j] = fc2.fc2_host(x3[i % 3], wq, wss[j], streams[j], outs[j], sync=False)
        last[j] = i % 3
    for j in range(2):
        evs[j].synchronize()
        assert torch.equal(outs[j].view(torch.int16), ref3[last[j]].view(torch.int16))
    # a host input whose rows are longer than 2k (the copy takes the first 2k)
    wide = torch.zeros(m, 2 * k + 64, dtype=torch.bfloat16).pin_memory()
    wide[:, : 2 * k] = x_host
    got = fc2.fc2_host(wide[:, : 2 * k], wq)
    assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16))


# FC1 on the same kernel: M x (2 * 14336) x 5376.  Its input is the block's
# modulated hidden state, whose modulation is not on the pages; here it is a
# BF16 [M, 5376] matrix of the activation law, quantised to NVFP4 by the
# plain (non-SwiGLU) quantiser.  K = 5376 is 21 k-tiles: an odd count.
FC1_N, FC1_K = 2 * 14336, 5376


def build_fc1_case(m, seed):
    x = synth.quant_input(m, FC1_K, seed=seed)
    w = synth.weight(FC1_N, FC1_K, seed=seed)
    a_ref = oracle.quantize(x, FC1_K, swiglu=False)
    w_ref = oracle.quantize(w, FC1_K, swiglu=False)
    a_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(x))
    w_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(w))
    return a_ref, w_ref, a_dev, w_dev


def test_fc1_all_rows():
    """FC1 shape, M = 300 (a ragged 256-row tile): every output element."""
    m = 300
    a_ref, w_ref, a_dev, w_dev = build_fc1_case(m, seed=11)
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    (ok, worst), _, _ = gemm_check(out, a_ref, w_ref, np.arange(m), FC1_N, FC1_K)
    assert ok, f"worst error / bound = {worst}"


def test_fc1_canonical_sampled_rows():
    """FC1 at the canonical M = 37810: 1024 seeded rows, and the output is
    the gate|up layout the SwiGLU producer reads (N = 2 x 14336)."""
    m = 37810
    a_ref, w_ref, a_dev, w_dev = build_fc1_case(m, seed=12)
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (m, FC1_N)
    rows = sample_rows(m, 1024, seed=12 + 7)
    (ok, worst), _, _ = gemm_check(out, a_ref, w_ref, rows, FC1_N, FC1_K)
    assert ok, f"worst error / bound = {worst}"


def _fc1_fused_vs_unfused(m, f, k, seed):
    """Composition check on the activation law: nvfp4_fc1_swiglu + quantise
    pass against nvfp4_fc2_gemm (BF16 gate|up) + swiglu_nvfp4_quantize give
    the same NVFP4 activation bytes and record, and h equals the producer's
    SwiGLU of the unfused gate|up."""
    x = synth.quant_input(m, k, seed=seed)
    w = synth.weight(2 * f, k, seed=seed)
    a_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(x))
    w_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(w))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gate_up = fc2.nvfp4_fc2_gemm(a_dev, w_dev, status=status)
    act_u = fc2.swiglu_nvfp4_quantize(gate_up)
    h, act_f = fc2.nvfp4_fc1_swiglu(a_dev, w_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert fc2.read_rec(act_f) == fc2.read_rec(act_u)
    assert torch.equal(act_f.qdata, act_u.qdata)
    assert torch.equal(act_f.scales, act_u.scales)
    # h against the producer's own SwiGLU of the unfused output
    L = fc2._lib.load()
    g = gate_up[:, :f].contiguous().view(torch.int16)
    u = gate_up[:, f:].contiguous().view(torch.int16)
    h_ref = torch.empty_like(g)
    fc2._lib.check(L.nvfp4_diag_swiglu(fc2._ptr(g), fc2._ptr(u), fc2._ptr(h_ref), g.numel(),
                                       fc2._stream(None)), "swiglu")
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), h_ref)


@pytest.mark.parametrize("m,f,k", [(300, 256, 512), (1, 128, 256), (257, 384, 768)])
def test_fc1_swiglu_fused_small(m, f, k):
    _fc1_fused_vs_unfused(m, f, k, seed=m + f + k)


def test_fc1_swiglu_fused_canonical():
    """FC1 at the canonical size, f = 14336, k = 5376, M = 37810."""
    _fc1_fused_vs_unfused(37810, 14336, 5376, seed=21)


def exact_case(m, n, k, seed):
    """NVFP4 operands whose FP32 accumulation is exact (grid inputs, unit
    scales; tests/_edge.py), with the oracle's bytes for both, the device
    tensors, and the oracle's exact FP64 products for all rows."""
    x = grid_matrix(m, k, seed, 0)
    w = grid_matrix(n, k, seed + 1, 16)
    a_ref = oracle.quantize(x, k, swiglu=False)
    w_ref = oracle.quantize(w, k, swiglu=False)
    a_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(x))
    w_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(w))
    torch.cuda.synchronize()
    assert compare_quant(a_dev, *a_ref, m, k) is None and compare_quant(w_dev, *w_ref, n, k) is None
    return a_ref, w_ref, a_dev, w_dev


@pytest.mark.parametrize("m,n,k", [(300, 256, 1024), (1000, 384, 2048), (130, 5376, 14336), (129, 28672, 5376)])
def test_gemm_bit_exact_when_accumulation_is_exact(m, n, k):
    """Every output element equals the oracle's RNE_bf16(RN(acc * alpha)) bit
    for bit when no partial sum rounds: the epilogue's arithmetic (alpha,
    the binary32 product, the BF16 rounding) pinned exactly, not within a
    tolerance."""
    a_ref, w_ref, a_dev, w_dev = exact_case(m, n, k, seed=m + n + k)
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    ref = oracle.gemm_rows(a_ref[0], a_ref[1], a_ref[2]["global_scale"], w_ref[0], w_ref[1],
                           w_ref[2]["global_scale"], n, k, np.arange(m))
    alpha = np.float32(a_ref[2]["global_scale"]) * np.float32(w_ref[2]["global_scale"])
    want = oracle.epilogue_bf16(ref, alpha)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} elements differ; first {tuple(bad[0])}"


def _fc1_fused_vs_oracle(m, f, k, seed, rows=None):
    """nvfp4_fc1_swiglu + its quantise pass against the oracle on operands
    whose FC1 accumulation is exact: the oracle forms FC1's BF16 gate|up
    (its epilogue rounding of the exact FP64 products), then h and the
    two-pass NVFP4 bytes of h.  h is compared bit for bit on `rows` (all
    rows by default); with all rows the QDATA, scales and record are too.
    With a row sample, the record's max is checked against the h the same
    call wrote."""
    a_ref, w_ref, a_dev, w_dev = exact_case(m, 2 * f, k, seed)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    h, act = fc2.nvfp4_fc1_swiglu(a_dev, w_dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.arange(m) if rows is None else rows
    ref = oracle.gemm_rows(a_ref[0], a_ref[1], a_ref[2]["global_scale"], w_ref[0], w_ref[1],
                           w_ref[2]["global_scale"], 2 * f, k, sel)
    alpha = np.float32(a_ref[2]["global_scale"]) * np.float32(w_ref[2]["global_scale"])
    gate_up = oracle.epilogue_bf16(ref, alpha)
    h_want = oracle.swiglu_rows(gate_up, f)
    h_got = h[torch.from_numpy(sel).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    bad = np.argwhere(h_got != h_want)
    assert bad.size == 0, f"h: {len(bad)} elements differ; first {tuple(bad[0])}"
    if rows is None:
        q, s, rec = oracle.quantize(gate_up, f, swiglu=True)
        err = compare_quant(act, q, s, rec, m, f)
        assert err is None, err
    else:
        hmax = h.float().abs().max().item()
        assert fc2.read_rec(act)["amax_bits"] == int(np.float32(hmax).view(np.uint32))


@pytest.mark.parametrize("m,f,k", [(300, 256, 512), (1, 128, 256), (257, 384, 768), (513, 1024, 5376)])
def test_fc1_swiglu_fused_matches_oracle(m, f, k):
    _fc1_fused_vs_oracle(m, f, k, seed=m + f + k)


def test_fc1_swiglu_fused_matches_oracle_canonical_rows():
    """Canonical FC1 shape (M = 37810, f = 14336, k = 5376): h on 256 seeded
    rows (always the first and the last) bit-exact against the oracle."""
    m = 37810
    _fc1_fused_vs_oracle(m, 14336, 5376, seed=31, rows=sample_rows(m, 256, seed=31 + 7))


# The block's other NVFP4 projections on the same kernel.  The pages give
# their launch grids (296 x 168 and 296 x 42 tiles of 128 x 128): N = 21504
# for qkv and N = 5376 for attention_output.  qkv reads the hidden state
# (K = 5376; 21504 = 3 x 7168); attention_output reads the 7168-feature
# attention output ("GB10 component-2 nsys summary", native_pack_validation)
# and writes the hidden size.
@pytest.mark.parametrize("n,k", [(21504, 5376), (5376, 7168)], ids=["qkv", "attention_output"])
def test_block_projection_sampled_rows(n, k):
    m = 37810
    x = synth.quant_input(m, k, seed=n)
    w = synth.weight(n, k, seed=n)
    a_ref = oracle.quantize(x, k, swiglu=False)
    w_ref = oracle.quantize(w, k, swiglu=False)
    a_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(x))
    w_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(w))
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    rows = sample_rows(m, 512, seed=n + 7)
    (ok, worst), _, _ = gemm_check(out, a_ref, w_ref, rows, n, k)
    assert ok, f"worst error / bound = {worst}"


def test_fc1_swiglu_nonfinite_propagates():
    """An Inf in FC1's input makes FC1's outputs, h and its global max
    non-finite: the record says so, and FC2 on that activation gives NaN --
    the same outcome as the unfused path."""
    m, f, k = 64, 256, 256
    x = synth.quant_input(m, k, seed=9)
    w = synth.weight(2 * f, k, seed=9)
    xd = to_dev_bf16(x)
    xd[5, 3] = float("inf")
    a_dev = fc2.nvfp4_quantize_weight(xd)
    w_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(w))
    _, act_f = fc2.nvfp4_fc1_swiglu(a_dev, w_dev)
    act_u = fc2.swiglu_nvfp4_quantize(fc2.nvfp4_fc2_gemm(a_dev, w_dev))
    torch.cuda.synchronize()
    rf, ru = fc2.read_rec(act_f), fc2.read_rec(act_u)
    assert rf["status"] == ru["status"] == fc2._lib.NVFP4_ENONFINITE
    assert rf["amax_bits"] == ru["amax_bits"] >= 0x7F800000
    w2 = fc2.nvfp4_quantize_weight(to_dev_bf16(synth.weight(128, f, seed=9)))
    out = fc2.nvfp4_fc2_gemm(act_f, w2)
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()


@pytest.mark.parametrize("m,n,k", [(37810, 5376, 14336), (37810, 28672, 5376)], ids=["fc2", "fc1"])
def test_gemm_full_output_matches_library(m, n, k):
    """Every output element of the canonical-size GEMM against an independent
    block-scaled NVFP4 matmul (cuBLASLt) on the same NVFP4 bytes, times the
    same alpha: |gpu - lib| <= 1e-2 |lib| + 1e-3 rms(lib).  The oracle covers
    1,024 seeded rows of this shape (its FP64 GEMM over all rows is beyond
    the CPU); this covers all of them."""
    import _cublaslt
    x = synth.quant_input(m, k, seed=m % 97 + n % 89)
    w = synth.weight(n, k, seed=n % 83)
    a_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(x))
    w_dev = fc2.nvfp4_quantize_weight(to_dev_bf16(w))
    out = fc2.nvfp4_fc2_gemm(a_dev, w_dev)
    torch.cuda.synchronize()
    lib = _cublaslt.nvfp4_matmul(a_dev.qdata, a_dev.scales, w_dev.qdata, w_dev.scales, m, n, k)
    alpha = np.float32(fc2.read_rec(a_dev)["global_scale"]) * np.float32(fc2.read_rec(w_dev)["global_scale"])
    ref = lib * float(alpha)
    rms = ref.double().pow(2).mean().sqrt().item()
    err = (out.float() - ref).abs()
    bound = 1e-2 * ref.abs() + 1e-3 * rms
    worst = (err / bound).max().item()
    assert bool((err <= bound).all()), f"worst error / bound = {worst}"
