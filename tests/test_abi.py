"""The C ABI without a GPU: the library loads, exports every symbol the
headers declare, its size queries agree with the oracle and the pages'
byte counts, and argument errors come back synchronously (no CUDA call is
made before the checks, so these run on a CPU-only host)."""
import ctypes
import json
import os
import re

import pytest

import diffusion_transformer_mlp_gb300 as fc2
from diffusion_transformer_mlp_gb300 import _lib
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    L = _lib.load()
    decl = declared_symbols()
    assert {"nvfp4_quantize_weight", "swiglu_nvfp4_quantize", "nvfp4_fc2_gemm"} <= decl
    assert decl == set(_lib.EXPORTED)
    for name in decl:
        assert hasattr(L, name), name
    assert L.nvfp4_version() >> 16 == 1


def test_library_is_in_tree():
    assert os.path.realpath(_lib.LIB_PATH).startswith(os.path.realpath(ROOT))


@pytest.mark.parametrize("rows,cols", [(1, 16), (37810, 14336), (37824, 14336), (5376, 14336),
                                       (300, 1040), (128, 48), (37810, 7168)])
def test_sizes_match_oracle(rows, cols):
    assert fc2.padded_rows(rows) == oracle.padded_rows(rows)
    assert fc2.qdata_bytes(rows, cols) == oracle.qdata_bytes(rows, cols)
    assert fc2.scale_bytes(rows, cols) == oracle.scale_bytes(rows, cols)
    for r, c in [(0, 0), (rows - 1, cols // 16 - 1), (rows // 2, cols // 32), (min(rows - 1, 129), 5 % (cols // 16))]:
        assert fc2.scale_offset(r, c, cols) == oracle.scale_offset(r, c, cols)


def test_sizes_reproduce_pages_footprint():
    fp = json.load(open(os.path.join(ROOT, "tests", "golden", "footprint.json")))
    n, k = fp["n"], fp["k"]
    assert fc2.qdata_bytes(n, k) + fc2.scale_bytes(n, k) == fp["weight_qdata_plus_scales"]
    a = fc2.qdata_bytes(fp["logical_m"], k) + fc2.scale_bytes(fp["logical_m"], k)
    assert (n // 128) * a == fp["requested_activation_bytes"]
    assert fc2.padded_rows(fp["logical_m"]) // 128 * (n // 128) == fp["ctas"]


def test_empty_and_negative_sizes():
    assert fc2.padded_rows(0) == 0 and fc2.qdata_bytes(0, 64) == 0 and fc2.scale_bytes(-3, 64) == 0


# fake, never dereferenced pointers: every check below fails before any CUDA call
P16 = ctypes.c_void_p(0x10000)
P8 = ctypes.c_void_p(0x10008)
NUL = ctypes.c_void_p(0)


def test_quantizer_argument_errors():
    L = _lib.load()
    q = L.swiglu_nvfp4_quantize
    assert q(NUL, 4, 64, 128, P16, P16, P16, NUL) == _lib.NVFP4_EINVAL          # null input
    assert q(P16, 0, 64, 128, P16, P16, P16, NUL) == _lib.NVFP4_EINVAL          # empty M
    assert q(P16, 4, 8, 16, P16, P16, P16, NUL) == _lib.NVFP4_EINVAL            # cols < 16
    assert q(P16, 4, 40, 80, P16, P16, P16, NUL) == _lib.NVFP4_EUNSUPPORTED     # cols % 16
    assert q(P16, 4, 64, 100, P16, P16, P16, NUL) == _lib.NVFP4_EINVAL          # ld < 2k
    assert q(P16, 4, 64, 132, P16, P16, P16, NUL) == _lib.NVFP4_EALIGN          # ld % 8
    assert q(P8, 4, 64, 128, P16, P16, P16, NUL) == _lib.NVFP4_EALIGN           # misaligned
    assert "ld" in _lib.last_error() or "aligned" in _lib.last_error()
    w = L.nvfp4_quantize_weight
    assert w(P16, 4, 64, 32, P16, P16, P16, NUL) == _lib.NVFP4_EINVAL           # ld < cols
    assert w(P16, 4, 64, 64, P16, P16, P8, NUL) == _lib.NVFP4_EALIGN            # rec misaligned
    # the kernels index in 32 bits: sizes they cannot address are refused
    assert w(P16, 1 << 31, 16, 16, P16, P16, P16, NUL) == _lib.NVFP4_EUNSUPPORTED     # padded rows
    assert w(P16, 1 << 24, 1 << 16, 1 << 16, P16, P16, P16, NUL) == _lib.NVFP4_EUNSUPPORTED  # 2^31 units
    assert w(P16, 4, 64, 1 << 31, P16, P16, P16, NUL) == _lib.NVFP4_EUNSUPPORTED     # row stride
    assert w(P16, 4, (1 << 30) + 16, (1 << 30) + 16, P16, P16, P16, NUL) == _lib.NVFP4_EUNSUPPORTED
    assert "too large" in _lib.last_error()
    # the binding limit at the FC2 width is the scale array: about 2.4 M rows,
    # far above the canonical 37,888
    assert fc2.scale_bytes(2_390_000, 14336) < (1 << 31) <= fc2.scale_bytes(2_400_000, 14336)


def test_gemm_argument_errors():
    L = _lib.load()
    g = L.nvfp4_fc2_gemm
    ok = [P16] * 6
    assert g(*ok, 4, 128, 256, NUL, 128, NUL, NUL) == _lib.NVFP4_EINVAL         # null out
    assert g(*ok, 0, 128, 256, P16, 128, NUL, NUL) == _lib.NVFP4_EINVAL         # m = 0
    assert g(*ok, 4, 100, 256, P16, 128, NUL, NUL) == _lib.NVFP4_EUNSUPPORTED   # n % 128
    assert g(*ok, 4, 128, 320, P16, 128, NUL, NUL) == _lib.NVFP4_EUNSUPPORTED   # k % 256
    assert g(*ok, 4, 128, 256, P16, 64, NUL, NUL) == _lib.NVFP4_EINVAL          # ldo < n
    assert g(*ok, 4, 128, 256, P16, 132, NUL, NUL) == _lib.NVFP4_EALIGN         # ldo % 8
    f1 = L.nvfp4_fc1_swiglu
    assert f1(*ok, 4, 0, 256, P16, 128, P16, NUL, NUL) == _lib.NVFP4_EINVAL        # f = 0
    assert f1(*ok, 4, 192, 256, P16, 192, P16, NUL, NUL) == _lib.NVFP4_EUNSUPPORTED  # f % 128
    assert f1(*ok, 4, 128, 256, P16, 128, NUL, NUL, NUL) == _lib.NVFP4_EINVAL      # null h_rec
    assert f1(*ok, 4, 128, 256, P16, 64, P16, NUL, NUL) == _lib.NVFP4_EINVAL       # ldh < f
    assert f1(*ok, 4, 128, 256, P16, 128, P8, NUL, NUL) == _lib.NVFP4_EALIGN       # h_rec misaligned
    assert f1(*ok, 4, 128, 320, P16, 128, P16, NUL, NUL) == _lib.NVFP4_EUNSUPPORTED  # k % 256
    qa = L.nvfp4_quantize_with_amax
    assert qa(P16, 4, 64, 32, P16, P16, P16, NUL) == _lib.NVFP4_EINVAL             # ld < cols
    assert qa(P16, 4, 40, 40, P16, P16, P16, NUL) == _lib.NVFP4_EUNSUPPORTED       # cols % 16
    assert g(P8, *ok[1:], 4, 128, 256, P16, 128, NUL, NUL) == _lib.NVFP4_EALIGN  # misaligned A


def test_diag_argument_errors():
    L = _lib.load()
    assert L.nvfp4_diag_code_transitions(2, P16, 10, P16, P16, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_wait_timeout(0, P16, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_wait_timeout(10 ** 10, P16, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_mma_peak(0, P16, NUL, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_mma_peak(64, P16, ctypes.c_void_p(0x1004), NUL) == _lib.NVFP4_EINVAL  # clk misaligned
    assert L.nvfp4_diag_quotient_codes(1, 0, P16, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_quotient_codes(0x7F80, 1, P16, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_quotient_codes(1, 0x7F80, P16, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_quotient_codes(1, 1, NUL, NUL) == _lib.NVFP4_EINVAL
    assert L.nvfp4_diag_mma_peak((1 << 22) + 1, P16, NUL, NUL) == _lib.NVFP4_EINVAL
    # the clocked GEMM wants its record buffer (checked before any CUDA call)
    g = L.nvfp4_diag_fc2_gemm_clock
    assert g(P16, P16, P16, P16, P16, P16, 256, 256, 256, P16, 256, NUL, NUL, NUL) == _lib.NVFP4_EINVAL
    assert g(P16, P16, P16, P16, P16, P16, 256, 256, 256, P16, 256, NUL, ctypes.c_void_p(0x1004), NUL) == \
        _lib.NVFP4_EINVAL


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "diffusion_transformer_mlp_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "nvfp4_oracle" not in text, f


def _host_nvfp4(rows, cols, qbytes=None, sbytes=None, rec=16):
    import torch
    q = torch.zeros(qbytes if qbytes is not None else fc2.qdata_bytes(rows, cols), dtype=torch.uint8)
    s = torch.zeros(sbytes if sbytes is not None else fc2.scale_bytes(rows, cols), dtype=torch.uint8)
    return fc2.NVFP4Tensor(q, s, torch.zeros(rec, dtype=torch.uint8), rows, cols)


def test_python_wrappers_reject_mismatched_nvfp4_buffers():
    """A caller-supplied NVFP4Tensor whose shape or byte counts do not fit the
    call is refused before anything reaches the library (a buffer kept from
    a smaller M would otherwise receive device writes past its end)."""
    import torch
    x = torch.zeros(300, 2 * 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"\[200, 64\]"):
        fc2.swiglu_nvfp4_quantize(x, out=_host_nvfp4(200, 64))
    with pytest.raises(ValueError, match="qdata has"):
        fc2.swiglu_nvfp4_quantize(x, out=_host_nvfp4(300, 64, qbytes=fc2.qdata_bytes(200, 64)))
    with pytest.raises(ValueError, match="scales has"):
        fc2.nvfp4_quantize_weight(x, out=_host_nvfp4(300, 128, sbytes=100))
    with pytest.raises(ValueError, match="rec has"):
        fc2.nvfp4_quantize_weight(x, out=_host_nvfp4(300, 128, rec=8))
    a = _host_nvfp4(300, 256)
    w_small = _host_nvfp4(128, 256, qbytes=128 * 64)
    with pytest.raises(ValueError, match="w.qdata has"):
        fc2.nvfp4_fc2_gemm(a, w_small)
    a_big = fc2.NVFP4Tensor(a.qdata, a.scales, a.rec, 400, 256)  # claims more rows than its buffers hold
    with pytest.raises(ValueError, match="a.qdata has"):
        fc2.nvfp4_fc2_gemm(a_big, _host_nvfp4(128, 256))
    with pytest.raises(ValueError, match="act holds"):
        fc2.nvfp4_fc1_swiglu(a, _host_nvfp4(256, 256), act=_host_nvfp4(200, 128))
    strided = fc2.NVFP4Tensor(torch.zeros(2 * fc2.qdata_bytes(300, 256), dtype=torch.uint8)[::2], a.scales,
                              a.rec, 300, 256)
    with pytest.raises(ValueError, match="contiguous"):
        fc2.nvfp4_fc2_gemm(strided, _host_nvfp4(128, 256))


def test_host_step_argument_errors():
    """nvfp4_fc2_host refuses bad arguments before it enqueues anything (no
    CUDA call is made, so this runs without a GPU)."""
    L = _lib.load()
    p = ctypes.c_void_p(16)
    args = lambda **kw: [kw.get("gu", p), kw.get("m", 256), kw.get("k", 1024), kw.get("ld", 2048), p, p, p,
                         kw.get("n", 512), kw.get("x", p), p, p, p, p, p, None, None]
    assert L.nvfp4_fc2_host(*args(gu=None)) == _lib.NVFP4_EINVAL
    assert L.nvfp4_fc2_host(*args(x=None)) == _lib.NVFP4_EINVAL
    assert L.nvfp4_fc2_host(*args(m=0)) == _lib.NVFP4_EINVAL
    assert L.nvfp4_fc2_host(*args(ld=2000)) == _lib.NVFP4_EINVAL
    assert L.nvfp4_fc2_host(*args(k=1040, ld=2080)) == _lib.NVFP4_EUNSUPPORTED
    assert L.nvfp4_fc2_host(*args(n=200)) == _lib.NVFP4_EUNSUPPORTED
    assert L.nvfp4_fc2_host(*args(x=ctypes.c_void_p(24))) == _lib.NVFP4_EALIGN
    assert "nvfp4_fc2_host" in _lib.last_error()
