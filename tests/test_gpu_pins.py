"""Pins of the oracle's NVFP4 byte conventions against consumers that are
not part of this repository, on the GPU.

- Nibble order ("even element in the low nibble"): the tensor core reads the
  oracle's QDATA in a kind::f8f6f4 MMA against an E4M3 identity, which
  gives every element by its index (an E2M1 x E2M1 GEMM cannot: the same
  swap inside every byte of both operands leaves each dot product as it
  was).  The values it reads must be the oracle's inputs.
- Scale layout (the general 128-row by 4-scale-column tiled offset,
  "GB10 component-2 nsys summary", native_pack_validation): cuBLASLt's
  block-scaled NVFP4 matmul (vector-16 UE4M3 scales in its own documented
  tiled layout) reads the oracle's QDATA and scale bytes; its product times
  gA gW must match the oracle's FP64 GEMM within the GEMM tolerance, at the
  feature widths 5376, 7168 and 14336 the pages name.
- The block-scale encoder of the producer against E4M3(RN(bmax / d)) over
  every BF16 global max and block max.
"""
import numpy as np
import pytest
import torch

import diffusion_transformer_mlp_gb300 as fc2
import oracle
import synth

pytestmark = pytest.mark.gpu

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def f32_to_bf16_exact(v: np.ndarray) -> np.ndarray:
    """BF16 bits of float32 values that are BF16 values already."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exact in BF16"
    return (b >> 16).astype(np.uint16)


def test_tensor_core_reads_oracle_nibbles():
    """Rows 0..127 hold E2M1 grid values of both signs (-0 included), each
    16-element block with a +-6 so that its scale is 1; row 128 holds 2688
    so that the global scale is 1.  The oracle's QDATA bytes of rows 0..127,
    read by the tensor core, give back the inputs element by element."""
    rng = np.random.default_rng(2024)
    x = rng.choice(E2M1_GRID, size=(129, 32)) * rng.choice([-1.0, 1.0], size=(129, 32))
    for r in range(128):
        for b in range(2):
            x[r, 16 * b + rng.integers(16)] = rng.choice([-6.0, 6.0])
    x[128] = 0.0
    x[128, 5] = 2688.0
    q, s, rec = oracle.quantize(f32_to_bf16_exact(x), 32, swiglu=False)
    assert rec["global_scale"] == np.float32(1.0)
    assert np.all(s[[oracle.scale_offset(r, b, 32) for r in range(128) for b in range(2)]] == 0x38)
    qd = torch.from_numpy(np.ascontiguousarray(q[:128])).cuda()
    out = torch.empty(128, 32, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = fc2._lib.load()
    fc2._lib.check(L.nvfp4_diag_tc_e2m1_read(fc2._ptr(qd), fc2._ptr(out), fc2._ptr(status), fc2._stream(None)),
                   "nvfp4_diag_tc_e2m1_read")
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != x[:128])
    assert bad.size == 0, f"{len(bad)} elements differ; first {tuple(bad[0])}: {got[tuple(bad[0])]} vs " \
                          f"{x[:128][tuple(bad[0])]}"
    # the same bytes with the two nibbles of every byte swapped read differently,
    # so the comparison above does depend on the order
    swapped = ((q[:128] >> 4) | (q[:128] << 4)).astype(np.uint8)
    assert not np.array_equal(swapped, q[:128])


def blocky_input(rows: int, cols: int, seed: int) -> np.ndarray:
    """BF16 [rows, cols]: the activation law with each 16-element block
    multiplied by its own power of two 2^e, e uniform in -8..8, so the block
    scales of neighbouring rows and columns differ by large factors."""
    x = synth.bf16_to_f32(synth.quant_input(rows, cols, seed=seed))
    e = np.random.default_rng(seed).integers(-8, 9, size=(rows, cols // 16))
    return f32_to_bf16_exact(x * np.repeat(np.exp2(e), 16, axis=1).astype(np.float32))


@pytest.mark.parametrize("m,n,k", [(256, 256, 1024), (200, 384, 5376), (130, 128, 7168), (129, 256, 14336)])
def test_library_nvfp4_matmul_reads_oracle_bytes(m, n, k):
    import _cublaslt
    x = blocky_input(m, k, seed=m + k)
    w = blocky_input(n, k, seed=n + k + 1)
    aq, as_, ar = oracle.quantize(x, k, swiglu=False)
    wq, ws, wr = oracle.quantize(w, k, swiglu=False)
    # the scale codes really vary: a misplaced scale byte changes the product
    assert len(np.unique(as_)) > 40 and len(np.unique(ws)) > 40
    dev = [torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in (aq, as_, wq, ws)]
    lib = _cublaslt.nvfp4_matmul(dev[0], dev[1], dev[2], dev[3], m, n, k).cpu().numpy().astype(np.float64)
    ref = oracle.gemm_rows(aq, as_, ar["global_scale"], wq, ws, wr["global_scale"], n, k, np.arange(m))
    got = lib * float(ar["global_scale"]) * float(wr["global_scale"])
    ok, worst = oracle.check_gemm_tolerance(got, ref)
    assert ok, f"cuBLASLt on the oracle's bytes: worst error / bound = {worst}"


def test_block_scale_code_exhaustive():
    """Every BF16 global max x every finite BF16 block max: the producer's
    block-scale code equals E4M3(RN(bmax / RN(6 RN(A / 2688))))."""
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    L = fc2._lib.load()
    fc2._lib.check(L.nvfp4_diag_block_scale_codes(0, 0x7F80, fc2._ptr(counts), fc2._stream(None)),
                   "nvfp4_diag_block_scale_codes")
    torch.cuda.synchronize()
    bad, seen = counts.tolist()
    assert seen == 0x7F80 * 0x7F80
    assert bad == 0
