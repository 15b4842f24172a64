"""Inputs that drive the NVFP4 recipe through its edge cases.

With one element equal to 2688 the global scale is g = 2688 / 2688 = 1 and
d = 6 g = 6, so a 16-element block whose largest magnitude is B gets the
block ratio B / 6.  The blocks of edge_matrix() take, in turn:
- B = 6 E4M3(c) for every UE4M3 code c = 0x00 .. 0x7E (c = 0 is an
  all-zero block, 0x01 .. 0x07 the subnormal scales);
- B = 3 (E4M3(c) + E4M3(c + 1)): a ratio exactly half-way between two
  codes (ties to the even code);
- ratios 2^-11, 2^-10 (half-way to the smallest subnormal: rounds to 0) and
  1.5 2^-10 (rounds up to it);
- an all -0 block, and a block of one 6 and fifteen negatives that round to
  E2M1 zero or its neighbour (-0.1, -0.25, -0.26).
Inside a block, the other elements are the E2M1 rounding midpoints times the
block's decoded scale (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 times E4M3(c),
random signs) and uniform values below B.  A block never exceeds the
global max, so a saturating ratio cannot be formed this way: the exhaustive
encoder sweep covers it.  These are inputs only: the expected bytes come
from the oracle.
"""
from __future__ import annotations

import numpy as np

E4M3 = np.array([(m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
                 for e in range(16) for m in range(8)][:127])
MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _bf16_toward_zero(v: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    return (b >> 16).astype(np.uint16)


def _exact_bf16(v: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exact in BF16"
    return (b >> 16).astype(np.uint16)


def targets() -> list:
    t = [("code", c) for c in range(127)]
    t += [("mid", c) for c in range(126)]
    t += [("ratio", 2.0 ** -11), ("ratio", 2.0 ** -10), ("ratio", 1.5 * 2.0 ** -10), ("negzero", 0), ("signs", 0)]
    return t


def _block(kind, arg, rng) -> np.ndarray:
    if kind == "negzero":
        return np.full(16, 0x8000, dtype=np.uint16)
    if kind == "signs":
        v = np.array([6.0] + [-0.1] * 5 + [-0.25] * 5 + [-0.26] * 5, dtype=np.float32)
        return _bf16_toward_zero(v)
    if kind == "code":
        scale, bmax = E4M3[arg], 6.0 * E4M3[arg]
    elif kind == "mid":
        scale, bmax = E4M3[arg], 3.0 * (E4M3[arg] + E4M3[arg + 1])
    else:
        scale, bmax = arg, 6.0 * arg
    if bmax == 0.0:
        return np.zeros(16, dtype=np.uint16)
    vals = np.empty(16)
    vals[0] = bmax
    vals[1:8] = MIDPOINTS * scale
    vals[8:] = rng.uniform(0.0, bmax, size=8)
    vals *= rng.choice([-1.0, 1.0], size=16)
    rng.shuffle(vals)
    # the block max and the midpoint multiples are BF16 values (at most 7
    # significant bits); truncation only moves the uniform ones, toward zero
    return _bf16_toward_zero(vals.astype(np.float32))


def edge_matrix(rows: int, cols: int, seed: int = 0) -> np.ndarray:
    """BF16 bits [rows, cols] (cols % 16 == 0); element (0, 0) is 2688."""
    assert cols % 16 == 0
    rng = np.random.default_rng(seed)
    t = targets()
    x = np.empty((rows, cols), dtype=np.uint16)
    nb = cols // 16
    for i in range(rows * nb):
        r, b = divmod(i, nb)
        kind, arg = t[i % len(t)]
        x[r, 16 * b:16 * b + 16] = _block(kind, arg, rng)
    x[0, 0] = _exact_bf16(np.array([2688.0]))[0]
    return x


def swiglu_input(h: np.ndarray) -> np.ndarray:
    """gate|up BF16 [rows, 2 cols] whose SwiGLU is h: gate = 8 (silu rounds
    to 8 in BF16) and up = h / 8 (exact: a power of two)."""
    hf = (h.astype(np.uint32) << 16).view(np.float32)
    up = _exact_bf16(hf / np.float32(8.0))
    gate = np.full_like(h, _exact_bf16(np.array([8.0]))[0])
    return np.ascontiguousarray(np.concatenate([gate, up], axis=1))


E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def grid_matrix(rows: int, cols: int, seed: int, big_col: int) -> np.ndarray:
    """BF16 bits [rows, cols] of E2M1 grid values (random signs, -0 among
    them), each 16-element block holding a +-6, and 2688 at (0, big_col).
    Quantised, the global scale is 1 and every block scale 1 except that of
    the block holding 2688 (448, its other elements encode as zero): the
    dequantised values are the inputs, multiples of 1/2 up to 6 (and 2688).
    With big_col = 0 for one GEMM operand and 16 for the other, every product
    of a dot product over K <= 2^14 is a multiple of 1/4 of magnitude
    <= 6 * 2688 and every partial sum stays below 2^22, so the FP32
    accumulation is exact in any order."""
    rng = np.random.default_rng(seed)
    x = rng.choice(E2M1_GRID, size=(rows, cols)) * rng.choice([-1.0, 1.0], size=(rows, cols))
    nb = cols // 16
    pos = rng.integers(0, 16, size=(rows, nb))
    x.reshape(rows, nb, 16)[np.arange(rows)[:, None], np.arange(nb)[None, :], pos] = \
        rng.choice([-6.0, 6.0], size=(rows, nb))
    x[0, big_col] = 2688.0
    return _exact_bf16(x.astype(np.float32))
