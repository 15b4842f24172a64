"""The GEMM's grouped tile order (csrc/gemm.cu, tile_coords and the group
size chosen in gemm_launch), restated: every (M panel, N tile) is visited
exactly once for the block's shapes and for a sweep of small ones, including
groups that do not divide the N tiles; within a group the walk is
M-panel-major; and the group size follows the 48 MB / 16 MB rule."""
import itertools

import pytest

PAIR_N = 256


def group_n(num_n_tiles: int, k: int) -> int:
    tile_bytes = PAIR_N * (k // 2 + k // 16)
    g = num_n_tiles if tile_bytes * num_n_tiles <= (48 << 20) else (16 << 20) // tile_bytes
    return max(1, min(num_n_tiles, g))


def tile_coords(t: int, num_m: int, num_n: int, gn: int) -> tuple[int, int]:
    span = gn * num_m
    g = t // span
    g0 = g * gn
    gs = min(gn, num_n - g0)
    r = t - g * span
    mt = r // gs
    return mt, g0 + (r - mt * gs)


def check_order(num_m: int, num_n: int, gn: int) -> None:
    seen = [tile_coords(t, num_m, num_n, gn) for t in range(num_m * num_n)]
    assert sorted(seen) == [(m, n) for m in range(num_m) for n in range(num_n)]
    # inside each group: M-panel-major, N tiles of the group in increasing order
    for g0 in range(0, num_n, gn):
        gs = min(gn, num_n - g0)
        base = g0 * num_m
        block = seen[base:base + gs * num_m]
        assert block == [(m, g0 + j) for m in range(num_m) for j in range(gs)]


@pytest.mark.parametrize("name,m,n,k,expect_group", [
    ("fc2", 37810, 5376, 14336, 21),
    ("fc1", 37810, 28672, 5376, 21),
    ("qkv", 37810, 21504, 5376, 21),
    ("attention_output", 37810, 5376, 5376, 21),
])
def test_block_shapes(name, m, n, k, expect_group):
    m_pad = (m + 127) // 128 * 128
    num_m, num_n = (m_pad + 255) // 256, (n + 255) // 256
    gn = group_n(num_n, k)
    assert gn == expect_group, name
    check_order(num_m, num_n, gn)


def test_small_sweep():
    for num_m, num_n, gn in itertools.product(range(1, 7), range(1, 12), range(1, 13)):
        check_order(num_m, num_n, min(gn, num_n))


def test_group_rule():
    # a weight that fits 48 MB is one group; a larger one goes in 16 MB groups
    assert group_n(21, 14336) == 21                      # 43 MB
    assert group_n(112, 5376) == (16 << 20) // (256 * (2688 + 336))
    assert group_n(1000, 1 << 20) == 1                   # a tile above 16 MB still makes progress
