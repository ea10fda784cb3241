"""Pins of the swizzled block-scale layout and the gate/up interleave."""
import numpy as np
import pytest

import oracle


def _offset(r, j, cp):
    """Byte offset of scale (row r, column j): derived from the 128x4 tile
    picture (tiles row-major over (row block, column block); inside a 512-byte
    tile, 32 lines of 16 bytes = 4 row groups x 4 columns)."""
    return ((((r // 128) * (cp // 4) + j // 4) * 32 + r % 32) * 4 + (r % 128) // 32) * 4 + j % 4


@pytest.mark.parametrize("rows,cols", [(1, 4), (128, 4), (130, 6), (256, 16), (300, 37), (4, 448)])
def test_swizzle_matches_offset_formula(rows, cols):
    g = np.random.default_rng(rows * 1000 + cols)
    sf = g.integers(1, 256, (rows, cols), dtype=np.uint8)
    flat = oracle.sf_swizzle_128x4(sf)
    rp, cp = -(-rows // 128) * 128, -(-cols // 4) * 4
    assert flat.size == rp * cp == oracle.sf_swizzled_bytes(rows, cols)
    ref = np.zeros(rp * cp, dtype=np.uint8)
    for r in range(rows):
        for j in range(cols):
            ref[_offset(r, j, cp)] = sf[r, j]
    assert np.array_equal(flat, ref)


@pytest.mark.parametrize("rows,cols", [(130, 6), (384, 12)])
def test_swizzle_is_a_bijection_with_zero_padding(rows, cols):
    ids = np.arange(1, rows * cols + 1, dtype=np.int64).reshape(rows, cols)
    flat = oracle.sf_swizzle_128x4(ids)
    nz = flat[flat != 0]
    assert np.array_equal(np.sort(nz), np.arange(1, rows * cols + 1))
    assert np.array_equal(oracle.sf_unswizzle_128x4(flat, rows, cols), ids)


def test_interleave_row_map_brute_force():
    inter = 192
    w = np.arange(2 * inter)[:, None] * np.ones((1, 3), dtype=np.int64)  # row id in every column
    out = oracle.interleave_gate_up(w)
    for o in range(2 * inter):
        b, j = divmod(o, 128)
        src = inter + 64 * b + j if j < 64 else 64 * b + j - 64   # up rows first, then gate
        assert out[o, 0] == src and out[o, 2] == src


def test_interleave_rejects_ragged():
    with pytest.raises(ValueError):
        oracle.interleave_gate_up(np.zeros((192, 2)))


def test_interleaved_scales_equal_interleave_then_swizzle():
    g = np.random.default_rng(9)
    sf = g.integers(0, 127, (256, 8), dtype=np.uint8)
    a = oracle.interleave_gate_up_scales_then_swizzle(sf)
    back = oracle.sf_unswizzle_128x4(a, 256, 8)
    assert np.array_equal(back, oracle.interleave_gate_up(sf))
