"""Data layouts: the 128x4 swizzled block-scale layout and the gate/up
interleave of the fused gate_up weight.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Swizzled scales ("the dense swizzled layout fp4_gemm expects"): [P1]
"关键源码片段", qwen2_moe.py excerpt, re-lays a 6-D scale tensor of shape
(32, 4, m_blocks, 4, K/64, 1) with ``permute(2, 4, 0, 1, 3, 5)`` and
``reshape(m_padded, -1)``, m_padded = 128 * m_blocks.  Reading (the pages do
not say which 4-wide dim is which): dim 0 = row % 32, dim 1 = (row % 128) // 32,
dim 2 = row // 128, dim 3 = scale column % 4, dim 4 = scale column // 4.
Rows pad to a multiple of 128 and scale columns to a multiple of 4, with zero
bytes.  ``sf_swizzle_128x4`` builds exactly that 6-D tensor and applies the
pages' permute.  Pinned by tests/test_oracle_layouts.py against the explicit
byte-offset formula derived independently, by bijectivity, and on the GPU by
every GEMM's parity (a wrong reading fails them all).

Gate/up interleave: [P2] "关键源码片段", modelopt_quant.py excerpt: the
gate_up weight is [gate; up] (``gate_w, up_w = w.chunk(2, dim=0)``); the fused
kernel's weight is ``interleave_linear_and_gate(cat(up, gate), group_size=64)``
and its scales get the same interleave on the *un-swizzled* scales, then the
2-D swizzle.  Reading of ``interleave_linear_and_gate``: output rows are
blocks of 128 = [64 rows of the first half; the same 64 row indices of the
second half], i.e. block b = [up rows 64b..64b+63; gate rows 64b..64b+63].
Pinned by tests/test_oracle_layouts.py (brute-force row map, inverse).
"""
import numpy as np


def _ceil(a, b):
    return (a + b - 1) // b * b


def sf_swizzled_bytes(rows, sf_cols):
    return _ceil(rows, 128) * _ceil(sf_cols, 4)


def sf_swizzle_128x4(sf_lin):
    """Linear scales uint8 [rows, C] -> flat uint8 in the swizzled layout,
    size ceil128(rows) * ceil4(C)."""
    sf_lin = np.asarray(sf_lin)
    rows, c = sf_lin.shape
    rp, cp = _ceil(rows, 128), _ceil(c, 4)
    pad = np.zeros((rp, cp), dtype=sf_lin.dtype)
    pad[:rows, :c] = sf_lin
    mb, kb = rp // 128, cp // 4
    # pad[(mb*4 + r4)*32 + r32, kb*4 + c4]  ->  six[r32, r4, mb, c4, kb, 0]
    six = pad.reshape(mb, 4, 32, kb, 4).transpose(2, 1, 0, 4, 3)[..., None]
    dense = six.transpose(2, 4, 0, 1, 3, 5).reshape(rp, -1)   # the pages' permute
    return np.ascontiguousarray(dense).reshape(-1)


def sf_unswizzle_128x4(flat, rows, c):
    """Inverse of sf_swizzle_128x4: flat swizzled bytes -> uint8 [rows, C]."""
    rp, cp = _ceil(rows, 128), _ceil(c, 4)
    flat = np.asarray(flat).reshape(-1)
    if flat.size != rp * cp:
        raise ValueError("swizzled scale buffer has the wrong size")
    dense = flat.reshape(rp // 128, cp // 4, 32, 4, 4)       # (mb, kb, r32, r4, c4)
    pad = dense.transpose(0, 3, 2, 1, 4).reshape(rp, cp)      # (mb, r4, r32, kb, c4)
    return np.ascontiguousarray(pad[:rows, :c])


def interleave_gate_up(w, group=64):
    """Rows [gate; up] (2I rows) -> the fused kernel's row order: blocks of
    2*group rows = [up 64b..64b+63 ; gate 64b..64b+63]."""
    w = np.asarray(w)
    n = w.shape[0]
    if n % (2 * group):
        raise ValueError("gate_up rows must be a multiple of 128")
    i = n // 2
    gate, up = w[:i], w[i:]
    cat = np.concatenate([up, gate], axis=0)
    halves = cat.reshape(2, i // group, group, *w.shape[1:])
    return np.ascontiguousarray(np.swapaxes(halves, 0, 1)).reshape(w.shape)


def interleave_gate_up_scales_then_swizzle(sf_lin, group=64):
    """Linear scales of [gate; up] -> interleaved, then swizzled (flat)."""
    return sf_swizzle_128x4(interleave_gate_up(sf_lin, group))
