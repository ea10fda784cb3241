"""The acceptance checker must reject plausible mistakes (planted in oracle
outputs on the CPU) and accept boundary-only differences."""
import numpy as np
import pytest

import oracle
from tolerance import assert_gemm_close, check_requant


def _h(seed=0):
    g = np.random.default_rng(seed)
    return (g.standard_normal((8, 256)) * 0.3).astype(np.float32)


def test_identical_passes():
    h = _h()
    gs = oracle.global_scale(np.abs(h).max())
    p, s = oracle.quantize_nvfp4(h, gs)
    assert check_requant(p, s, h, gs) == (0, 0)


def test_flipped_code_away_from_boundary_fails():
    h = _h()
    gs = oracle.global_scale(np.abs(h).max())
    p, s, d = oracle.quantize_nvfp4(h, gs, detail=True)
    # find an element far from any boundary and bump its code by one step
    v = np.abs(d["v"])
    far = np.where((np.abs(v - 1.0) < 0.05))
    r, c = far[0][0], far[1][0]
    p = p.copy()
    if c % 2 == 0:
        p[r, c // 2] = (p[r, c // 2] & 0xF0) | ((p[r, c // 2] & 0x0F) + 1)
    else:
        p[r, c // 2] = (p[r, c // 2] & 0x0F) | (((p[r, c // 2] >> 4) + 1) << 4)
    with pytest.raises(AssertionError):
        check_requant(p, s, h, gs)


def test_swapped_nibbles_fail():
    h = _h(1)
    gs = oracle.global_scale(np.abs(h).max())
    p, s = oracle.quantize_nvfp4(h, gs)
    swapped = ((p >> 4) | (p << 4)).astype(np.uint8)
    with pytest.raises(AssertionError):
        check_requant(swapped, s, h, gs)


def test_wrong_scale_fails():
    h = _h(2)
    gs = oracle.global_scale(np.abs(h).max())
    p, s = oracle.quantize_nvfp4(h, gs)
    s = s.copy()
    s[0, 0] += 1
    with pytest.raises(AssertionError):
        check_requant(p, s, h, gs)


def test_boundary_flip_accepted():
    h = np.full((1, 16), 0.0, dtype=np.float32)
    h[0, 0] = 6.0
    h[0, 1] = 1.25 * (1 + 5e-4)          # v just above the 1.25 boundary -> 1.5 (code 3)
    gs = np.float32(448.0)               # s = 448 -> SF = 448, r = 1
    p, s = oracle.quantize_nvfp4(h, gs)
    assert (p[0, 0] >> 4) == 3
    p2 = p.copy()
    p2[0, 0] = (p2[0, 0] & 0x0F) | (2 << 4)   # the neighbour below: 1.0
    assert check_requant(p2, s, h, gs, max_frac=1.0) == (1, 0)


def test_gemm_tolerance():
    g = np.random.default_rng(3)
    ref = oracle.bf16_round(g.standard_normal((16, 64)))
    assert_gemm_close(ref * (1 + 5e-4), ref)
    with pytest.raises(AssertionError):
        assert_gemm_close(ref.T.copy().reshape(16, 64), ref)   # transposed operand
    with pytest.raises(AssertionError):
        assert_gemm_close(ref * 1.01, ref)
