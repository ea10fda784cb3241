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


def _set_code(p, r, c, code):
    p = p.copy()
    if c % 2 == 0:
        p[r, c // 2] = (p[r, c // 2] & 0xF0) | code
    else:
        p[r, c // 2] = (p[r, c // 2] & 0x0F) | (code << 4)
    return p


def _one_block(v1):
    """One 16-block with SF = 448 and r = 1 (gs = 448, amax 6), so the second
    element's scaled value is exactly v1."""
    h = np.zeros((1, 16), dtype=np.float32)
    h[0, 0] = 6.0
    h[0, 1] = v1
    gs = np.float32(448.0)
    p, s = oracle.quantize_nvfp4(h, gs)
    return h, gs, p, s


def test_two_step_flip_at_a_boundary_fails():
    h, gs, p, s = _one_block(1.25 * (1 + 5e-4))      # oracle: 1.5 (code 3)
    with pytest.raises(AssertionError):
        check_requant(_set_code(p, 0, 1, 1), s, h, gs, max_frac=1.0)   # 0.5: two steps down


def test_flip_one_percent_from_a_boundary_fails():
    h, gs, p, s = _one_block(5.0 * 1.01)              # oracle: 6 (code 7); 1 % above the 5 boundary
    with pytest.raises(AssertionError):
        check_requant(_set_code(p, 0, 1, 6), s, h, gs, max_frac=1.0)   # 4: one step, but not near


def test_wrong_sign_next_to_zero_fails():
    h, gs, p, s = _one_block(0.25 * (1 - 5e-4))       # oracle: +0 (code 0), next to the 0.25 boundary
    assert check_requant(_set_code(p, 0, 1, 1), s, h, gs, max_frac=1.0) == (1, 0)   # +0.5 is fine
    with pytest.raises(AssertionError):
        check_requant(_set_code(p, 0, 1, 9), s, h, gs, max_frac=1.0)   # -0.5 has the wrong sign


def test_sign_flip_of_a_nonzero_code_fails():
    h, gs, p, s = _one_block(3.0)                     # oracle: 3 (code 5)
    with pytest.raises(AssertionError):
        check_requant(_set_code(p, 0, 1, 13), s, h, gs, max_frac=1.0)  # -3


def test_too_many_boundary_flips_fail():
    """Every flip below is a legal one-step flip at a boundary, but 2 of 16
    elements (12.5 %) is above the 0.5 % allowance."""
    h = np.zeros((1, 16), dtype=np.float32)
    h[0, 0] = 6.0
    h[0, 1] = h[0, 2] = 1.25 * (1 + 5e-4)
    gs = np.float32(448.0)
    p, s = oracle.quantize_nvfp4(h, gs)
    p2 = _set_code(_set_code(p, 0, 1, 2), 0, 2, 2)
    assert check_requant(p2, s, h, gs, max_frac=1.0) == (2, 0)
    with pytest.raises(AssertionError):
        check_requant(p2, s, h, gs)


def test_scale_two_steps_off_at_a_midpoint_fails():
    """amax 6.375 with gs 1: s = 1.0625, exactly the midpoint of E4M3 1.0
    (0x38) and 1.125 (0x39); the oracle ties to 0x38 and codes 6.375 as 6.
    A GPU scale of 0x39 is one step at a midpoint: accepted, and with it the
    value 6.375 / 1.125 = 5.67 still codes as 6.  0x3a is two steps: rejected."""
    h = np.zeros((1, 16), dtype=np.float32)
    h[0, 0] = 6.375
    gs = np.float32(1.0)
    p, s = oracle.quantize_nvfp4(h, gs)
    assert s[0, 0] == 0x38 and (p[0, 0] & 0x0F) == 7
    s1, s2 = s.copy(), s.copy()
    s1[0, 0], s2[0, 0] = 0x39, 0x3A
    assert check_requant(p, s1, h, gs, max_frac=1.0) == (0, 1)
    with pytest.raises(AssertionError):
        check_requant(p, s2, h, gs, max_frac=1.0)


def test_gemm_tolerance_bound_is_tight():
    g = np.random.default_rng(4)
    ref = oracle.bf16_round(g.standard_normal((16, 64)))
    assert_gemm_close(ref * (1 + 9e-4), ref)
    with pytest.raises(AssertionError):
        assert_gemm_close(ref * (1 + 2e-3), ref)
    bad = ref.copy()
    bad[0, 0] = np.nan
    with pytest.raises(AssertionError):
        assert_gemm_close(bad, ref)
