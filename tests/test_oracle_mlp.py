"""Pins of the oracle's contractions, SwiGLU and requantize."""
import itertools
import math

import ml_dtypes
import numpy as np
import pytest

import oracle
import synth


def _lib_decode(packed, sf):
    """Independent decode: ml_dtypes for E2M1 codes and E4M3 scales."""
    codes = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2], codes[:, 1::2] = packed & 0xF, packed >> 4
    vals = codes.view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    sc = sf.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    return vals * np.repeat(sc, 16, axis=1)


def _rand_nvfp4(rows, k, seed):
    g = np.random.default_rng(seed)
    packed = g.integers(0, 256, (rows, k // 2), dtype=np.uint8)
    sf = g.integers(0x20, 0x48, (rows, k // 16), dtype=np.uint8)
    return packed, sf


@pytest.mark.parametrize("m,n,k", [(1, 1, 16), (3, 5, 32), (4, 8, 64), (2, 7, 48)])
def test_w4a4_gemm_brute_force(m, n, k):
    a, sa = _rand_nvfp4(m, k, 1)
    b, sb = _rand_nvfp4(n, k, 2)
    alpha = np.float32(0.37)
    d = oracle.gemm_w4a4(a, sa, b, sb, alpha, round_bf16=False)
    av, bv = _lib_decode(a, sa), _lib_decode(b, sb)
    for i, j in itertools.product(range(m), range(n)):
        acc = 0.0
        for kk in range(k):
            acc += av[i, kk] * bv[j, kk]
        assert d[i, j] == pytest.approx(float(alpha) * acc, rel=1e-12, abs=1e-12)


def test_w4a4_gemm_exact_integers():
    # SF = 1.0 (0x38) and codes whose values are integers: the GEMM is an exact integer matmul
    g = np.random.default_rng(3)
    m, n, k = 6, 10, 128
    ia = g.choice([0, 2, 4, 5, 6, 7, 10, 12, 13, 14, 15], (m, k)).astype(np.uint8)  # |v| in {0,1,2,3,4,6}
    ib = g.choice([0, 2, 4, 5, 6, 7, 10, 12, 13, 14, 15], (n, k)).astype(np.uint8)
    pk = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    one = np.full((m, k // 16), 0x38, np.uint8), np.full((n, k // 16), 0x38, np.uint8)
    d = oracle.gemm_w4a4(pk(ia), one[0], pk(ib), one[1], np.float32(1.0), round_bf16=False)
    lut = np.array([0, 0, 1, 0, 2, 3, 4, 6, 0, 0, -1, 0, -2, -3, -4, -6], dtype=np.int64)
    exact = lut[ia] @ lut[ib].T
    assert np.array_equal(d, exact.astype(np.float64))


def test_w4a16_gemm_brute_force_and_alpha():
    g = np.random.default_rng(4)
    x = synth.to_bf16_bits(g.standard_normal((3, 32)).astype(np.float32))[1]
    b, sb = _rand_nvfp4(5, 32, 5)
    d = oracle.gemm_w4a16(x, b, sb, np.float32(0.5), round_bf16=False)
    bv = _lib_decode(b, sb)
    for i in range(3):
        for j in range(5):
            assert d[i, j] == pytest.approx(0.5 * sum(float(x[i, t]) * bv[j, t] for t in range(32)), rel=1e-12)


def test_w4a16_equals_w4a4_on_representable_x():
    # every block holds a +-6 code and a power-of-two scale, so quantize(x, gs=1) recovers x exactly
    g = np.random.default_rng(11)
    m, k = 4, 128
    codes = g.integers(0, 16, (m, k), dtype=np.uint8)
    codes[:, ::16] = 7
    sf = g.choice([0x30, 0x38, 0x40, 0x48], (m, k // 16)).astype(np.uint8)  # 0.5, 1, 2, 4
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    x = oracle.dequantize_nvfp4(packed, sf).astype(np.float32)
    qp, qs = oracle.quantize_nvfp4(x, np.float32(1.0))
    assert np.array_equal(qs, sf)
    assert np.array_equal(oracle.e2m1_decode(oracle.unpack_codes(qp)), oracle.e2m1_decode(codes))
    b, sb = _rand_nvfp4(9, k, 12)
    d16 = oracle.gemm_w4a16(x, b, sb, np.float32(0.25), round_bf16=False)
    d44 = oracle.gemm_w4a4(qp, qs, b, sb, np.float32(0.25), round_bf16=False)
    assert np.array_equal(d16, d44)


def test_silu_closed_forms():
    x = np.linspace(-30, 30, 1201)
    s = oracle.silu(x)
    assert oracle.silu(0.0) == 0.0
    assert np.allclose(s - oracle.silu(-x), x, rtol=0, atol=1e-12)       # silu(x) - silu(-x) = x
    sig = s / np.where(x == 0, 1, x)
    assert np.allclose((sig + oracle.silu(-x) / np.where(x == 0, 1, -x))[x != 0], 1.0, atol=1e-12)
    assert oracle.silu(-800.0) == 0.0 and oracle.silu(800.0) == 800.0
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


def test_swiglu_uses_gate_first_half():
    gu = np.array([[1.0, -2.0, 3.0, 0.5]])
    h = oracle.swiglu_h(gu)
    assert h[0, 0] == np.float32(oracle.silu(1.0) * 3.0)
    assert h[0, 1] == np.float32(oracle.silu(-2.0) * 0.5)


def test_silu_mul_bf16_single_rounding():
    gu = np.array([[2.0, 1.0 + 2.0 ** -7]])
    want = oracle.bf16_round(oracle.silu(2.0) * (1.0 + 2.0 ** -7))
    assert oracle.silu_mul_bf16(gu)[0, 0] == want


def test_fused_and_unfused_requant_agree_within_tolerance():
    """The fused path (h from the unrounded GEMM) and the unfused one (h from
    the bf16-rounded gate_up) give the same NVFP4 codes except near rounding
    boundaries -- the agreement the pages report for their fused kernel."""
    from tolerance import check_requant
    w = synth.WORKLOADS[0]
    _, x = synth.activations(0, 4)
    gs_x = oracle.global_scale(np.abs(x).max())
    wgu = synth.weight(0, "gate_up")
    gs_w = oracle.global_scale(np.abs(wgu).max())
    wq, ws = oracle.quantize_nvfp4(wgu, gs_w)
    xq, xs = oracle.quantize_nvfp4(x, gs_x)
    alpha = np.float32(1.0) / (gs_x * gs_w)
    d = oracle.gemm_w4a4(xq, xs, wq, ws, alpha, round_bf16=False)
    h = oracle.swiglu_h(d)
    gs_h = oracle.global_scale(np.abs(h).max())
    uq, us = oracle.silu_mul_quant(oracle.bf16_round(d), gs_h)
    # bf16 rounding of gate_up moves h by up to ~2^-8 relative: widen the window accordingly
    check_requant(uq, us, h, gs_h, max_frac=0.05, what="fused vs unfused", window=2.0 ** -7)
    assert h.shape == (4, w.inter)


def test_masked_groups_reduce_to_dense_calls():
    """Each group of the masked form is the dense SiLU*mul quantize of its
    valid rows; a group with masked_m = 0 produces nothing."""
    g = np.random.default_rng(21)
    gu = (g.standard_normal((3, 10, 64)) * 1.5).astype(np.float32)
    out = oracle.silu_mul_quant_masked(gu, [10, 4, 0], np.float32(20.0))
    for e, valid in enumerate([10, 4, 0]):
        ref = oracle.silu_mul_quant(gu[e, :valid], np.float32(20.0))
        assert np.array_equal(out[e][0], ref[0]) and np.array_equal(out[e][1], ref[1])
    assert out[2][0].shape == (0, 16)


def test_per_token_gemm_is_row_scaled_gemm():
    a, sa = _rand_nvfp4(4, 64, 41)
    b, sb = _rand_nvfp4(6, 64, 42)
    rs = np.array([0.5, 2.0, 1.0, 0.125], dtype=np.float32)
    d = oracle.gemm_w4a4_per_token(a, sa, rs, b, sb, np.float32(0.25), round_bf16=False)
    base = oracle.gemm_w4a4(a, sa, b, sb, np.float32(0.25), round_bf16=False)
    assert np.array_equal(d, base * rs[:, None].astype(np.float64))


def test_awq_prescale_hand_worked_roundings():
    # bf16 keeps 7 fraction bits; each product below was worked by hand
    cases = [
        (1.0078125, 1.5, 1.515625),         # 1.51171875 lies halfway: ties to the even 1.515625
        (1.0078125, 1.0078125, 1.015625),   # 1 + 2^-6 + 2^-14: the 2^-14 is below half an ulp
        (-3.0, 0.5, -1.5),
        (0.0, -2.0, -0.0),
        (1.5 * 2.0 ** 127, 2.0, math.inf),  # past the largest bf16: overflows
        (2.0 ** -130, 0.5, 2.0 ** -131),    # subnormal, exact
    ]
    for x, s, want in cases:
        got = oracle.awq_prescale([[x]], [s])[0, 0]
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (x, s, got)


def test_awq_prescale_matches_library_bf16_multiply():
    g = np.random.default_rng(51)
    x = g.standard_normal((7, 96)).astype(ml_dtypes.bfloat16)
    s = g.uniform(0.05, 8.0, 96).astype(ml_dtypes.bfloat16)
    want = (x * s[None, :]).astype(np.float64)     # float32 product, one rounding to bf16
    got = oracle.awq_prescale(x.astype(np.float64), s.astype(np.float64))
    assert np.array_equal(got, want)


def test_prescaled_w4a16_brute_force():
    # the scale runs along K (input channels), not along M or N
    g = np.random.default_rng(52)
    m, n, k = 3, 5, 48
    x = g.standard_normal((m, k)).astype(ml_dtypes.bfloat16)
    s = g.uniform(0.1, 3.0, k).astype(ml_dtypes.bfloat16)
    b, sb = _rand_nvfp4(n, k, 53)
    d = oracle.gemm_w4a16_prescaled(x.astype(np.float64), s.astype(np.float64), b, sb, np.float32(0.5),
                                    round_bf16=False)
    bv = _lib_decode(b, sb)
    for i in range(m):
        for j in range(n):
            acc = sum(float(x[i, t] * s[t]) * bv[j, t] for t in range(k))
            assert d[i, j] == pytest.approx(0.5 * acc, rel=1e-12, abs=1e-12)


# -- whole-MLP pin: a hand-built case whose every step is exact --------------
#
# H = I = 16 (one scale block everywhere), two tokens, all block scales 1.0
# (E4M3 byte 0x38).  x holds E2M1 values with |x| up to 6 and x[:, 0] = 4.
# Gate row j reads only x[0] with weight s_j = +-1 and alpha 8, so the gate is
# +-32: silu(32) = 32 / (1 + e^-32) differs from 32 by 1.3e-14 relative, far
# below half an fp32/bf16 ulp, and silu(-32) ~ -4e-13 vanishes in the NVFP4
# requantize.  Up row j reads only x[p_j] with weight 1, so u_j = 8 x[p_j] and
# h_j = 256 x[p_j] for s_j > 0.  With gs_h = 1/256 every selected block has
# amax 1536, scale 1.0 and codes equal to x[p_j] exactly.  Down row n holds
# d_n = +-1 at column sigma(n); alpha_down = 256 (= 1/gs_h) undoes gs_h, so
#     out[m, n] = 256 d_n x[m, p_sigma(n)]  if s_sigma(n) > 0, else 0
# in every composition; the W4A16 chain keeps the bf16 h and alpha_down = 1.
# A swapped gate/up half, a transposed weight, a lost alpha or a wrong index
# map changes this output.

_E2M1_CODE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
_X = np.array([[4, 1, -2, 0.5, 3, -6, 1.5, 2, 0, -1, 6, -0.5, 4, -3, 2, 1],
               [4, -1.5, 0, 6, -4, 2, -0.5, 3, 1, -2, 0.5, -6, 1.5, 0, -3, 4]], dtype=np.float64)
_P = [(3 * j + 1) % 16 for j in range(16)]                 # up row j reads x[p_j]
_S = [+1, -1, +1, +1, -1, +1, +1, -1, -1, +1, -1, -1, +1, -1, +1, +1]
_SIGMA = [(5 * n + 2) % 16 for n in range(16)]             # down row n reads h[sigma(n)]
_D = [+1 if n % 2 == 0 else -1 for n in range(16)]


def _code(v):
    return _E2M1_CODE[abs(v)] | (8 if v < 0 else 0)


def _pack_rows(dense):
    """Hand-coded E2M1 packing of a [rows, 16] matrix of E2M1 values; scale 1.0."""
    codes = np.array([[_code(v) for v in row] for row in dense], dtype=np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, np.full((dense.shape[0], 1), 0x38, dtype=np.uint8)


def _exact_mlp_case():
    gate = np.zeros((16, 16))
    up = np.zeros((16, 16))
    down = np.zeros((16, 16))
    for j in range(16):
        gate[j, 0] = _S[j]
        up[j, _P[j]] = 1.0
    for n in range(16):
        down[n, _SIGMA[n]] = _D[n]
    expected = np.zeros((2, 16))
    for m in range(2):
        for n in range(16):
            j = _SIGMA[n]
            expected[m, n] = 256.0 * _D[n] * _X[m, _P[j]] if _S[j] > 0 else 0.0
    return _pack_rows(np.vstack([gate, up])), _pack_rows(down), expected


def test_exact_mlp_case_is_well_posed():
    # each token's selected h block reaches |x| = 6, so its scale is exactly 1.0
    for m in range(2):
        assert max(abs(_X[m, _P[j]]) for j in range(16) if _S[j] > 0) == 6.0
    assert sorted(_P) == list(range(16)) and sorted(_SIGMA) == list(range(16))
    _, _, expected = _exact_mlp_case()
    # a few entries worked by hand: n = 0 -> sigma 2 (s +) -> p 7; n = 1 -> sigma 7 (s -)
    assert expected[0, 0] == 512.0 and expected[1, 0] == 768.0
    assert expected[0, 1] == 0.0 and expected[1, 1] == 0.0
    # n = 2 -> sigma 12 (s +) -> p 5, d = +1: x[0, 5] = -6, x[1, 5] = 2
    assert expected[0, 2] == -1536.0 and expected[1, 2] == 512.0


def test_whole_mlp_w4a4_fused_and_unfused_exact():
    w_gu, w_down, expected = _exact_mlp_case()
    args = (_X, 1.0, w_gu, 8.0, 1.0 / 256.0, w_down, 256.0)
    for fn in (oracle.mlp_w4a4_fused, oracle.mlp_w4a4_unfused):
        out = fn(*args)
        np.testing.assert_array_equal(out, expected, err_msg=fn.__name__)


def test_whole_mlp_w4a16_exact():
    w_gu, w_down, expected = _exact_mlp_case()
    out = oracle.mlp_w4a16(_X, w_gu, 8.0, w_down, 1.0)
    # the negative-gate rows keep silu(-32) * u ~ 1e-12 in bf16 here (no requantize)
    np.testing.assert_allclose(out, expected, rtol=0, atol=1e-6)
    nz = expected != 0
    np.testing.assert_array_equal(out[nz], expected[nz])


def test_silu_mul_bf16_rounds_once_from_the_exact_product():
    """Worked by hand: silu(17) = 17 / (1 + e^-17) = 16.99999929..., times
    1.1875 gives 20.18749916..., just below 20.1875, the midpoint between
    the bf16 neighbours 20.125 and 20.25 (quantum 1/8 on [16, 32)): one
    rounding gives 20.125.  Rounding to fp32 first would land exactly on the
    midpoint (fp32 spacing there is 2^-19) and tie to the even 20.25."""
    out = oracle.silu_mul_bf16(np.array([[17.0, 1.1875]]))
    assert out[0, 0] == 20.125


def _pack_e2m1_row(vals):
    codes = [_code(v) for v in vals]
    return np.array([codes[j] | (codes[j + 1] << 4) for j in range(0, 16, 2)], dtype=np.uint8)


def test_fused_swiglu_takes_the_unrounded_gate_up():
    """Worked by hand (one 16-block, scales 1.0, alpha 0.5, gs_h 1/8):
    x = [6, 6, 4, 0.5, 0...].  Gate row 0 = [6, 6, 2, 0.5] gives
    0.5 * 80.25 = 40.125; gate row 1 = [6, 6, 6] gives 48; up rows 0 and 1 =
    [0, 0, 0.5] give 1.  h = silu(g) * u is 40.125 and 48 (silu(g) = g within
    1e-16 here); the block amax 48 makes the scale 48/6 * 1/8 = 1.0, so the
    scaled values are 5.015625 -> E2M1 6 (code 7) and 6 (code 7).  Had the
    gate_up been rounded to bf16 first, 40.125 (a tie between 40 and 40.25)
    would become 40, the scaled value exactly 5, and the tie would go to the
    even 4 (code 6) -- which is what the unfused chain on a bf16 gate_up does."""
    x = np.zeros((1, 8), dtype=np.uint8)
    x[0] = _pack_e2m1_row([6, 6, 4, 0.5] + [0] * 12)
    w = np.zeros((32, 8), dtype=np.uint8)
    w[0] = _pack_e2m1_row([6, 6, 2, 0.5] + [0] * 12)
    w[1] = _pack_e2m1_row([6, 6, 6] + [0] * 13)
    w[16] = w[17] = _pack_e2m1_row([0, 0, 0.5] + [0] * 13)
    one = np.full((1, 1), 0x38, dtype=np.uint8)
    wsf = np.full((32, 1), 0x38, dtype=np.uint8)
    hq, hs = oracle.gemm_swiglu_quant(x, one, w, wsf, np.float32(0.5), np.float32(0.125))
    assert hs[0, 0] == 0x38
    assert list(hq[0]) == [0x77] + [0] * 7
    gu = oracle.gemm_w4a4(x, one, w, wsf, np.float32(0.5))          # the unfused chain's bf16 gate_up
    assert gu[0, 0] == 40.0 and gu[0, 1] == 48.0
    uq, us = oracle.silu_mul_quant(gu, np.float32(0.125))
    assert us[0, 0] == 0x38 and list(uq[0]) == [0x76] + [0] * 7
