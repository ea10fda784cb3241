"""Pins of the oracle's NVFP4 quantize: the hand-worked golden blocks, the
E2M1 / E4M3 steps reducing to library routines, and error bounds."""
import os

import ml_dtypes
import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_block.txt")


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        lines = f.read().splitlines()
    for line in lines:
        if not line.strip() or line.startswith("#"):
            continue
        name, gs, xs, sf, packed = [f.strip() for f in line.split("|")]
        cases.append((name, np.float32(gs), np.array(xs.split(), dtype=np.float32),
                      int(sf, 16), bytes.fromhex(packed.replace(" ", ""))))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_golden_blocks(case):
    name, gs, x, sf, packed = case
    p, s = oracle.quantize_nvfp4(x[None, :], gs)
    assert int(s[0, 0]) == sf
    assert bytes(p[0]) == packed


def test_steps_reduce_to_library_conversions():
    g = np.random.default_rng(5)
    x = (g.standard_normal((64, 256)) * np.exp(g.uniform(-3, 3, (64, 1)))).astype(np.float32)
    gs = oracle.global_scale(np.abs(x).max())
    p, sf, d = oracle.quantize_nvfp4(x, gs, detail=True)
    # step 3 = library E4M3 conversion of s (s <= 448 here by construction of gs)
    assert np.all(d["s"] <= np.float32(448.0 * (1 + 1e-6)))
    lib_sf = np.minimum(d["s"], np.float32(448)).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(sf, lib_sf)
    # step 6 = library E2M1 conversion of v
    lib_codes = d["v"].astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(oracle.e2m1_decode(d["codes"]), oracle.e2m1_decode(lib_codes))
    # step 7: low nibble holds the even (lower-K) element
    assert np.array_equal(p & 0xF, d["codes"][:, 0::2]) and np.array_equal(p >> 4, d["codes"][:, 1::2])


def test_max_block_maps_to_largest_scale():
    g = np.random.default_rng(6)
    x = g.standard_normal((8, 128)).astype(np.float32)
    gs = oracle.global_scale(np.abs(x).max())
    _, sf = oracle.quantize_nvfp4(x, gs)
    assert sf.max() == 0x7E          # the block holding amax(x) gets SF = 448


def test_roundtrip_error_bounds():
    g = np.random.default_rng(7)
    x = g.standard_normal((256, 512)).astype(np.float32)
    gs = oracle.global_scale(np.abs(x).max())
    p, sf, d = oracle.quantize_nvfp4(x, gs, detail=True)
    v = d["v"].astype(np.float64)
    q = oracle.e2m1_decode(d["codes"])
    mag = np.abs(v)
    # half the gap between neighbouring E2M1 magnitudes around |v|
    half_step = np.where(mag < 2, 0.25, np.where(mag < 4, 0.5, 1.0))
    bound = np.maximum(half_step, mag - 6.0)
    assert np.all(np.abs(v - q) <= bound + 1e-12)
    # saturation excess: r <= 6 / (amax * (1 - 2^-4)) for normal SF, so |v| <= 6.4
    assert np.all(mag <= 6.0 / (1 - 2.0 ** -4) + 1e-6)
    s = d["s"].astype(np.float64)
    sfv = oracle.e4m3_decode(sf)
    normal = s >= 2.0 ** -6
    assert np.all(np.abs(sfv[normal] - s[normal]) <= s[normal] * 2.0 ** -4 + 1e-12)
    # dequantized tensor is close to x (FP4 relative error of a Gaussian ~ 0.1)
    xd = oracle.dequantize_nvfp4(p, sf) / float(gs)
    rel = np.linalg.norm(xd - x) / np.linalg.norm(x)
    assert 0.02 < rel < 0.15


def test_zero_scale_blocks_copy_sign():
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 16:] = -1e-30
    p, sf = oracle.quantize_nvfp4(x, np.float32(1.0))
    assert list(sf[0]) == [0, 0]
    assert np.all(p[0, :8] == 0x00) and np.all(p[0, 8:] == 0x88)


def test_unpack_inverts_packing():
    g = np.random.default_rng(8)
    codes = g.integers(0, 16, (7, 64), dtype=np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(oracle.unpack_codes(packed), codes)


def test_per_token_reduces_to_static_when_rows_share_amax():
    """Rows with equal amax: per-token quantize equals the static quantize with
    the shared global scale, and the row scale is its reciprocal."""
    g = np.random.default_rng(31)
    x = g.standard_normal((6, 128)).astype(np.float32)
    x[:, 0] = np.float32(5.0)                 # every row's amax is exactly 5
    x = np.clip(x, -4.5, 4.5).astype(np.float32)
    x[:, 0] = np.float32(5.0)
    p, s, rs = oracle.quantize_nvfp4_per_token(x)
    gs = oracle.global_scale(5.0)
    p2, s2 = oracle.quantize_nvfp4(x, gs)
    assert np.array_equal(p, p2) and np.array_equal(s, s2)
    assert np.all(rs == np.float32(np.float32(1.0) / gs))


def test_per_token_row_independence_and_zero_rows():
    g = np.random.default_rng(32)
    x = g.standard_normal((5, 64)).astype(np.float32) * np.array([1, 10, 0.01, 0, 1000], np.float32)[:, None]
    p, s, rs = oracle.quantize_nvfp4_per_token(x)
    assert rs[3] == np.float32(1.0) and np.all(s[3] == 0)
    assert np.all(oracle.e2m1_decode(oracle.unpack_codes(p[3:4])) == 0)   # +-0 codes
    for r in (0, 1, 2, 4):
        assert s[r].max() == 0x7E            # each row's own max block maps to SF 448
        p1, s1, r1 = oracle.quantize_nvfp4_per_token(x[r:r + 1])
        assert np.array_equal(p1[0], p[r]) and r1[0] == rs[r]
    # dequantized rows recover x within the FP4 error
    xd = oracle.dequantize_nvfp4(p, s) * rs[:, None].astype(np.float64)
    for r in (0, 1, 2, 4):
        assert np.linalg.norm(xd[r] - x[r]) <= 0.15 * np.linalg.norm(x[r])
