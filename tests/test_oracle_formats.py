"""Pins of the oracle's scalar formats against library routines and
hand-derived values (E2M1 / E4M3 tables of the OCP MX v1.0 spec)."""
import ml_dtypes
import numpy as np
import pytest
import torch

import oracle

B_E2M1 = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]


def _ml_e2m1(v):
    return np.asarray(v, dtype=np.float32).astype(ml_dtypes.float4_e2m1fn).astype(np.float64)


def test_e2m1_decode_matches_library_table():
    codes = np.arange(16, dtype=np.uint8)
    lib = codes.view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    ours = oracle.e2m1_decode(codes)
    assert np.array_equal(ours, lib)
    assert np.array_equal(np.signbit(ours), np.signbit(lib))
    assert list(ours[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e2m1_encode_boundaries_and_neighbours():
    vals = []
    for b in B_E2M1 + [0.5, 1, 1.5, 2, 3, 4, 6]:
        b32 = np.float32(b)
        vals += [b32, np.nextafter(b32, np.float32(0)), np.nextafter(b32, np.float32(10))]
    vals = np.array(vals, dtype=np.float32)
    vals = np.concatenate([vals, -vals])
    ours = oracle.e2m1_decode(oracle.e2m1_encode(vals))
    assert np.array_equal(ours, _ml_e2m1(vals))
    # ties go to the even code
    tie_codes = oracle.e2m1_encode(np.array(B_E2M1, dtype=np.float32))
    assert list(tie_codes) == [0, 2, 2, 4, 4, 6, 6]


def test_e2m1_encode_random_vs_library():
    g = np.random.default_rng(1)
    v = (g.random(2_000_000, dtype=np.float32) * 12 - 6).astype(np.float32)
    assert np.array_equal(oracle.e2m1_decode(oracle.e2m1_encode(v)), _ml_e2m1(v))


def test_e2m1_saturates_and_keeps_sign_of_zero():
    v = np.array([6.0, 6.5, 7.0, 1e9, -8.0, -0.1, -0.0, 0.0, -0.25], dtype=np.float32)
    codes = oracle.e2m1_encode(v)
    assert list(codes) == [7, 7, 7, 7, 15, 8, 8, 0, 8]


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(0x7F, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_decode(codes), lib)
    assert oracle.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert oracle.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9


def test_e4m3_encode_midpoints_vs_libraries():
    t = oracle.e4m3_table()
    mids = ((t[1:] + t[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e4)),
                           t.astype(np.float32)]).astype(np.float32)
    ours = oracle.e4m3_encode(vals)
    lib_t = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    lib_m = vals.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(ours, lib_t)
    assert np.array_equal(ours, lib_m)


def test_e4m3_encode_random_vs_library_and_saturation():
    g = np.random.default_rng(2)
    v = np.exp(g.uniform(np.log(1e-5), np.log(448.0), 1_000_000)).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), lib)
    big = np.array([448.0, 449.0, 464.0, 479.9, 480.0, 1e6, 3.4e38], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    tiny = np.array([0.0, 2.0 ** -11, 2.0 ** -10, np.nextafter(np.float32(2.0 ** -10), np.float32(1))], dtype=np.float32)
    assert list(oracle.e4m3_encode(tiny)) == [0, 0, 0, 1]   # 2^-10 is the tie between 0 and 2^-9 -> even (0)


def test_bf16_round_vs_torch_on_float32_inputs():
    g = np.random.default_rng(3)
    v = (g.standard_normal(1_000_000) * np.exp(g.uniform(-30, 30, 1_000_000))).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_round(v.astype(np.float64)), lib)


def test_bf16_round_single_rounding_from_double():
    # 1 + 2^-8 + 2^-30 is just above the bf16 tie 1 + 2^-8: correct rounding gives 1 + 2^-7,
    # whereas rounding through float32 first lands on the tie and then on 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert oracle.bf16_round(x) == 1.0 + 2.0 ** -7
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 1.0            # exact tie -> even
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie -> even mantissa
    assert oracle.bf16_round(3.4e38) == np.inf
    assert oracle.bf16_round(-3.0e38) == np.float64(torch.tensor(-3.0e38).to(torch.bfloat16).item())
    assert oracle.bf16_round(2.0 ** -135) == 0.0                 # below half the smallest subnormal
    assert oracle.bf16_round(3 * 2.0 ** -134) == 2.0 ** -132


@pytest.mark.parametrize("x", [0.0, -0.0, 1.0, -2.5])
def test_bf16_round_identity_on_representable(x):
    y = oracle.bf16_round(x)
    assert y == x and np.signbit(y) == np.signbit(x)
