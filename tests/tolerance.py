"""Acceptance rules for comparing the CUDA path with the CPU oracle.

* bf16 GEMM outputs: relative Frobenius error <= 1e-3 against the oracle's
  float64 result rounded once to bf16.  (Rounding to bf16 alone already costs
  ~1.7e-3 against the unrounded double, so the bound is read against the
  bf16-rounded reference.)
* Requantized NVFP4 outputs (codes + E4M3 scales): a block scale may differ by
  one E4M3 step only where the oracle's pre-rounding s lies within 1e-3
  relative of an E4M3 rounding midpoint; such blocks are re-quantized by the
  oracle with the GPU's scale before codes are compared.  A code may differ by
  one E2M1 step only where the oracle's pre-rounding |v| lies within 1e-3
  relative of an E2M1 rounding boundary, on at most 0.5% of elements.
"""
import numpy as np

import oracle

E2M1_BOUNDARIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_T = oracle.e4m3_table()
E4M3_MIDPOINTS = (_T[1:] + _T[:-1]) / 2.0
REL_WINDOW = 1e-3
MAX_FLIP_FRAC = 0.005
GEMM_REL_FROB = 1e-3


def rel_frobenius(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def assert_gemm_close(got, ref, tol=GEMM_REL_FROB, what="gemm"):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = rel_frobenius(got, ref)
    assert err <= tol, f"{what}: relative Frobenius error {err:.3e} > {tol:.1e}"
    return err


def _signed_ordinal(codes):
    idx = (codes & 7).astype(np.int64)
    return np.where((codes & 8) != 0, -idx, idx)


def near(values, boundaries, window=REL_WINDOW):
    values = np.abs(np.asarray(values, dtype=np.float64))[..., None]
    return np.any(np.abs(values - boundaries) <= window * boundaries, axis=-1)


def check_requant(got_packed, got_sf_lin, h, gs, max_frac=MAX_FLIP_FRAC, what="requant", window=REL_WINDOW):
    """got_*: GPU codes [rows, K/2] and linear SF [rows, K/16]; h: the
    oracle's fp32 pre-quantization tensor [rows, K]; gs: global scale.
    Returns (number of flipped codes, number of differing scale bytes)."""
    h = np.asarray(h, dtype=np.float32)
    rows, k = h.shape
    ref_packed, ref_sf, det = oracle.quantize_nvfp4(h, gs, detail=True)
    got_sf_lin = np.asarray(got_sf_lin, dtype=np.uint8)
    assert got_sf_lin.shape == ref_sf.shape
    sf_diff = got_sf_lin != ref_sf
    if np.any(sf_diff):
        s_bad = det["s"][sf_diff]
        ok = near(s_bad, E4M3_MIDPOINTS, window) & (np.abs(got_sf_lin[sf_diff].astype(int) - ref_sf[sf_diff].astype(int)) == 1)
        assert np.all(ok), (f"{what}: {int((~ok).sum())} block scales differ away from an E4M3 midpoint; "
                            f"first got={got_sf_lin[sf_diff][~ok][:4]} ref={ref_sf[sf_diff][~ok][:4]} s={s_bad[~ok][:4]}")
    # reference codes and pre-rounding values, with the GPU's scale in differing blocks
    ref_codes = det["codes"].copy()
    v = det["v"].copy()
    if np.any(sf_diff):
        sf_val = oracle.e4m3_decode(got_sf_lin).astype(np.float32)
        with np.errstate(divide="ignore"):
            r = np.where(got_sf_lin == 0, np.float32(0), np.float32(gs) / sf_val).astype(np.float32)
        v2 = (h.reshape(rows, k // 16, 16) * r[..., None]).astype(np.float32).reshape(rows, k)
        blk = np.repeat(sf_diff, 16, axis=1)
        v = np.where(blk, v2, v)
        ref_codes = np.where(blk, oracle.e2m1_encode(v2), ref_codes)
    got_codes = oracle.unpack_codes(got_packed)
    assert got_codes.shape == ref_codes.shape
    vg, vr = oracle.e2m1_decode(got_codes), oracle.e2m1_decode(ref_codes)
    diff = vg != vr                      # +0 and -0 compare equal
    if np.any(diff):
        step = np.abs(_signed_ordinal(got_codes[diff]) - _signed_ordinal(ref_codes[diff]))
        step = np.where((got_codes[diff] & 7) == 0, np.abs(_signed_ordinal(ref_codes[diff])), step)
        step = np.where((ref_codes[diff] & 7) == 0, np.abs(_signed_ordinal(got_codes[diff])), step)
        nb = near(v[diff], E2M1_BOUNDARIES, window)
        # a non-zero code must carry the sign of the pre-rounding value
        sign_ok = ((got_codes[diff] & 7) == 0) | (((got_codes[diff] & 8) != 0) == np.signbit(v[diff]))
        bad = ~((step == 1) & nb & sign_ok)
        assert not np.any(bad), (f"{what}: {int(bad.sum())} codes differ by more than one step or away from a "
                                 f"rounding boundary; v={v[diff][bad][:6]} got={got_codes[diff][bad][:6]} "
                                 f"ref={ref_codes[diff][bad][:6]}")
    nflip = int(diff.sum())
    assert nflip <= max_frac * diff.size, f"{what}: {nflip} flipped codes > {max_frac:.1%} of {diff.size}"
    return nflip, int(sf_diff.sum())
