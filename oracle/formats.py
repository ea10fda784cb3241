"""Scalar number formats of NVFP4, written from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* E2M1 (4-bit float, 1 sign, 2 exponent, 1 mantissa bit, no inf/NaN): the
  element type of NVFP4 data.  OCP MX v1.0, FP4 E2M1 table: magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}; code bits 0-2 index that list, bit 3 is the
  sign.  Pinned by tests/test_oracle_formats.py against ml_dtypes.float4_e2m1fn
  and against every rounding boundary.
* E4M3 ("e4m3fn": bias 7, no inf, 0x7F/0xFF NaN, max 448, subnormals down to
  2^-9): the per-16-element block-scale type (the pages view the scales as
  ``torch.float8_e4m3fn`` in [P3] "关键源码片段", MoE excerpt).  Pinned
  against torch.float8_e4m3fn and ml_dtypes.float8_e4m3fn.
* bf16: correctly rounded (round-to-nearest-even) from float64 in one step.
  Pinned against torch's float32 -> bfloat16 cast on float32-exact inputs and
  against a hand-derived double-rounding case.

Rounding rule used by both encoders (the plainest reading of "round to
nearest even, saturate to the largest finite value"): pick the nearest
representable magnitude; on an exact tie pick the one whose code is even
(its mantissa LSB is 0); magnitudes above the largest finite value map to
it.  The sign bit is copied from the input's sign bit, so a negative value
that rounds to zero becomes -0.
"""
import numpy as np

E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e4m3_table():
    """Magnitudes of the 127 finite non-negative E4M3 codes 0x00..0x7E."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        if e == 0:
            vals.append(m / 8.0 * 2.0 ** -6)
        else:
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_E4M3 = e4m3_table()
_E2M1 = np.array(E2M1_MAGNITUDES, dtype=np.float64)


def _round_to_table(mag, table):
    """Index of the nearest entry of ascending ``table`` to each ``mag``
    (non-negative float64), ties to the even index, saturating at the end."""
    mag = np.minimum(np.asarray(mag, dtype=np.float64), table[-1])
    hi = np.searchsorted(table, mag, side="left")  # table[hi-1] < mag <= table[hi]
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - table[lo]
    d_hi = table[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag == table[hi], hi, idx)
    return idx.astype(np.uint8)


def e2m1_encode(v):
    """float32/float64 array -> E2M1 codes (uint8, low nibble used)."""
    v = np.asarray(v)
    idx = _round_to_table(np.abs(v.astype(np.float64)), _E2M1)
    return (idx | (np.signbit(v).astype(np.uint8) << 3)).astype(np.uint8)


def e2m1_decode(codes):
    """E2M1 codes (uint8, low nibble) -> float64 values (code 8 gives -0.0)."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = _E2M1[codes & 7]
    return np.where((codes & 8) != 0, -mag, mag)


def e4m3_encode(s):
    """Non-negative float32/float64 array -> E4M3 codes, RNE, satfinite."""
    s = np.asarray(s, dtype=np.float64)
    if np.any(s < 0) or np.any(np.isnan(s)):
        raise ValueError("block scales are non-negative and finite")
    return _round_to_table(s, _E4M3)


def e4m3_decode(codes):
    """E4M3 codes (0x00..0x7E, non-negative) -> float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    if np.any((codes & 0x7F) == 0x7F):
        raise ValueError("NaN code in a block scale")
    mag = _E4M3[codes & 0x7F]
    return np.where((codes & 0x80) != 0, -mag, mag)


_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x):
    """float64 -> float64 holding the bf16 value nearest to x (RNE), rounded
    once from the double (no intermediate float32); overflow gives +-inf."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    q = np.maximum(e.astype(np.int64) - 8, -133)  # 8 significant bits; subnormal quantum 2^-133
    y = np.ldexp(np.round(np.ldexp(x, -q)), q)    # np.round is half-to-even
    return np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, x), y)
