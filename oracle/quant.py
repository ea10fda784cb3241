"""NVFP4 block quantize / dequantize.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix: activations are quantized with a static fp32 per-tensor
global scale ``input_scale_inv`` ([P2] "关键源码片段", deepseek_v2.py excerpt:
``fp4_quantize(x, gate_up_proj.input_scale_inv)``), into packed E2M1 data
``[rows, K/2]`` ([P1] "关键源码片段", qwen2_moe.py excerpt) with one E4M3 scale
per 16 elements along K ([P3] "关键源码片段", MoE excerpt:
``_FP4_SF_VEC_SIZE``, ``hidden_size // _FP4_SF_VEC_SIZE``).

What the pages leave open, and the reading taken (each step is a correctly
rounded IEEE float32 operation, in this order), for one block b of 16:

  1. amax = max_i |x_i|
  2. s    = fp32( fp32(amax / 6) * gs )
  3. SF   = E4M3(s)                     round-to-nearest-even, satfinite
  4. r    = 0 if SF == 0 else fp32(gs / float(SF))
  5. v_i  = fp32(x_i * r)
  6. code_i = E2M1(v_i)                 round-to-nearest-even, satfinite, sign kept
  7. packed byte j = code_{2j} | code_{2j+1} << 4   (lower K in the low nibble)

Dequantized value: E2M1(code) * float(SF); the 1/gs factor lives in the GEMM
alpha ([P2] "关键源码片段": one ``alpha`` handed to the fused kernel).

Global scale: gs = fp32(448 * 6 / amax(tensor)) -- the value that maps the
tensor's largest magnitude onto the largest E4M3 scale times the largest E2M1
magnitude.  Pinned by tests/test_oracle_quant.py: E2M1/E4M3 reduce to
library routines, round-trip error bounds, the max block mapping to SF=448,
and a hand-computed worked block (tests/golden/quant_block.txt).
"""
import numpy as np

from .formats import e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode

BLOCK = 16


def global_scale(amax):
    """fp32(448 * 6 / amax)."""
    return np.float32(np.float32(448.0 * 6.0) / np.float32(amax))


def quantize_nvfp4(x, gs, detail=False):
    """x: float32 [rows, K] with K % 16 == 0; gs: float32 global scale.

    Returns (packed uint8 [rows, K/2], sf uint8 [rows, K/16] linear).  With
    ``detail`` also returns a dict of every intermediate (amax, s, r, v,
    codes) so that tests can locate rounding boundaries."""
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    if k % BLOCK:
        raise ValueError("K must be a multiple of 16")
    gs = np.float32(gs)
    xb = x.reshape(rows, k // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=-1)                                   # step 1
    s = (amax / np.float32(6.0)).astype(np.float32) * gs             # step 2
    s = s.astype(np.float32)
    sf = e4m3_encode(s)                                              # step 3
    sf_val = e4m3_decode(sf).astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(sf == 0, np.float32(0.0), gs / sf_val).astype(np.float32)  # step 4
    v = (xb * r[..., None]).astype(np.float32)                       # step 5
    codes = e2m1_encode(v).reshape(rows, k)                          # step 6
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)  # step 7
    if not detail:
        return packed, sf
    return packed, sf, dict(amax=amax, s=s, r=r, v=v.reshape(rows, k), codes=codes)


def unpack_codes(packed):
    """uint8 [rows, K/2] -> E2M1 codes uint8 [rows, K] (low nibble first)."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, kh = packed.shape
    codes = np.empty((rows, kh * 2), dtype=np.uint8)
    codes[:, 0::2] = packed & 0x0F
    codes[:, 1::2] = packed >> 4
    return codes


def dequantize_nvfp4(packed, sf):
    """(packed [rows, K/2], linear sf [rows, K/16]) -> float64 [rows, K]
    holding E2M1(code) * float(SF), without the global 1/gs factor."""
    vals = e2m1_decode(unpack_codes(packed))
    rows, k = vals.shape
    scale = e4m3_decode(np.asarray(sf, dtype=np.uint8)[:, : k // BLOCK])
    return (vals.reshape(rows, k // BLOCK, BLOCK) * scale[..., None]).reshape(rows, k)


def quantize_nvfp4_per_token(x):
    """Per-token dynamic global scale ([P3] "关键源码片段", MoE excerpt:
    nvfp4_quantize(..., per_token_activation=True) returns a per-token scale).
    Reading: each row r gets its own gs_r = fp32(448 * 6 / amax(row r)) (an
    all-zero row uses gs_r = 1) and is quantized exactly as quantize_nvfp4 with
    it; the returned row scale fp32(1 / gs_r) is the per-row dequant factor a
    GEMM multiplies into row r.  Returns (packed, linear sf, row_scale)."""
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    packed = np.empty((rows, k // 2), dtype=np.uint8)
    sf = np.empty((rows, k // 16), dtype=np.uint8)
    row_scale = np.empty(rows, dtype=np.float32)
    for r in range(rows):
        amax = np.abs(x[r]).max()
        gs = global_scale(amax) if amax > 0 else np.float32(1.0)
        packed[r:r + 1], sf[r:r + 1] = quantize_nvfp4(x[r:r + 1], gs)
        row_scale[r] = np.float32(np.float32(1.0) / gs)
    return packed, sf, row_scale
