"""The MLP contractions and the SwiGLU requantize, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

W4A4 GEMM ([P3] "关键源码片段", fp4_gemm with quant_mode "w4a4"):
    D[m, n] = alpha * sum_k (E2M1(A)*SF_A)[m, k] * (E2M1(B)*SF_B)[n, k]
in float64, then rounded once to bf16 (RNE).  alpha is the fp32 device scalar
1/(gs_a*gs_b), widened exactly to double.

W4A16 GEMM ([P3] "关键源码片段", fp4_gemm with quant_mode "w4a16";
"实现拆解" item 3: alpha holds only the weight dequant factor):
    D[m, n] = alpha * sum_k x[m, k] * (E2M1(B)*SF_B)[n, k], alpha = 1/gs_b.

NVFP4_AWQ pre-scale ([P3] "实现拆解" item 2: in W4A16 mode apply keeps the
AWQ pre_quant_scale multiply): x' = bf16(x[m, k] * s[k]), one rounding of the
exact product, then the W4A16 GEMM on x'.

SwiGLU ([P2] "实现拆解" item 1: gate_up GEMM -> silu -> FP4 quantize;
[P2] "关键源码片段": gate_up rows are [gate; up]):
    g = D[:, :I], u = D[:, I:] taken in float64 *before* bf16 rounding,
    silu(g) = g / (1 + exp(-g)),  h = fp32(silu(g) * u),
then h is quantized to NVFP4 with the static down_proj input scale.  Reading:
the fused path does not round h to bf16 (the pages are silent; their fused
kernel was checked against the unfused quantize "up to FP4 rounding ties").

silu_mul_nvfp4_quantize ([P1] "关键源码片段", qwen2_moe.py excerpt: one
kernel replaces act_fn + FP4 quant): the same h from a bf16 gate_up [M, 2I].
silu_mul_bf16 (the unfused ``act_fn``, used by the W4A16 chain): h rounded
once to bf16 from float64.

Pins (tests/test_oracle_mlp.py): brute-force triple loops on tiny shapes,
exact integer results with power-of-two scales, silu closed forms
(silu(0)=0, silu(x)-silu(-x)=x, limits), the fused == unfused invariant, and
W4A16 == W4A4 when x is exactly representable, hand-worked bf16 products of
the AWQ pre-scale and agreement with ml_dtypes' bf16 multiply.  The three MLP
compositions are pinned by a hand-built case whose every step is exact (gates
of +-32, power-of-two scales, permutation weights): the output is a signed,
scaled permutation of x worked out by hand, zero where the gate is negative.
"""
import numpy as np

from .formats import bf16_round
from .quant import dequantize_nvfp4, quantize_nvfp4


def gemm_w4a4(a_packed, a_sf, b_packed, b_sf, alpha, round_bf16=True):
    """A [M, K/2] + linear SF [M, K/16]; B [N, K/2] + linear SF [N, K/16]."""
    a = dequantize_nvfp4(a_packed, a_sf)
    b = dequantize_nvfp4(b_packed, b_sf)
    d = float(np.float32(alpha)) * (a @ b.T)
    return bf16_round(d) if round_bf16 else d


def gemm_w4a4_per_token(a_packed, a_sf, a_row_scale, b_packed, b_sf, alpha, round_bf16=True):
    """W4A4 GEMM with a per-row activation dequant factor:
    D[m, n] = alpha * row_scale[m] * sum_k (E2M1(A)*SF_A)(E2M1(B)*SF_B)."""
    a = dequantize_nvfp4(a_packed, a_sf)
    b = dequantize_nvfp4(b_packed, b_sf)
    rs = np.asarray(a_row_scale, dtype=np.float32).astype(np.float64)[:, None]
    d = float(np.float32(alpha)) * rs * (a @ b.T)
    return bf16_round(d) if round_bf16 else d


def gemm_w4a16(x, b_packed, b_sf, alpha, round_bf16=True):
    """x: bf16 values as float32/float64 [M, K]."""
    b = dequantize_nvfp4(b_packed, b_sf)
    d = float(np.float32(alpha)) * (np.asarray(x, dtype=np.float64) @ b.T)
    return bf16_round(d) if round_bf16 else d


def awq_prescale(x, pre_quant_scale):
    """NVFP4_AWQ activation pre-scale ([P3] "实现拆解" item 2: the W4A16 branch
    of the linear layer's apply multiplies x by the per-input-channel
    pre_quant_scale before the bf16 x FP4 GEMM).  Both are bf16 values; the
    product is taken in the activation type, i.e. the exact product rounded
    once to bf16 (exact in double: 8 x 8 significant bits).
    x [M, K], pre_quant_scale [K] -> [M, K] bf16 values as float64."""
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(pre_quant_scale, dtype=np.float64).reshape(1, -1)
    return bf16_round(x * s)


def gemm_w4a16_prescaled(x, pre_quant_scale, b_packed, b_sf, alpha, round_bf16=True):
    """W4A16 GEMM on the AWQ-pre-scaled activations ([P3] "实现拆解" item 2)."""
    return gemm_w4a16(awq_prescale(x, pre_quant_scale), b_packed, b_sf, alpha, round_bf16)


def silu(g):
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_h(gate_up):
    """float64 [M, 2I] = [gate | up] -> h = fp32(silu(gate) * up)."""
    gate_up = np.asarray(gate_up, dtype=np.float64)
    i = gate_up.shape[1] // 2
    return (silu(gate_up[:, :i]) * gate_up[:, i:]).astype(np.float32)


def silu_mul_quant(gate_up_bf16, gs_h, detail=False):
    """bf16 [M, 2I] (as float) -> NVFP4 (packed [M, I/2], linear SF)."""
    return quantize_nvfp4(swiglu_h(gate_up_bf16), gs_h, detail=detail)


def silu_mul_quant_masked(gate_up_groups, masked_m, gs_h):
    """Masked multi-group form ([P1] "关键源码片段", qwen2_moe.py excerpt:
    silu_and_mul_scaled_nvfp4_experts_quantize(gate_up[G, M, 2I], masked_m)):
    group e quantizes only its first masked_m[e] rows.  Returns per group
    (packed [valid, I/2], linear SF [valid, I/16]); the rows past masked_m[e]
    carry no data and zero scales."""
    out = []
    for e, g in enumerate(np.asarray(gate_up_groups)):
        valid = int(min(max(int(masked_m[e]), 0), g.shape[0]))
        out.append(silu_mul_quant(g[:valid], gs_h))
    return out


def silu_mul_bf16(gate_up_bf16):
    gate_up = np.asarray(gate_up_bf16, dtype=np.float64)
    i = gate_up.shape[1] // 2
    return bf16_round(silu(gate_up[:, :i]) * gate_up[:, i:])


def gemm_swiglu_quant(a_packed, a_sf, w_packed, w_sf, alpha, gs_h, detail=False):
    """The fused gate_up: plain [gate; up] weight (never the interleaved one)."""
    d = gemm_w4a4(a_packed, a_sf, w_packed, w_sf, alpha, round_bf16=False)
    return quantize_nvfp4(swiglu_h(d), gs_h, detail=detail)


def mlp_w4a4_fused(x, gs_x, w_gu, alpha_gu, gs_h, w_down, alpha_down):
    """quantize -> fused gate_up+SwiGLU+requant -> down_proj, bf16 out.
    w_gu / w_down are (packed, linear SF) tuples."""
    xq, xs = quantize_nvfp4(x, gs_x)
    hq, hs = gemm_swiglu_quant(xq, xs, *w_gu, alpha_gu, gs_h)
    return gemm_w4a4(hq, hs, *w_down, alpha_down)


def mlp_w4a4_unfused(x, gs_x, w_gu, alpha_gu, gs_h, w_down, alpha_down):
    """quantize -> gate_up GEMM (bf16) -> silu_mul_quant -> down_proj."""
    xq, xs = quantize_nvfp4(x, gs_x)
    gu = gemm_w4a4(xq, xs, *w_gu, alpha_gu)
    hq, hs = silu_mul_quant(gu, gs_h)
    return gemm_w4a4(hq, hs, *w_down, alpha_down)


def mlp_w4a16(x, w_gu, alpha_gu, w_down, alpha_down):
    """bf16 x -> gate_up (bf16) -> silu_mul_bf16 -> down_proj (bf16)."""
    gu = gemm_w4a16(x, *w_gu, alpha_gu)
    h = silu_mul_bf16(gu)
    return gemm_w4a16(h, *w_down, alpha_down)
