"""CPU oracle for the NVFP4-quantized dense MLP.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or run it.  It shares no
code, table or helper with the CUDA library in ``nvfp4_quantized_dense_gb300``.

It is deliberately plain and slow: NumPy, float64 for every contraction, and
float32 only where the quantize recipe fixes single-precision rounding.

Sources (web pages on the subject, cited by title and section):

* [P1] sglang PR #34859 digest, "Add Qwen3.8-27B" (prhub.com.cn): the
  fused SiLU x mul + NVFP4 quantize of the dense MLP down_proj input and the
  6-D -> dense swizzled block-scale re-layout ("关键源码片段", qwen2_moe.py
  excerpt).
* [P2] sglang PR #26626 digest, "fused NVFP4 gate_up GEMM + SwiGLU + output
  quantize" (prhub.com.cn): the gate/up interleave in groups of 64 and the
  block-scale 2-D swizzle ("关键源码片段", modelopt_quant.py excerpt), the
  quantize -> fused GEMM -> down_proj call chain (deepseek_v2.py excerpt).
* [P3] sglang PR #35120 report, "FlashInfer CuTe DSL NVFP4 W4A16 mode":
  fp4_gemm W4A4 / W4A16 semantics ("关键源码片段", fp4_gemm), the linear
  [rows, K/16] E4M3 scale view ("关键源码片段", MoE excerpt), and "alpha holds
  only the weight dequant factor" in W4A16 ("实现拆解" item 3).
* OCP Microscaling Formats (MX) Specification v1.0: the E2M1 (FP4) and E4M3
  (FP8) element encodings, whose value tables the pages do not print.

Parity status per function is listed in each module header.
"""
from .formats import (E2M1_MAGNITUDES, e2m1_decode, e2m1_encode, e4m3_decode,
                      e4m3_encode, e4m3_table, bf16_round)
from .quant import quantize_nvfp4, quantize_nvfp4_per_token, dequantize_nvfp4, unpack_codes, global_scale
from .layouts import (sf_swizzle_128x4, sf_unswizzle_128x4, sf_swizzled_bytes,
                      interleave_gate_up, interleave_gate_up_scales_then_swizzle)
from .mlp import (gemm_w4a4, gemm_w4a4_per_token, gemm_w4a16, awq_prescale, gemm_w4a16_prescaled, silu, swiglu_h, silu_mul_quant, silu_mul_quant_masked,
                  silu_mul_bf16, gemm_swiglu_quant, mlp_w4a4_fused, mlp_w4a4_unfused,
                  mlp_w4a16)

__all__ = [n for n in dir() if not n.startswith("_")]
