"""Tensor-parallel split of the NVFP4 dense MLP: the host-side plan.

The source pages show the dense MLP's one multi-GPU step: down_proj is
followed by a tensor-parallel all-reduce (or reduce-scatter) that the model
may skip when a fused variant performs it ([P2] sglang PR #26626 digest,
"关键源码片段", deepseek_v2.py excerpt: ``down_proj(..., skip_all_reduce=...)``).
The split that makes that all-reduce the only exchange:

* gate_up is column-parallel over the intermediate features I.  Rank r owns
  features [f0, f1), a multiple of 64 wide, so that whole groups of the
  fused kernel's gate/up interleave (64 up rows + 64 gate rows per 128-row
  block) stay on one rank.  Its gate_up shard is rows gate[f0:f1] and
  up[f0:f1] of the [gate; up] weight, in that order, and is prepared on the
  rank by nvfp4_prepare_gate_up_interleaved exactly as the full weight.
* down_proj is row-parallel over its K = I: rank r owns the input columns
  [f0, f1) of the down weight (whole 16-element scale blocks, and a K that
  is a multiple of 64 as the GEMMs require).
* Every shard uses the unsharded tensors' global scales: gs_x, one gs_w per
  weight and one static gs_h, hence one alpha for gate_up and one for
  down_proj on every rank.  h's 16-element blocks lie inside one rank's
  features, so each rank's NVFP4 h equals the matching columns of the
  unsharded h bit for bit.
* The exchange: each rank's partial down_proj output [M, H] in fp32, summed
  over the ranks by one all-reduce and rounded once to bf16.  Partials
  rounded to bf16 first would add one rounding per rank (about 2^-9 relative
  each), more than the 1e-3 GEMM tolerance.

This module only plans and slices; it runs no kernel.  The sharded chain is
checked on the CPU with gloo ranks against the unsharded oracle.  It has not
been run on more than one GPU.
"""
import numpy as np

GROUP = 64     # features per gate/up interleave group


def shard_features(inter, world):
    """[(f0, f1)] per rank: contiguous feature ranges of whole 64-feature
    groups, as even as the group count allows."""
    if inter <= 0 or inter % GROUP != 0:
        raise ValueError(f"intermediate size {inter} is not a positive multiple of {GROUP}")
    groups = inter // GROUP
    if world < 1 or groups < world:
        raise ValueError(f"{groups} feature groups cannot be split over {world} ranks")
    bounds = [(r * groups // world) * GROUP for r in range(world + 1)]
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def gate_up_rows(inter, f0, f1):
    """Row indices of a rank's gate_up shard in the [gate; up] weight:
    gate rows f0..f1-1, then up rows I+f0..I+f1-1."""
    return np.concatenate([np.arange(f0, f1), inter + np.arange(f0, f1)])


def shard_gate_up(codes, sf_linear, inter, f0, f1):
    """The rank's gate_up codes [2(f1-f0), H/2] and linear scales
    [2(f1-f0), H/16] from the unsharded [gate; up] ones (arrays indexable by
    an integer row array)."""
    rows = gate_up_rows(inter, f0, f1)
    return codes[rows], sf_linear[rows]


def shard_down(codes, sf_linear, f0, f1):
    """The rank's down_proj codes [H, (f1-f0)/2] and linear scales
    [H, (f1-f0)/16]: input columns f0..f1-1 (two codes per byte, one scale
    per 16 columns)."""
    if f0 % GROUP or f1 % GROUP:
        raise ValueError("down_proj shards start and end on 64-column boundaries")
    return codes[:, f0 // 2:f1 // 2], sf_linear[:, f0 // 16:f1 // 16]
