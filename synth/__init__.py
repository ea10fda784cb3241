"""Seeded synthetic inputs for the NVFP4 dense-MLP workloads.

This module holds no NVFP4 arithmetic: it only draws the raw tensors (bf16
activations, fp32 weights) that both the CPU oracle and the CUDA path then
consume.  Recipe:

* generator: NumPy ``Generator(PCG64(SeedSequence([seed, workload_id, tensor_id])))``
  with seed 0 everywhere;
* x ~ N(0, 1) in fp32, rounded to bf16 (RNE) -- drawn at the workload's
  largest M, smaller M take the leading rows;
* the DeepSeek-V3-shaped decode workload adds outliers: each element is, with
  probability 0.01 (seeded Bernoulli mask), multiplied by 20 before the bf16
  cast;
* weights W_gu [2I, H] (rows [gate; up]) and W_down [H, I] ~ N(0, 0.02) fp32.
"""
from dataclasses import dataclass

import numpy as np
import torch

SEED = 0


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    hidden: int
    inter: int
    ms: tuple
    mode: str            # "w4a4" or "w4a16"
    outliers: bool = False
    fused: bool = True   # gate_up through the fused SwiGLU+requant kernel


WORKLOADS = {
    0: Workload(0, "tiny NVFP4 dense MLP (H256 I512)", 256, 512, (4,), "w4a4"),
    1: Workload(1, "decode dense MLP W4A4 (H5120 I17408)", 5120, 17408, (1, 2, 4, 8, 16), "w4a4",
                fused=False),
    2: Workload(2, "decode dense MLP W4A4 DeepSeek-V3-shaped (H7168 I18432)", 7168, 18432,
                (1, 8, 32, 64), "w4a4", outliers=True),
    3: Workload(3, "prefill dense MLP W4A4 (H7168 I18432)", 7168, 18432, (1024, 4096, 8192), "w4a4"),
    4: Workload(4, "W4A16 dense MLP (H5120 I17408)", 5120, 17408, (1, 16, 128, 1024), "w4a16"),
}

T_X, T_WGU, T_WDOWN, T_OUTLIER, T_AWQ = 0, 1, 2, 3, 4

# Workloads with the same MLP shape draw the same weights: the prefill
# workload reuses the DeepSeek-V3-shaped decode weights and the W4A16 workload
# the H5120/I17408 ones.
WEIGHT_SOURCE = {3: 2, 4: 1}


def rng(wid, tensor_id, seed=SEED):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, wid, tensor_id])))


def to_bf16_bits(x_f32):
    """fp32 ndarray -> (uint16 bf16 bit patterns, float32 values of those bf16)."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    return bits, t.to(torch.float32).numpy()


def activations(wid, m, k=None, outliers=None, seed=SEED):
    """bf16 x [m, k] as (bits uint16, values float32)."""
    w = WORKLOADS[wid]
    k = w.hidden if k is None else k
    mmax = max(max(w.ms), m)
    x = rng(wid, T_X, seed).standard_normal((mmax, k), dtype=np.float32)
    if (w.outliers if outliers is None else outliers):
        mask = rng(wid, T_OUTLIER, seed).random((mmax, k)) < 0.01
        x = np.where(mask, x * np.float32(20.0), x).astype(np.float32)
    return to_bf16_bits(x[:m])


def weight(wid, which, rows=None, cols=None, seed=SEED):
    """fp32 weights ~ N(0, 0.02): which='gate_up' -> [2I, H], 'down' -> [H, I]."""
    wid = WEIGHT_SOURCE.get(wid, wid)
    w = WORKLOADS[wid]
    if which == "gate_up":
        shape, tid = (2 * w.inter, w.hidden), T_WGU
    elif which == "down":
        shape, tid = (w.hidden, w.inter), T_WDOWN
    else:
        raise ValueError(which)
    shape = (rows or shape[0], cols or shape[1])
    return (rng(wid, tid, seed).standard_normal(shape, dtype=np.float32) * np.float32(0.02)).astype(np.float32)


def awq_pre_quant_scale(wid, k=None, seed=SEED):
    """Per-input-channel AWQ activation scales, bf16 [k] as (bits, values):
    positive, log-uniform over [1/4, 4] (AWQ scales are positive factors near
    1 that grow on the channels with large activations)."""
    w = WORKLOADS[wid]
    k = w.hidden if k is None else k
    e = rng(wid, T_AWQ, seed).uniform(-2.0, 2.0, k)
    return to_bf16_bits(np.exp2(e).astype(np.float32))


def random_matrix(shape, seed_key, scale=1.0, dtype=np.float32):
    """Generic seeded N(0, scale^2) matrix for shape sweeps in tests."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([SEED, 1000] + list(seed_key))))
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(scale)).astype(dtype)
