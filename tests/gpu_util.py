"""Helpers for the GPU parity tests: device upload, oracle-quantized weight
sets (cached per process), and sampling of large outputs."""
import functools

import numpy as np
import torch

import oracle
import synth


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def scalar(v):
    return torch.tensor([np.float32(v)], dtype=torch.float32, device="cuda")


def host(t):
    return t.detach().cpu().numpy()


def bf16_host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def quantize_big(w, gs, chunk=4096):
    """oracle.quantize_nvfp4 applied block of rows by block of rows."""
    packed = np.empty((w.shape[0], w.shape[1] // 2), dtype=np.uint8)
    sf = np.empty((w.shape[0], w.shape[1] // 16), dtype=np.uint8)
    for r in range(0, w.shape[0], chunk):
        packed[r:r + chunk], sf[r:r + chunk] = oracle.quantize_nvfp4(w[r:r + chunk], gs)
    return packed, sf


class WeightSet:
    """One NVFP4 weight tensor: oracle codes + linear scales + global scale."""

    def __init__(self, w_f32):
        self.n, self.k = w_f32.shape
        self.gs = oracle.global_scale(np.abs(w_f32).max())
        self.packed, self.sf = quantize_big(w_f32, self.gs)
        self._dev = {}

    def device_prepared(self, nv):
        """Codes + swizzled scales on the device, made by nvfp4_prepare_weights."""
        if "plain" not in self._dev:
            w = dev(self.packed)
            sfo = torch.empty(nv.nvfp4_sf_bytes(self.n, self.k), dtype=torch.uint8, device="cuda")
            nv.nvfp4_prepare_weights(w, dev(self.sf), self.n, self.k, w, sfo)
            self._dev["plain"] = (w, sfo)
        return self._dev["plain"]

    def device_interleaved(self, nv):
        if "inter" not in self._dev:
            w = torch.empty_like(dev(self.packed))
            sfo = torch.empty(nv.nvfp4_sf_bytes(self.n, self.k), dtype=torch.uint8, device="cuda")
            nv.nvfp4_prepare_gate_up_interleaved(dev(self.packed), dev(self.sf), self.n, self.k, w, sfo)
            self._dev["inter"] = (w, sfo)
        return self._dev["inter"]


@functools.lru_cache(maxsize=None)
def weights(wid, which):
    return WeightSet(synth.weight(wid, which))


@functools.lru_cache(maxsize=None)
def small_weights(rows, cols, key):
    return WeightSet(synth.random_matrix((rows, cols), (7, rows, cols, key), scale=0.02))


def quantized_activation(wid, m, k=None):
    """(bf16 bits, fp32 values, gs, packed, linear sf) of the workload's x[:m]."""
    bits, x = synth.activations(wid, m, k)
    gs = oracle.global_scale(np.abs(x).max())
    packed, sf = oracle.quantize_nvfp4(x, gs)
    return bits, x, gs, packed, sf


def sample_rows(n, count, seed=0, block=1):
    """Sorted sample of row indices (whole blocks of `block` rows), stratified:
    the n // block blocks are cut into `count` equal strata and one block is
    drawn from each, the first and the last block always included, so that a
    sample at least as large as the number of kernel tiles touches every tile."""
    g = np.random.default_rng(seed)
    nb = n // block
    if count >= nb:
        pick = np.arange(nb)
    else:
        edges = np.linspace(0, nb, count + 1).astype(np.int64)
        pick = np.array([g.integers(lo, hi) for lo, hi in zip(edges[:-1], edges[1:])], dtype=np.int64)
        pick[0], pick[-1] = 0, nb - 1
        pick = np.unique(pick)
    return (pick[:, None] * block + np.arange(block)[None, :]).reshape(-1)
