"""GPU parity of nvfp4_quantize_gemm_swiglu_quant (the activation quantize
folded into the fused gate_up launch) against the oracle.

Per call:
  * the quantized x it writes (codes and swizzled scales, padding rows of the
    scale block zero) is bit-exact against oracle.quantize_nvfp4;
  * h passes the requantize rule of tests/tolerance.py against the oracle's
    SwiGLU of the oracle's GEMM on that x (all features, or stratified
    16-feature blocks that touch every weight tile at full size);
  * h is bit-identical to the two launches it stands for (nvfp4_quantize,
    then nvfp4_gemm_swiglu_quant_ex on the swap-AB path) on the same inputs;
  * a second call on the same workspace gives the same bits and leaves the
    workspace's counter area at zero.
Shapes span the mixed split and the cluster split, ragged K, the 16/32/64
token tiles and both full decode workloads; larger M and a missing
workspace take the two-launch path.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, host, sample_rows, scalar, small_weights, weights
from tolerance import check_requant

pytestmark = pytest.mark.gpu

TC_SWAPAB = 3
COUNTER_AREA = 64 * 1024


def _buffers(nv, m, n, k, fill):
    inter = n // 2
    u8 = dict(dtype=torch.uint8, device="cuda")
    return (torch.full((m, k // 2), fill, **u8), torch.full((nv.nvfp4_sf_bytes(m, k),), fill, **u8),
            torch.full((m, inter // 2), fill, **u8), torch.full((nv.nvfp4_sf_bytes(m, inter),), fill, **u8))


def _case(nv, wid, m, n, k, ws, sampled_blocks=None, use_workspace=True):
    inter = n // 2
    xbits, x = synth.activations(wid, m, k)
    gs_x = oracle.global_scale(np.abs(x).max())
    xq_ref, xs_ref = oracle.quantize_nvfp4(x, gs_x)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    feats = np.arange(inter) if sampled_blocks is None else \
        sample_rows(inter, sampled_blocks, seed=m + 7, block=16)
    rows = np.concatenate([feats, inter + feats])           # gate rows, then up rows
    h = oracle.swiglu_h(oracle.gemm_w4a4(xq_ref, xs_ref, ws.packed[rows], ws.sf[rows], alpha, round_bf16=False))
    gs_h = oracle.global_scale(np.abs(h).max())
    wi = ws.device_interleaved(nv)
    xd = bf16_dev(xbits)
    nbytes = nv.nvfp4_quantize_gemm_swiglu_quant_workspace_bytes(m, n, k) if use_workspace else 0
    wsp = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    xq, xs, hq, hs = _buffers(nv, m, n, k, 0xAB)
    args = [xd, scalar(gs_x), xq, xs, wi[0], wi[1], scalar(alpha), scalar(gs_h), hq, hs, m, n, k,
            wsp if use_workspace else None, nbytes]
    nv.nvfp4_quantize_gemm_swiglu_quant(*args)
    torch.cuda.synchronize()
    got = [host(t).copy() for t in (xq, xs, hq, hs)]

    assert np.array_equal(got[0], xq_ref), "quantized x codes differ"
    assert np.array_equal(got[1], oracle.sf_swizzle_128x4(xs_ref)), "quantized x scales differ"
    s_lin = oracle.sf_unswizzle_128x4(got[3], m, inter // 16)
    codes = oracle.unpack_codes(got[2])[:, feats]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    nflip, nsf = check_requant(packed, s_lin[:, feats[::16] // 16], h, gs_h, what=f"fold m={m} n={n} k={k}")

    # the two launches it stands for, on fresh buffers and workspace
    xq2, xs2, hq2, hs2 = _buffers(nv, m, n, k, 0xCD)
    # (without a workspace both split the weight tiles the same way: whole tiles per CTA)
    wb2 = nv.nvfp4_workspace_bytes(m, n, k, TC_SWAPAB if m <= 64 else 0) if use_workspace else 0
    ws2 = torch.zeros(max(wb2, 16), dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize(xd, m, k, scalar(gs_x), xq2, xs2)
    nv.nvfp4_gemm_swiglu_quant_ex(xq2, xs2, wi[0], wi[1], scalar(alpha), scalar(gs_h), hq2, hs2, m, n, k,
                                  ws2 if use_workspace else None, wb2, TC_SWAPAB if m <= 64 else 0)
    torch.cuda.synchronize()
    assert np.array_equal(host(hq2), got[2]) and np.array_equal(host(hs2), got[3]), \
        "the fold and the two launches give different h"

    # again on the same workspace: same bits, counters back at zero
    for t in (xq, xs, hq, hs):
        t.fill_(0xCD)
    nv.nvfp4_quantize_gemm_swiglu_quant(*args)
    torch.cuda.synchronize()
    assert all(np.array_equal(host(t), g) for t, g in zip((xq, xs, hq, hs), got)), "reused workspace differs"
    if use_workspace:
        assert not host(wsp[:min(nbytes, COUNTER_AREA)].view(torch.int32)).any(), "counters not reset"
    print(f"fold m={m} n={n} k={k}: {nflip} boundary flips, {nsf} scale diffs")


# (33, 3072, 2048) takes the cluster split (24 tiles x 6 CTAs)
SMALL = [(1, 256, 256), (4, 1024, 256), (3, 128, 320), (16, 384, 4096), (40, 256, 512),
         (64, 1024, 1024), (16, 4096, 1024), (33, 3072, 2048)]


@pytest.mark.parametrize("m,n,k", SMALL)
def test_fold_small_shapes(lib, m, n, k):
    _case(lib, 0, m, n, k, small_weights(n, k, 6))


@pytest.mark.parametrize("m", [1, 4, 16])
def test_fold_h5120_full_size_sampled(lib, m):
    """The decode step's gate_up (interleaved 34816 x 5120 weight): 272
    stratified 16-feature blocks, one in each 128-row weight tile."""
    ws = weights(1, "gate_up")
    _case(lib, 1, m, ws.n, ws.k, ws, sampled_blocks=272)


@pytest.mark.parametrize("m", [1, 8, 64])
def test_fold_deepseek_full_size_sampled(lib, m):
    """DeepSeek-V3-shaped decode gate_up (36864 x 7168), x with outliers."""
    ws = weights(2, "gate_up")
    _case(lib, 2, m, ws.n, ws.k, ws, sampled_blocks=288)


@pytest.mark.parametrize("m,n,k", [(65, 1024, 512), (130, 256, 256)])
def test_fold_larger_m_takes_two_launches(lib, m, n, k):
    _case(lib, 0, m, n, k, small_weights(n, k, 6))


def test_fold_without_workspace_takes_two_launches(lib):
    _case(lib, 0, 4, 1024, 256, small_weights(1024, 256, 6), use_workspace=False)


def test_fold_bounded_wait_gives_up_cleanly(lib):
    """With a wait limit of one poll the phase-A and pipeline waits run out:
    the kernel records NVFP4_ERR_DEVICE_TIMEOUT and returns; on a fresh
    workspace the next normal call is correct."""
    m, n, k = 4, 1024, 4096
    ws = small_weights(n, k, 6)
    xbits, x = synth.activations(0, m, k)
    gs_x = oracle.global_scale(np.abs(x).max())
    wi = ws.device_interleaved(lib)
    nbytes = lib.nvfp4_quantize_gemm_swiglu_quant_workspace_bytes(m, n, k)
    wsp = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    xq, xs, hq, hs = _buffers(lib, m, n, k, 0)
    assert lib.nvfp4_get_device_status() == 0
    lib.nvfp4_set_wait_limit(1)
    try:
        lib.nvfp4_quantize_gemm_swiglu_quant(bf16_dev(xbits), scalar(gs_x), xq, xs, wi[0], wi[1], scalar(1e-3),
                                             scalar(1.0), hq, hs, m, n, k, wsp, nbytes)
        torch.cuda.synchronize()
    finally:
        lib.nvfp4_set_wait_limit(0)
    assert lib.nvfp4_get_device_status() == lib.ERR_DEVICE_TIMEOUT
    assert lib.nvfp4_get_device_status() == 0
    _case(lib, 0, m, n, k, ws)


def test_fold_argument_errors(lib):
    m, n, k = 4, 1024, 256
    ws = small_weights(n, k, 6)
    wi = ws.device_interleaved(lib)
    x = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    one = scalar(1.0)
    base = [x, one, buf, buf, wi[0], wi[1], one, one, buf, buf, m, n, k, buf, 1 << 20]

    def status(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        with pytest.raises(lib.Nvfp4Error) as e:
            lib.nvfp4_quantize_gemm_swiglu_quant(*a)
        return e.value.status

    assert status(a0=None) == lib.ERR_INVALID_ARG                  # missing x
    assert status(a1=None) == lib.ERR_INVALID_ARG                  # missing x scale
    assert status(a11=1000) == lib.ERR_UNSUPPORTED_SHAPE           # n % 128
    assert status(a12=100) == lib.ERR_UNSUPPORTED_SHAPE            # k % 64
    assert lib.nvfp4_quantize_gemm_swiglu_quant_workspace_bytes(0, n, k) == 0


def test_fold_m_zero_is_a_noop(lib):
    m, n, k = 0, 1024, 256
    ws = small_weights(n, k, 6)
    wi = ws.device_interleaved(lib)
    buf = torch.full((1 << 16,), 0x5A, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, k), dtype=torch.bfloat16, device="cuda")
    one = scalar(1.0)
    lib.nvfp4_quantize_gemm_swiglu_quant(x, one, buf, buf, wi[0], wi[1], one, one, buf, buf, m, n, k, None, 0)
    torch.cuda.synchronize()
    assert bool((buf == 0x5A).all()), "an M = 0 call wrote to its outputs"
