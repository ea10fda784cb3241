"""GPU parity of bf16_fp4_gemm_prescaled (W4A16 with the NVFP4_AWQ
activation pre-scale) against the oracle's awq_prescale + W4A16 GEMM.

Checks:
  * the standalone pre-scale pass, bit-exact against the oracle's bf16
    products (also in place);
  * an identity weight (code 1.0, scale 1.0 on the diagonal), so the GEMM
    returns the pre-scaled activations themselves: bit-exact against the
    oracle's bf16 products, which pins the rounding of x * s in the kernels;
  * random weights: relative Frobenius error <= 1e-3, at small shapes that
    span several tiles and ragged tails and at the full W4A16 shapes (sampled).
The GEMV scales as it loads; the tensor-core path runs the standalone pass
into the call's workspace first: both are covered.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, bf16_host, dev, sample_rows, scalar, small_weights, weights
from tolerance import assert_gemm_close

pytestmark = pytest.mark.gpu

GEMV, TC = 1, 2


def run_prescaled(nv, xbits, sbits, wdev, alpha, m, n, k, algo):
    d = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    nbytes = nv.bf16_fp4_gemm_prescaled_workspace_bytes(m, n, k, algo)
    # the scaled-activation part needs no initial contents; the split-K part
    # after it must start zero-filled
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    if nbytes:
        ws[:(m * k * 2 + 255) // 256 * 256].fill_(0x7F)
    x = bf16_dev(xbits)
    nv.bf16_fp4_gemm_prescaled(x, bf16_dev(sbits), wdev[0], wdev[1], scalar(alpha), d, m, n, k, ws, nbytes,
                               algo=algo)
    torch.cuda.synchronize()
    assert np.array_equal(x.view(torch.int16).cpu().numpy().view(np.uint16), xbits), "input modified"
    return bf16_host(d)


def identity_weight(nv, n):
    codes = np.zeros((n, n), dtype=np.uint8)
    codes[np.arange(n), np.arange(n)] = 2                 # E2M1 code 2 = 1.0
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sf = np.full((n, n // 16), 0x38, dtype=np.uint8)      # E4M3 0x38 = 1.0
    w = dev(packed)
    sfo = torch.empty(nv.nvfp4_sf_bytes(n, n), dtype=torch.uint8, device="cuda")
    nv.nvfp4_prepare_weights(w, dev(sf), n, n, w, sfo)
    return w, sfo


@pytest.mark.parametrize("m,k", [(1, 64), (37, 5120), (300, 192), (1024, 5120)])
def test_standalone_prescale_bit_exact(lib, m, k):
    xbits, x = synth.activations(4, m, k)
    sbits, s = synth.awq_pre_quant_scale(4, k)
    xd, sd = bf16_dev(xbits), bf16_dev(sbits)
    out = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.bf16_awq_prescale(xd, sd, out, m, k)
    lib.bf16_awq_prescale(xd, sd, xd, m, k)          # in place
    torch.cuda.synchronize()
    want = oracle.awq_prescale(x, s)
    assert np.array_equal(bf16_host(out), want)
    assert np.array_equal(bf16_host(xd), want)


@pytest.mark.parametrize("m,algo", [(1, GEMV), (7, GEMV), (1, TC), (16, TC), (45, TC), (64, TC), (65, TC),
                                    (200, TC)])
def test_prescale_rounding_bit_exact(lib, m, algo):
    k = 256
    xbits, x = synth.activations(4, m, k)
    sbits, s = synth.awq_pre_quant_scale(4, k)
    got = run_prescaled(lib, xbits, sbits, identity_weight(lib, k), np.float32(1.0), m, k, k, algo)
    want = oracle.awq_prescale(x, s)
    assert np.array_equal(got, want), f"{int((got != want).sum())} of {got.size} differ"


SHAPES_GEMV = [(1, 256, 512), (16, 1024, 256), (5, 96, 320)]
SHAPES_TC = [(1, 256, 512), (16, 1024, 256), (5, 96, 320), (33, 128, 128), (64, 384, 1024),
             (100, 256, 640), (300, 1024, 512)]


@pytest.mark.parametrize("m,n,k,algo", [(m, n, k, GEMV) for m, n, k in SHAPES_GEMV] +
                         [(m, n, k, TC) for m, n, k in SHAPES_TC])
def test_prescaled_small_shapes(lib, m, n, k, algo):
    ws = small_weights(n, k, 9)
    xbits, x = synth.activations(4, m, k)
    sbits, s = synth.awq_pre_quant_scale(4, k)
    alpha = np.float32(1.0) / ws.gs
    got = run_prescaled(lib, xbits, sbits, ws.device_prepared(lib), alpha, m, n, k, algo)
    ref = oracle.gemm_w4a16_prescaled(x, s, ws.packed, ws.sf, alpha)
    err = assert_gemm_close(got, ref)
    print(f"w4a16 awq algo={algo} m={m} n={n} k={k}: rel err {err:.2e}")


@pytest.mark.parametrize("m", [1, 16, 1024])
def test_prescaled_full_size_sampled(lib, m):
    ws = weights(4, "gate_up")
    xbits, x = synth.activations(4, m)
    sbits, s = synth.awq_pre_quant_scale(4)
    alpha = np.float32(1.0) / ws.gs
    got = run_prescaled(lib, xbits, sbits, ws.device_prepared(lib), alpha, m, ws.n, ws.k, TC)
    cols = sample_rows(ws.n, 512, seed=m + 5)
    toks = sample_rows(m, 128, seed=m + 6)
    ref = oracle.gemm_w4a16_prescaled(x[toks], s, ws.packed[cols], ws.sf[cols], alpha)
    err = assert_gemm_close(got[np.ix_(toks, cols)], ref)
    print(f"w4a16 awq gate_up m={m}: rel err {err:.2e}")


def test_prescaled_argument_errors(lib):
    m, n, k = 4, 256, 256
    ws = small_weights(n, k, 9)
    w, sfo = ws.device_prepared(lib)
    x = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    s = torch.ones(k + 8, dtype=torch.bfloat16, device="cuda")
    d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    a = scalar(1.0)
    with pytest.raises(lib.Nvfp4Error) as e:
        lib.bf16_fp4_gemm_prescaled(x, None, w, sfo, a, d, m, n, k)
    assert e.value.status == lib.ERR_INVALID_ARG
    with pytest.raises(lib.Nvfp4Error) as e:
        lib.bf16_fp4_gemm_prescaled(x, s[1:], w, sfo, a, d, m, n, k)   # 2-byte offset: not 16-byte aligned
    assert e.value.status == lib.ERR_UNSUPPORTED_SHAPE
    # on the tensor cores the call needs its workspace
    m2 = 65
    x2 = torch.zeros((m2, k), dtype=torch.bfloat16, device="cuda")
    d2 = torch.empty((m2, n), dtype=torch.bfloat16, device="cuda")
    need = lib.bf16_fp4_gemm_prescaled_workspace_bytes(m2, n, k, TC)
    xs_bytes = (m2 * k * 2 + 255) // 256 * 256           # the scaled activations come first
    assert need == xs_bytes + lib.bf16_fp4_gemm_workspace_bytes(m2, n, k, TC)
    small = torch.empty(xs_bytes - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.Nvfp4Error) as e:
        lib.bf16_fp4_gemm_prescaled(x2, s[:k], w, sfo, a, d2, m2, n, k, small, xs_bytes - 16, algo=TC)
    assert e.value.status == lib.ERR_INVALID_ARG
