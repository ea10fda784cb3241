"""Per-token dynamic activation scales (one global scale per row): quantize
bit-exact against the oracle, and the GEMMs that fold the per-row dequant
factor into their epilogues, on every kernel family."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, bf16_host, dev, host, scalar, small_weights
from tolerance import assert_gemm_close, check_requant

pytestmark = pytest.mark.gpu

GEMV, TC, TC_SWAPAB = 1, 2, 3


def _x(m, k, seed):
    """Rows with magnitudes spread over six decades, plus one all-zero row."""
    g = synth.random_matrix((m, k), (51, m, k, seed))
    scale = np.power(10.0, np.linspace(-3, 3, m)).astype(np.float32)[:, None]
    x = (g * scale).astype(np.float32)
    if m > 2:
        x[m // 2] = 0.0
    return synth.to_bf16_bits(x)


@pytest.mark.parametrize("layout", [0, 1], ids=["swizzled", "linear"])
@pytest.mark.parametrize("m,k", [(1, 256), (7, 320), (130, 512), (64, 7168)])
def test_quantize_per_token_bit_exact(lib, m, k, layout):
    bits, x = _x(m, k, 0)
    ref_q, ref_s, ref_rs = oracle.quantize_nvfp4_per_token(x)
    q = torch.empty((m, k // 2), dtype=torch.uint8, device="cuda")
    s = torch.full((lib.nvfp4_sf_bytes(m, k, layout),), 0xAB, dtype=torch.uint8, device="cuda")
    rs = torch.empty((m,), dtype=torch.float32, device="cuda")
    lib.nvfp4_quantize_per_token(bf16_dev(bits), m, k, q, s, layout, rs)
    torch.cuda.synchronize()
    assert np.array_equal(host(q), ref_q)
    if layout == 0:
        assert np.array_equal(host(s), oracle.sf_swizzle_128x4(ref_s))
    else:
        assert np.array_equal(host(s).reshape(m, k // 16), ref_s)
    assert np.array_equal(host(rs), ref_rs)


def _operands(m, n, k, seed):
    bits, x = _x(m, k, seed)
    xq, xs, rs = oracle.quantize_nvfp4_per_token(x)
    ws = small_weights(n, k, 60 + seed)
    return xq, xs, rs, ws


def _scratch(lib, m, n, k, algo):
    nb = lib.nvfp4_workspace_bytes(m, n, k, algo)
    return (torch.zeros(nb, dtype=torch.uint8, device="cuda"), nb) if nb else (None, 0)


@pytest.mark.parametrize("m,n,k,algo", [(4, 512, 512, GEMV), (16, 256, 1024, TC_SWAPAB), (3, 96, 320, TC_SWAPAB),
                                        (200, 512, 1024, TC), (130, 160, 320, TC)])
def test_gemm_per_token(lib, m, n, k, algo):
    xq, xs, rs, ws = _operands(m, n, k, 1)
    alpha = np.float32(1.0) / ws.gs
    w = ws.device_prepared(lib)
    d = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    scr, nb = _scratch(lib, m, n, k, algo)
    lib.nvfp4_gemm_per_token(dev(xq), dev(oracle.sf_swizzle_128x4(xs)), dev(rs), w[0], w[1], scalar(alpha), d,
                             m, n, k, scr, nb, algo=algo)
    torch.cuda.synchronize()
    ref = oracle.gemm_w4a4_per_token(xq, xs, rs, ws.packed, ws.sf, alpha)
    err = assert_gemm_close(bf16_host(d), ref)
    print(f"per-token gemm algo={algo} m={m}: rel err {err:.2e}")


@pytest.mark.parametrize("m,n,k,algo", [(4, 1024, 256, GEMV), (16, 512, 1024, TC_SWAPAB), (130, 384, 320, TC)])
def test_swiglu_per_token(lib, m, n, k, algo):
    xq, xs, rs, ws = _operands(m, n, k, 2)
    alpha = np.float32(1.0) / ws.gs
    d = oracle.gemm_w4a4_per_token(xq, xs, rs, ws.packed, ws.sf, alpha, round_bf16=False)
    h = oracle.swiglu_h(d)
    gs_h = oracle.global_scale(np.abs(h).max())
    wi = ws.device_interleaved(lib)
    inter = n // 2
    q = torch.full((m, inter // 2), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((lib.nvfp4_sf_bytes(m, inter),), 0xAB, dtype=torch.uint8, device="cuda")
    scr, nb = _scratch(lib, m, n, k, algo)
    lib.nvfp4_gemm_swiglu_quant_per_token(dev(xq), dev(oracle.sf_swizzle_128x4(xs)), dev(rs), wi[0], wi[1],
                                          scalar(alpha), scalar(gs_h), q, s, m, n, k, scr, nb, algo=algo)
    torch.cuda.synchronize()
    lin = oracle.sf_unswizzle_128x4(host(s), m, inter // 16)
    nflip, nsf = check_requant(host(q), lin, h, gs_h, what=f"per-token swiglu algo={algo}")
    print(f"per-token swiglu algo={algo} m={m}: {nflip} flips, {nsf} scale diffs")
