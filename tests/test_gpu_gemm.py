"""GPU parity of the GEMM entry points against the CPU oracle.

Each stage runs on oracle-made inputs (activation codes and scales from the
oracle's quantize, weights quantized by the oracle and prepared by the
library's prep call), so a GEMM's result is compared with the oracle's result
for exactly the same operands:
  * bf16 outputs: relative Frobenius error <= 1e-3 against the float64 result
    rounded once to bf16;
  * fused SwiGLU outputs: the requantize tolerance of tests/tolerance.py.
Full-size workloads compare sampled output columns (whole 16-feature blocks
for the fused kernel), computed by the oracle one weight row at a time.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (bf16_dev, bf16_host, dev, host, quantized_activation, sample_rows, scalar,
                      small_weights, weights)
from tolerance import assert_gemm_close, check_requant

pytestmark = pytest.mark.gpu

GEMV, TC, TC_SWAPAB, TC_1SM = 1, 2, 3, 4


def workspace(nv, m, n, k, algo):
    """Zero-filled scratch of the size the library asks for (None if none)."""
    nbytes = nv.nvfp4_workspace_bytes(m, n, k, algo)
    return (torch.zeros(nbytes, dtype=torch.uint8, device="cuda"), nbytes) if nbytes else (None, 0)


def run_w4a4(nv, xq, xs, wdev, alpha, m, n, k, algo, ws=None):
    d = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    w, nbytes = ws if ws is not None else workspace(nv, m, n, k, algo)
    nv.nvfp4_gemm_ex(dev(xq), dev(oracle.sf_swizzle_128x4(xs)), wdev[0], wdev[1], scalar(alpha), d,
                     m, n, k, w, nbytes, algo=algo)
    torch.cuda.synchronize()
    return bf16_host(d)


def run_swiglu(nv, xq, xs, wdev, alpha, gs_h, m, n, k, algo):
    inter = n // 2
    q = torch.full((m, inter // 2), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((nv.nvfp4_sf_bytes(m, inter),), 0xAB, dtype=torch.uint8, device="cuda")
    w, nbytes = workspace(nv, m, n, k, algo)
    nv.nvfp4_gemm_swiglu_quant_ex(dev(xq), dev(oracle.sf_swizzle_128x4(xs)), wdev[0], wdev[1],
                                  scalar(alpha), scalar(gs_h), q, s, m, n, k, w, nbytes, algo=algo)
    torch.cuda.synchronize()
    s = host(s)
    lin = oracle.sf_unswizzle_128x4(s, m, inter // 16)
    assert np.array_equal(oracle.sf_swizzle_128x4(lin), s), "scale padding not zero"
    return host(q), lin


def run_w4a16(nv, xbits, wdev, alpha, m, n, k, algo, split=False):
    """split: pass the split-K workspace (tokens <= 64 then run split along K
    over all SMs; without it every SM owns whole weight tiles)."""
    d = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    nbytes = nv.bf16_fp4_gemm_workspace_bytes(m, n, k, algo) if split else 0
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda") if split else None
    x = bf16_dev(xbits)
    nv.bf16_fp4_gemm_ex(x, wdev[0], wdev[1], scalar(alpha), d, m, n, k, ws, nbytes, algo=algo)
    torch.cuda.synchronize()
    if split and nbytes:
        first = bf16_host(d)
        nv.bf16_fp4_gemm_ex(x, wdev[0], wdev[1], scalar(alpha), d, m, n, k, ws, nbytes, algo=algo)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(d), first), "second split call on the same workspace differs"
    return bf16_host(d)


# ---------------------------------------------------------------- W4A4 GEMM
SMALL_SHAPES = [(4, 1024, 256), (1, 256, 512), (3, 96, 320), (16, 512, 256), (17, 128, 128),
                (130, 160, 320)]
# tensor-core tiles are 128 x 256 x 256 per CTA (a CTA pair takes 256 x 256):
# cover exact tiles, an odd number of 128-row tiles (the pair's second CTA
# past M), ragged M / N / K tails, several k-blocks, a weight tile whose
# second 128-row half is past N, and more tiles than SMs (persistent loop)
TC_SHAPES = [(128, 256, 256), (1, 256, 256), (130, 160, 320), (256, 512, 1024), (200, 96, 576),
             (384, 1024, 2048), (1000, 2304, 512), (4096, 4096, 256), (640, 384, 1280), (257, 128, 64)]


# swap-AB (weights as the MMA M operand): tokens padded to 16/32/64, split-K;
# (1, 20480, 512) and (5, 39168, 768) have more weight tiles than SMs (whole
# tiles per CTA after the shared ones: 160 tiles of 2 k-blocks, 306 tiles of
# 3 k-blocks); (3, 2560, 2048) and (40, 6144, 1280) take the cluster split
# (one tile per cluster: 20 tiles x 7 CTAs, 48 x 3 with 64-token tiles)
SWAP_SHAPES = [(1, 256, 256), (4, 1024, 256), (3, 96, 320), (16, 512, 2048), (17, 128, 128),
               (33, 384, 1024), (64, 256, 512), (8, 2048, 8192), (1, 20480, 512), (5, 39168, 768),
               (3, 2560, 2048), (16, 4864, 512), (40, 6144, 1280)]


@pytest.mark.parametrize("m,n,k,algo", [(m, n, k, GEMV) for m, n, k in SMALL_SHAPES] +
                         [(m, n, k, TC) for m, n, k in TC_SHAPES] +
                         [(m, n, k, TC_1SM) for m, n, k in TC_SHAPES] +
                         [(m, n, k, TC_SWAPAB) for m, n, k in SWAP_SHAPES])
def test_w4a4_small_shapes(lib, m, n, k, algo):
    ws = small_weights(n, k, 3)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    got = run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, n, k, algo)
    ref = oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, alpha)
    err = assert_gemm_close(got, ref)
    print(f"w4a4 algo={algo} m={m} n={n} k={k}: rel err {err:.2e}")


@pytest.mark.parametrize("algo", [GEMV, TC_SWAPAB])
@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
def test_w4a4_decode_full_size_sampled(lib, m, which, algo):
    """Decode workload H5120/I17408: gate_up 34816x5120 and down 5120x17408."""
    ws = weights(1, which)
    k = ws.k
    if which == "gate_up":
        _, _, gs_x, xq, xs = quantized_activation(1, m)
    else:  # down_proj input: an NVFP4 h drawn by the oracle
        hf = synth.random_matrix((m, k), (21, m), scale=0.05)
        gs_x = oracle.global_scale(np.abs(hf).max())
        xq, xs = oracle.quantize_nvfp4(hf, gs_x)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    got = run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, ws.n, k, algo)
    cols = sample_rows(ws.n, 512, seed=m)
    ref = oracle.gemm_w4a4(xq, xs, ws.packed[cols], ws.sf[cols], alpha)
    err = assert_gemm_close(got[:, cols], ref)
    print(f"decode {which} m={m} algo={algo}: rel err {err:.2e}")


@pytest.mark.parametrize("algo", [GEMV, TC, TC_SWAPAB, TC_1SM])
def test_w4a4_is_deterministic(lib, algo):
    m, n, k = 16, 1024, 4096
    ws = small_weights(n, k, 4)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    scratch = workspace(lib, m, n, k, algo)
    a = run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, n, k, algo, scratch)
    b = run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, n, k, algo, scratch)
    assert np.array_equal(a, b)
    if scratch[0] is not None:   # split-K arrival counters are back at zero
        ntiles = (n + 127) // 128
        assert int(scratch[0][: 4 * ntiles].view(torch.int32).abs().sum()) == 0


def test_swapab_after_w4a16_on_a_shared_workspace(lib):
    """One buffer serves a W4A16 call and then swap-AB calls, as the header
    allows.  The W4A16 call leaves its fp32 partials and f16 activations
    where the swap-AB kernel keeps its partial tiles (16 tiles of 16 k-blocks
    over 128 CTAs: every tile shared by 16 CTAs); the swap-AB result must not
    depend on them, and a second call on the same buffer is identical."""
    m, n, k = 16, 1024, 4096
    ws = small_weights(n, k, 4)
    wdev = ws.device_prepared(lib)
    nbytes = max(lib.nvfp4_workspace_bytes(m, n, k, TC_SWAPAB), lib.bf16_fp4_gemm_workspace_bytes(m, n, k, TC))
    buf = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    xbits, _ = synth.activations(4, m, k)
    d16 = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    lib.bf16_fp4_gemm_ex(bf16_dev(xbits), wdev[0], wdev[1], scalar(1.0), d16, m, n, k, buf, nbytes, algo=TC)
    torch.cuda.synchronize()
    counter_area = 64 * 1024
    swap_need = lib.nvfp4_workspace_bytes(m, n, k, TC_SWAPAB)
    assert int(torch.count_nonzero(buf[counter_area:swap_need])) > 0, "no leftovers where the partials go"
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    first = run_w4a4(lib, xq, xs, wdev, alpha, m, n, k, TC_SWAPAB, (buf, nbytes))
    assert_gemm_close(first, oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, alpha))
    again = run_w4a4(lib, xq, xs, wdev, alpha, m, n, k, TC_SWAPAB, (buf, nbytes))
    assert np.array_equal(first, again)


# (1, 5120, 4096): 40 tiles of 16 k-blocks over 152 CTAs, runs crossing tiles
@pytest.mark.parametrize("m,n,k", [(16, 1024, 4096), (1, 5120, 4096)])
def test_swapab_bounded_wait_gives_up_cleanly(lib, m, n, k):
    """A wait limit of one poll makes the pipeline and partial-word waits
    run out: the kernel records NVFP4_ERR_DEVICE_TIMEOUT and returns; after
    the workspace is zero-filled again (as the header asks after a timeout)
    the next call on it is right."""
    ws = small_weights(n, k, 12)
    wdev = ws.device_prepared(lib)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    scratch = workspace(lib, m, n, k, TC_SWAPAB)
    assert scratch[0] is not None
    assert lib.nvfp4_get_device_status() == 0
    lib.nvfp4_set_wait_limit(1)
    try:
        run_w4a4(lib, xq, xs, wdev, alpha, m, n, k, TC_SWAPAB, scratch)
    finally:
        lib.nvfp4_set_wait_limit(0)
    assert lib.nvfp4_get_device_status() == lib.ERR_DEVICE_TIMEOUT
    scratch[0].zero_()
    got = run_w4a4(lib, xq, xs, wdev, alpha, m, n, k, TC_SWAPAB, scratch)
    assert lib.nvfp4_get_device_status() == 0
    assert_gemm_close(got, oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, alpha))


def test_swapab_without_workspace_still_correct(lib):
    """Too little scratch: the kernel runs one unit per weight tile instead."""
    m, n, k = 4, 512, 4096
    ws = small_weights(n, k, 11)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    got = run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, n, k, TC_SWAPAB, (None, 0))
    assert_gemm_close(got, oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, alpha))


def test_gemm_m_zero_is_a_noop(lib):
    ws = small_weights(256, 256, 5)
    w = ws.device_prepared(lib)
    d = torch.full((1, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    a = torch.zeros((1, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((512,), dtype=torch.uint8, device="cuda")
    lib.nvfp4_gemm(a, s, w[0], w[1], scalar(1.0), d, 0, 256, 256)
    torch.cuda.synchronize()
    assert float(d.float().min()) == 3.0


# ------------------------------------------------------- fused gate_up SwiGLU
def _swiglu_case(nv, wid, m, n, k, ws, algo, sampled_blocks=None, sampled_tokens=None):
    inter = n // 2
    _, _, gs_x, xq, xs = quantized_activation(wid, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    feats = np.arange(inter) if sampled_blocks is None else \
        sample_rows(inter, sampled_blocks, seed=m + 7, block=16)
    toks = np.arange(m) if sampled_tokens is None else sample_rows(m, sampled_tokens, seed=m + 9)
    rows = np.concatenate([feats, inter + feats])           # gate rows, then up rows
    d = oracle.gemm_w4a4(xq[toks], xs[toks], ws.packed[rows], ws.sf[rows], alpha, round_bf16=False)
    h = oracle.swiglu_h(d)
    gs_h = oracle.global_scale(np.abs(h).max())
    q, s = run_swiglu(nv, xq, xs, ws.device_interleaved(nv), alpha, gs_h, m, n, k, algo)
    codes = oracle.unpack_codes(q[toks])[:, feats]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    nflip, nsf = check_requant(packed, s[toks][:, feats[::16] // 16], h, gs_h, what=f"swiglu m={m}")
    print(f"swiglu algo={algo} m={m} n={n} k={k}: {nflip} boundary flips, {nsf} scale diffs")


SWIGLU_GEMV = [(4, 1024, 256), (1, 256, 512), (3, 128, 320), (16, 384, 256), (130, 256, 128)]
SWIGLU_TC = [(128, 256, 256), (4, 1024, 256), (130, 384, 320), (256, 1024, 1024), (700, 2304, 512),
             (384, 640, 1280)]


# (33, 3072, 2048) takes the cluster split (24 tiles x 6 CTAs)
SWIGLU_SWAP = [(1, 256, 256), (4, 1024, 256), (3, 128, 320), (16, 384, 4096), (40, 256, 512),
               (64, 1024, 1024), (16, 4096, 1024), (33, 3072, 2048)]


@pytest.mark.parametrize("m,n,k,algo", [(m, n, k, GEMV) for m, n, k in SWIGLU_GEMV] +
                         [(m, n, k, TC) for m, n, k in SWIGLU_TC] +
                         [(m, n, k, TC_1SM) for m, n, k in SWIGLU_TC] +
                         [(m, n, k, TC_SWAPAB) for m, n, k in SWIGLU_SWAP])
def test_swiglu_small_shapes(lib, m, n, k, algo):
    _swiglu_case(lib, 0, m, n, k, small_weights(n, k, 6), algo)


@pytest.mark.parametrize("algo", [GEMV, TC_SWAPAB])
@pytest.mark.parametrize("m", [1, 8, 32, 64])
def test_swiglu_deepseek_decode_full_size_sampled(lib, m, algo):
    """DeepSeek-V3-shaped decode, x with 1% outliers x20, interleaved
    36864x7168 gate_up weight; 288 stratified 16-feature blocks, one in each
    64-feature (128-row) weight tile."""
    ws = weights(2, "gate_up")
    _swiglu_case(lib, 2, m, ws.n, ws.k, ws, algo, sampled_blocks=288)


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
def test_swiglu_decode_h5120_full_size_sampled(lib, m):
    """The bench's decode step: fused gate_up + SwiGLU + requant on the
    interleaved 34816x5120 weight (H5120/I17408) in the swap-AB launch the
    bench times (NT = 16, mixed split-K over all SMs); 272 stratified
    16-feature blocks, one in each 64-feature (128-row) weight tile."""
    ws = weights(1, "gate_up")
    _swiglu_case(lib, 1, m, ws.n, ws.k, ws, TC_SWAPAB, sampled_blocks=272)


@pytest.mark.parametrize("m", [1, 64])
def test_w4a4_deepseek_down_full_size_sampled(lib, m):
    """DeepSeek-V3-shaped decode down_proj 7168 x 18432 (56 weight tiles, all
    shared by CTAs along K) on an oracle-made NVFP4 h, in the launch the
    decode chain uses; 512 sampled output columns."""
    ws = weights(2, "down")
    hf = synth.random_matrix((m, ws.k), (22, m), scale=0.05)
    gs_x = oracle.global_scale(np.abs(hf).max())
    xq, xs = oracle.quantize_nvfp4(hf, gs_x)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    got = run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, ws.n, ws.k, 0)
    cols = sample_rows(ws.n, 512, seed=m)
    err = assert_gemm_close(got[:, cols], oracle.gemm_w4a4(xq, xs, ws.packed[cols], ws.sf[cols], alpha))
    print(f"deepseek down m={m}: rel err {err:.2e}")


@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("m", [1, 16])
def test_w4a4_decode_full_size_sampled_tc(lib, m, which):
    """The same decode shapes forced onto the 128-token-tile kernel (the
    bench's --algo tc)."""
    test_w4a4_decode_full_size_sampled(lib, m, which, TC)


@pytest.mark.parametrize("m,algo", [(1024, 0), (4096, 0), (8192, 0), (1024, TC_1SM)])
def test_swiglu_prefill_full_size_sampled(lib, m, algo):
    """Prefill H7168/I18432, M up to 8192, the launch the prefill chain uses
    (AUTO: CTA pairs with 2-SM MMAs): 256 stratified tokens x 144 stratified
    16-feature blocks (one in each 128-feature span of the 256-row weight
    tiles)."""
    ws = weights(3, "gate_up")
    _swiglu_case(lib, 3, m, ws.n, ws.k, ws, algo, sampled_blocks=144, sampled_tokens=256)


@pytest.mark.parametrize("m", [1024, 8192])
def test_down_prefill_full_size_sampled(lib, m):
    """Prefill down_proj 7168 x 18432 on an oracle-made NVFP4 h: 256 sampled
    tokens x 512 sampled output columns."""
    ws = weights(3, "down")
    hf = synth.random_matrix((m, ws.k), (24, m), scale=0.05)
    gs_h = oracle.global_scale(np.abs(hf).max())
    hq, hs = quantize_rows(hf, gs_h)
    alpha = np.float32(1.0) / (gs_h * ws.gs)
    got = run_w4a4(lib, hq, hs, ws.device_prepared(lib), alpha, m, ws.n, ws.k, 0)
    toks, cols = sample_rows(m, 256, seed=5), sample_rows(ws.n, 512, seed=6)
    ref = oracle.gemm_w4a4(hq[toks], hs[toks], ws.packed[cols], ws.sf[cols], alpha)
    err = assert_gemm_close(got[np.ix_(toks, cols)], ref)
    print(f"prefill down m={m}: rel err {err:.2e}")


def quantize_rows(x, gs):
    from gpu_util import quantize_big
    return quantize_big(x, gs)


@pytest.mark.parametrize("algo", [TC, TC_1SM])
def test_tc_bounded_wait_gives_up_cleanly(lib, algo):
    """A wait limit of one poll makes the pipeline waits run out: the kernel
    must record NVFP4_ERR_DEVICE_TIMEOUT and return, leaving the context
    usable for the next (normal) call."""
    m, n, k = 256, 512, 1024
    ws = small_weights(n, k, 9)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    assert lib.nvfp4_get_device_status() == 0
    lib.nvfp4_set_wait_limit(1)
    try:
        run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, n, k, algo)
    finally:
        lib.nvfp4_set_wait_limit(0)
    assert lib.nvfp4_get_device_status() == lib.ERR_DEVICE_TIMEOUT
    assert lib.nvfp4_get_device_status() == 0          # read clears it
    got = run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, n, k, algo)
    assert_gemm_close(got, oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, alpha))


@pytest.mark.parametrize("algo", [TC, TC_1SM])
def test_tc_swiglu_bounded_wait_gives_up_cleanly(lib, algo):
    """The fused gate_up instance with a wait limit of one poll: the scale
    writers and the MMA thread give up at their first waits, so the operand
    stages' full barriers (which count the writers' arrivals) never complete
    and the drain's own bounded waits run out; the kernel records
    NVFP4_ERR_DEVICE_TIMEOUT and returns, and the next normal call on the
    same weights passes the requantize rule."""
    m, n, k = 256, 1024, 1024
    inter = n // 2
    ws = small_weights(n, k, 6)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    wdev = ws.device_interleaved(lib)
    q = torch.zeros((m, inter // 2), dtype=torch.uint8, device="cuda")
    s = torch.zeros((lib.nvfp4_sf_bytes(m, inter),), dtype=torch.uint8, device="cuda")
    w, nbytes = workspace(lib, m, n, k, algo)
    assert lib.nvfp4_get_device_status() == 0
    lib.nvfp4_set_wait_limit(1)
    try:
        lib.nvfp4_gemm_swiglu_quant_ex(dev(xq), dev(oracle.sf_swizzle_128x4(xs)), wdev[0], wdev[1], scalar(alpha),
                                       scalar(1.0), q, s, m, n, k, w, nbytes, algo=algo)
        torch.cuda.synchronize()
    finally:
        lib.nvfp4_set_wait_limit(0)
    assert lib.nvfp4_get_device_status() == lib.ERR_DEVICE_TIMEOUT
    assert lib.nvfp4_get_device_status() == 0          # read clears it
    _swiglu_case(lib, 0, m, n, k, ws, algo)


def test_auto_dispatch_matches_forced_paths(lib):
    """AUTO picks GEMV for decode-sized M and the tensor cores above; both
    give the same result within tolerance at the crossover."""
    n, k = 512, 512
    ws = small_weights(n, k, 10)
    for m in (16, 17, 64, 65):
        _, _, gs_x, xq, xs = quantized_activation(0, m, k)
        alpha = np.float32(1.0) / (gs_x * ws.gs)
        ref = oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, alpha)
        for algo in (0, GEMV, TC) + ((TC_SWAPAB,) if m <= 64 else ()):
            assert_gemm_close(run_w4a4(lib, xq, xs, ws.device_prepared(lib), alpha, m, n, k, algo), ref)


# ------------------------------------------------------------------- W4A16
W4A16_GEMV = [(1, 256, 512), (16, 1024, 256), (5, 96, 320), (33, 128, 128)]
# tensor cores: token tiles of 16/32/64/128/256, ragged tokens, N and K tails
W4A16_TC = [(1, 256, 512), (16, 1024, 256), (5, 96, 320), (33, 128, 128), (64, 384, 1024),
            (100, 256, 640), (128, 512, 2048), (300, 1024, 512), (1024, 2048, 1024)]


@pytest.mark.parametrize("m,n,k,algo", [(m, n, k, GEMV) for m, n, k in W4A16_GEMV] +
                         [(m, n, k, TC) for m, n, k in W4A16_TC])
def test_w4a16_small_shapes(lib, m, n, k, algo):
    ws = small_weights(n, k, 8)
    xbits, x = synth.activations(4, m, k)
    alpha = np.float32(1.0) / ws.gs
    got = run_w4a16(lib, xbits, ws.device_prepared(lib), alpha, m, n, k, algo)
    ref = oracle.gemm_w4a16(x, ws.packed, ws.sf, alpha)
    err = assert_gemm_close(got, ref)
    print(f"w4a16 algo={algo} m={m} n={n} k={k}: rel err {err:.2e}")


# split-K along K (workspace given): tiles shared by 2..5 CTAs, ragged tails;
# the last three are 128- and 256-token tiles with too few weight tiles for
# whole tiles per CTA (128- and 256-token tiles, several token tiles)
W4A16_SPLIT = [(1, 256, 512), (5, 96, 320), (16, 1024, 256), (33, 128, 1024), (64, 384, 2048),
               (16, 2048, 4096), (3, 160, 640), (100, 640, 2048), (128, 1024, 1024), (300, 768, 512)]


@pytest.mark.parametrize("m,n,k", W4A16_SPLIT)
def test_w4a16_split_k_small_shapes(lib, m, n, k):
    ws = small_weights(n, k, 8)
    xbits, x = synth.activations(4, m, k)
    alpha = np.float32(1.0) / ws.gs
    assert lib.bf16_fp4_gemm_workspace_bytes(m, n, k, TC) > 0      # tiles really are shared
    got = run_w4a16(lib, xbits, ws.device_prepared(lib), alpha, m, n, k, TC, split=True)
    ref = oracle.gemm_w4a16(x, ws.packed, ws.sf, alpha)
    err = assert_gemm_close(got, ref)
    print(f"w4a16 split m={m} n={n} k={k}: rel err {err:.2e}")


@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("m,algo,split", [(1, GEMV, False), (16, GEMV, False), (1, TC, False), (16, TC, False),
                                          (1, TC, True), (16, TC, True), (64, TC, True), (128, TC, False),
                                          (1024, TC, False), (128, TC, True), (1024, TC, True)])
def test_w4a16_full_size_sampled(lib, m, which, algo, split):
    ws = weights(4, which)
    if which == "gate_up":
        xbits, x = synth.activations(4, m)
    else:
        xbits, x = synth.to_bf16_bits(synth.random_matrix((m, ws.k), (23, m), scale=0.1))
    alpha = np.float32(1.0) / ws.gs
    got = run_w4a16(lib, xbits, ws.device_prepared(lib), alpha, m, ws.n, ws.k, algo, split)
    cols = sample_rows(ws.n, 512, seed=m + 3)
    toks = sample_rows(m, 128, seed=m + 4)
    ref = oracle.gemm_w4a16(x[toks], ws.packed[cols], ws.sf[cols], alpha)
    err = assert_gemm_close(got[np.ix_(toks, cols)], ref)
    print(f"w4a16 {which} m={m} algo={algo}: rel err {err:.2e}")


# ------------------------------------------------------------- whole chains
def test_tiny_mlp_chain_end_to_end(lib):
    """H256/I512, M=4: quantize -> fused gate_up -> down, all on the GPU,
    against the oracle's own chain (one tolerance for the end-to-end error,
    since requant boundary flips may propagate)."""
    m = 4
    xbits, x = synth.activations(0, m)
    wgu, wdn = weights(0, "gate_up"), weights(0, "down")
    gs_x = oracle.global_scale(np.abs(x).max())
    a_gu = np.float32(1.0) / (gs_x * wgu.gs)
    xq, xs = oracle.quantize_nvfp4(x, gs_x)
    h = oracle.swiglu_h(oracle.gemm_w4a4(xq, xs, wgu.packed, wgu.sf, a_gu, round_bf16=False))
    gs_h = oracle.global_scale(np.abs(h).max())
    a_dn = np.float32(1.0) / (gs_h * wdn.gs)
    ref = oracle.mlp_w4a4_fused(x, gs_x, (wgu.packed, wgu.sf), a_gu, gs_h, (wdn.packed, wdn.sf), a_dn)

    h_, i_ = 256, 512
    xq_d = torch.empty((m, h_ // 2), dtype=torch.uint8, device="cuda")
    xs_d = torch.empty((lib.nvfp4_sf_bytes(m, h_),), dtype=torch.uint8, device="cuda")
    lib.nvfp4_quantize(bf16_dev(xbits), m, h_, scalar(gs_x), xq_d, xs_d)
    hq_d = torch.empty((m, i_ // 2), dtype=torch.uint8, device="cuda")
    hs_d = torch.empty((lib.nvfp4_sf_bytes(m, i_),), dtype=torch.uint8, device="cuda")
    wi = wgu.device_interleaved(lib)
    w1, n1 = workspace(lib, m, 2 * i_, h_, 0)
    lib.nvfp4_gemm_swiglu_quant(xq_d, xs_d, wi[0], wi[1], scalar(a_gu), scalar(gs_h), hq_d, hs_d,
                                m, 2 * i_, h_, w1, n1)
    out = torch.empty((m, h_), dtype=torch.bfloat16, device="cuda")
    wd = wdn.device_prepared(lib)
    w2, n2 = workspace(lib, m, h_, i_, 0)
    lib.nvfp4_gemm(hq_d, hs_d, wd[0], wd[1], scalar(a_dn), out, m, h_, i_, w2, n2)
    torch.cuda.synchronize()
    err = assert_gemm_close(bf16_host(out), ref, tol=5e-3, what="tiny MLP end to end")
    print(f"tiny MLP end-to-end rel err {err:.2e}")
