"""GPU checks of what is particular to the W4A16 TMEM kernel (workspace
given; 16/32/64-token tiles of 256-wide k-blocks, 128-token tiles of 128-wide
k-blocks): the f16 activation pre-pass with its power-of-two scale 2^e per
token row, undone by the epilogue.

* Identity weight (E2M1 code 1.0 times scale 1.0 on the diagonal): the GEMM
  returns the activations themselves, so the output must equal x bit for bit
  whenever every element of a row lies within 2^30 of the row's largest
  magnitude -- rows at magnitudes from 2^-120 to 2^120, an all-zero row, a row
  of bf16 subnormals, a row holding the largest bf16 value.  A wrong e, a
  wrong or missing 2^-e, or an inexact f16 conversion changes bits here.
* A row whose elements spread over more than 2^30: the small elements become
  f16 subnormals, rounded by at most 2^-25 in the scaled units, i.e.
  2^-(25+e) in the activation's own units.
* Random NVFP4 weights, token rows at magnitudes 2^-100 .. 2^100: every
  row's relative error against the oracle within the GEMM tolerance (one
  norm over all rows would hide the small ones).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, bf16_host, dev, scalar, small_weights
from tolerance import assert_gemm_close

pytestmark = pytest.mark.gpu

TC = 2


def identity_weight(nv, n):
    codes = np.zeros((n, n), dtype=np.uint8)
    codes[np.arange(n), np.arange(n)] = 2                 # E2M1 code 2 = 1.0
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sf = np.full((n, n // 16), 0x38, dtype=np.uint8)      # E4M3 0x38 = 1.0
    w = dev(packed)
    sfo = torch.empty(nv.nvfp4_sf_bytes(n, n), dtype=torch.uint8, device="cuda")
    nv.nvfp4_prepare_weights(w, dev(sf), n, n, w, sfo)
    return w, sfo


def run_tmem(nv, xbits, w, sfo, alpha, m, n, k):
    nbytes = nv.bf16_fp4_gemm_workspace_bytes(m, n, k, TC)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ws[64 * 1024:].fill_(0x7F)        # only the counter area needs zeros
    d = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.bf16_fp4_gemm_ex(bf16_dev(xbits), w, sfo, scalar(alpha), d, m, n, k, ws, nbytes, algo=TC)
    torch.cuda.synchronize()
    return bf16_host(d)


def bf16_bits(v):
    """float64 values that are bf16 -> their bit patterns."""
    f = np.asarray(v, dtype=np.float32).view(np.uint32)
    assert np.all((f & 0xFFFF) == 0)
    return (f >> 16).astype(np.uint16)


def rows_in_range(m, k, seed):
    """Row t: random signs and significands, magnitudes 2^(s_t - 20) ..
    2^s_t (within 2^30 of the row maximum), s_t from -120 to 120; special
    rows: all zeros, bf16 subnormals, the bf16 maximum."""
    g = np.random.default_rng(seed)
    scales = np.array([-120, -60, -20, 0, 7, 20, 60, 120])
    x = np.zeros((m, k))
    for t in range(m):
        s = scales[t % len(scales)]
        mant = g.integers(128, 256, size=k) / 128.0               # 8 significant bits
        x[t] = g.choice([-1.0, 1.0], size=k) * mant * np.exp2(s + g.integers(-20, 0, size=k))
    if m > 2:
        x[1] = 0.0
        x[2] = g.choice([-1.0, 1.0], size=k) * g.integers(1, 128, size=k) * 2.0 ** -133   # subnormals
    if m > 3:
        x[3, :] = np.exp2(g.integers(100, 128, size=k)) * (g.integers(128, 256, size=k) / 128.0)
        x[3, 5 % k] = float(np.frombuffer(np.uint32(0x7F7F0000).tobytes(), dtype=np.float32)[0])
    return oracle.bf16_round(x) + 0.0        # no negative zeros


@pytest.mark.parametrize("m,n", [(1, 256), (7, 256), (16, 320), (33, 1024), (64, 512), (130, 256), (300, 384)])
def test_identity_weight_returns_activations_bit_exact(lib, m, n):
    x = rows_in_range(m, n, seed=m)
    w, sfo = identity_weight(lib, n)
    got = run_tmem(lib, bf16_bits(x), w, sfo, np.float32(1.0), m, n, n)
    want = bf16_bits(x)
    gotb = bf16_bits(got)
    bad = np.argwhere(gotb != want)
    assert bad.size == 0, f"{len(bad)} differ, first at {bad[:4].tolist()}: got {got[tuple(bad[0])]}, want {x[tuple(bad[0])]}"


def test_wide_row_rounds_small_elements_within_bound(lib):
    m, n = 2, 256
    g = np.random.default_rng(5)
    x = np.zeros((m, n))
    x[0] = g.choice([-1.0, 1.0], size=n) * np.exp2(g.integers(-50, 1, size=n)) * (g.integers(128, 256, size=n) / 128)
    x[0, 0] = 3.0                                   # row max in [2, 4): e = 14
    x[1] = x[0] * 2.0 ** -90                        # the same pattern 2^90 smaller: e = 104
    x = oracle.bf16_round(x) + 0.0
    w, sfo = identity_weight(lib, n)
    got = run_tmem(lib, bf16_bits(x), w, sfo, np.float32(1.0), m, n, n)
    for t, e in ((0, 14), (1, 104)):
        err = np.abs(got[t] - x[t])
        bound = 2.0 ** -(24 + e) + np.abs(x[t]) * 2.0 ** -7     # f16 subnormal step + the bf16 output rounding
        assert np.all(err <= bound), f"row {t}: {int((err > bound).sum())} elements past the bound"
        big = np.abs(x[t]) >= 3.0 * 2.0 ** -30
        assert np.array_equal(got[t][big], x[t][big]), "elements within 2^30 of the row max are exact"


@pytest.mark.parametrize("m,n,k", [(1, 384, 1024), (16, 1024, 2048), (40, 256, 640), (64, 512, 512),
                                   (200, 512, 704), (129, 256, 1024)])
def test_rows_at_extreme_magnitudes_each_within_tolerance(lib, m, n, k):
    ws = small_weights(n, k, 10)
    xbits, x = synth.activations(4, m, k)
    scale = np.exp2(np.array([-100, -40, 0, 40, 100])[np.arange(m) % 5]).reshape(-1, 1)
    x = oracle.bf16_round(x * scale)
    alpha = np.float32(1.0) / ws.gs
    wd = ws.device_prepared(lib)
    got = run_tmem(lib, bf16_bits(x), wd[0], wd[1], alpha, m, n, k)
    ref = oracle.gemm_w4a16(x, ws.packed, ws.sf, alpha)
    for t in range(m):
        assert_gemm_close(got[t:t + 1], ref[t:t + 1], what=f"token row {t} (scale 2^{int(np.log2(scale[t, 0]))})")


@pytest.mark.parametrize("m,n,k", [(16, 1024, 2048), (200, 512, 1024)])
def test_bounded_wait_gives_up_cleanly(lib, m, n, k):
    """A wait limit of one poll makes the pipeline waits run out (one CTA per
    tile at 16 tokens, CTA pairs at 200): the kernel records
    NVFP4_ERR_DEVICE_TIMEOUT and returns, and the next call on a fresh
    workspace is correct."""
    ws = small_weights(n, k, 11)
    xbits, x = synth.activations(4, m, k)
    alpha = np.float32(1.0) / ws.gs
    wd = ws.device_prepared(lib)
    assert lib.nvfp4_get_device_status() == 0
    lib.nvfp4_set_wait_limit(1)
    try:
        run_tmem(lib, xbits, wd[0], wd[1], alpha, m, n, k)
    finally:
        lib.nvfp4_set_wait_limit(0)
    assert lib.nvfp4_get_device_status() == lib.ERR_DEVICE_TIMEOUT
    assert lib.nvfp4_get_device_status() == 0          # read clears it
    got = run_tmem(lib, xbits, wd[0], wd[1], alpha, m, n, k)
    assert_gemm_close(got, oracle.gemm_w4a16(x, ws.packed, ws.sf, alpha))


# 128-token tiles on CTA pairs, every weight tile shared: 2 pair tiles of 32
# k-blocks (32 contributors each), token tiles of one pair tile split over
# 68 k-blocks (~38 contributors), two token tiles with a ragged second one
@pytest.mark.parametrize("m,n,k", [(128, 512, 8192), (130, 256, 17408), (256, 768, 2048), (200, 512, 3072)])
def test_split_128_token_tiles(lib, m, n, k):
    """Tiles of 128 token rows shared by many CTA pairs: the last to arrive
    sums every contributor's 128-token partial in K order.  The result
    matches the oracle, a second call on the same workspace is bit for bit
    the first, and every counter is back at zero afterwards."""
    ws = small_weights(n, k, 16)
    xbits, x = synth.activations(4, m, k)
    alpha = np.float32(1.0) / ws.gs
    w, sfo = ws.device_prepared(lib)
    nbytes = lib.bf16_fp4_gemm_workspace_bytes(m, n, k, TC)
    scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        d = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        lib.bf16_fp4_gemm_ex(bf16_dev(xbits), w, sfo, scalar(alpha), d, m, n, k, scratch, nbytes, algo=TC)
        torch.cuda.synchronize()
        outs.append(bf16_host(d))
        assert int(torch.count_nonzero(scratch[:64 * 1024])) == 0, "counters not reset"
    assert np.array_equal(outs[0], outs[1])
    assert_gemm_close(outs[0], oracle.gemm_w4a16(x, ws.packed, ws.sf, alpha))
