"""GPU parity of nvfp4_mlp_decode (the whole decode MLP in one kernel)
against the oracle's chain on the same seeded inputs.

Per call three results are checked:
  * the quantized x: bit-exact against oracle.quantize_nvfp4 (codes and the
    swizzled scales, padding rows zero);
  * h: the requantize tolerance of tests/tolerance.py against the oracle's
    pre-quantization h (gate_up rounded to bf16 first when
    round_gate_up_bf16 is set, as the unfused chain does);
  * the bf16 output, as a GEMM stage: every token row whose requantized h
    (codes and scale bytes) is bit-identical to the oracle's gives the
    kernel's down_proj exactly the oracle's input, so those rows are held to
    the GEMM tolerance (1e-3 relative Frobenius) against the oracle's chain;
  * the bf16 output end to end: all rows against the oracle's chain with one
    end-to-end tolerance (a requantize boundary flip in h moves that row's
    output a little).
Shapes span several weight tiles, split-K tiles shared by up to four CTAs,
ragged K tails, the 16/32/64 token tiles, and the two full decode workloads.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, bf16_host, host, scalar, small_weights, weights
from tolerance import assert_gemm_close, check_requant

pytestmark = pytest.mark.gpu

E2E_TOL = 5e-3


def oracle_gemm(aq, asf, ws, alpha, round_bf16, chunk=4096):
    """oracle.gemm_w4a4 over the weight rows in blocks (bounded host memory)."""
    parts = [oracle.gemm_w4a4(aq, asf, ws.packed[r:r + chunk], ws.sf[r:r + chunk], alpha, round_bf16=round_bf16)
             for r in range(0, ws.n, chunk)]
    return np.concatenate(parts, axis=1)


def oracle_chain(x, wgu, wdn, round_bf16):
    gs_x = oracle.global_scale(np.abs(x).max())
    xq, xs = oracle.quantize_nvfp4(x, gs_x)
    a_gu = np.float32(1.0) / (gs_x * wgu.gs)
    gate_up = oracle_gemm(xq, xs, wgu, a_gu, round_bf16)
    h = oracle.swiglu_h(gate_up)
    gs_h = oracle.global_scale(np.abs(h).max())
    hq, hs = oracle.quantize_nvfp4(h, gs_h)
    a_dn = np.float32(1.0) / (gs_h * wdn.gs)
    out = oracle_gemm(hq, hs, wdn, a_dn, True)
    return dict(gs_x=gs_x, xq=xq, xs=xs, a_gu=a_gu, h=h, hq=hq, hs=hs, gs_h=gs_h, a_dn=a_dn, out=out)


def run_fused(nv, xbits, m, hid, inter, wgu, wdn, ref, round_bf16):
    xq = torch.full((m, hid // 2), 0xAB, dtype=torch.uint8, device="cuda")
    xs = torch.full((nv.nvfp4_sf_bytes(m, hid),), 0xAB, dtype=torch.uint8, device="cuda")
    hq = torch.full((m, inter // 2), 0xAB, dtype=torch.uint8, device="cuda")
    hs = torch.full((nv.nvfp4_sf_bytes(m, inter),), 0xAB, dtype=torch.uint8, device="cuda")
    out = torch.full((m, hid), float("nan"), dtype=torch.bfloat16, device="cuda")
    nbytes = nv.nvfp4_mlp_decode_workspace_bytes(m, hid, inter)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    wi, wd = wgu.device_interleaved(nv), wdn.device_prepared(nv)
    args = [bf16_dev(xbits), scalar(ref["gs_x"]), wi[0], wi[1], scalar(ref["a_gu"]), scalar(ref["gs_h"]),
            wd[0], wd[1], scalar(ref["a_dn"]), xq, xs, hq, hs, out, m, hid, inter, round_bf16, ws, nbytes]
    # first a call on other activations, then the checked call on the same
    # workspace: stale counters left by the first call would let the second
    # read h before it is written.  The checked call must also match a call
    # on a fresh workspace bit for bit.
    other = bf16_dev(np.ascontiguousarray(xbits ^ np.uint16(0x8000)))     # -x
    nv.nvfp4_mlp_decode(other, *args[1:])
    nv.nvfp4_mlp_decode(*args)
    torch.cuda.synchronize()
    got = (host(xq), host(xs), host(hq), host(hs), bf16_host(out))
    ws.zero_()
    out.fill_(float("nan"))
    nv.nvfp4_mlp_decode(*args)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out), got[4]), "reused workspace gives another result"
    assert np.array_equal(host(hq), got[2]), "reused workspace gives another h"
    assert not host(ws[:256].view(torch.int32)).any(), "phase counters not reset"
    return got


def check_all(nv, m, hid, inter, xbits, x, wgu, wdn, round_bf16):
    ref = oracle_chain(x, wgu, wdn, round_bf16)
    gxq, gxs, ghq, ghs, gout = run_fused(nv, xbits, m, hid, inter, wgu, wdn, ref, round_bf16)
    assert np.array_equal(gxq, ref["xq"]), "quantized x codes differ"
    assert np.array_equal(gxs, oracle.sf_swizzle_128x4(ref["xs"])), "quantized x scales differ"
    assert np.array_equal(oracle.sf_swizzle_128x4(oracle.sf_unswizzle_128x4(ghs, m, inter // 16)), ghs), \
        "h scale padding not zero"
    ghs_lin = oracle.sf_unswizzle_128x4(ghs, m, inter // 16)
    flips, sfd = check_requant(ghq, ghs_lin, ref["h"], ref["gs_h"], what="fused MLP h")
    rq, rs = ref["hq"], ref["hs"]
    same = np.array([np.array_equal(ghq[t], rq[t]) and np.array_equal(ghs_lin[t], rs[t]) for t in range(m)])
    assert same.sum() >= (m + 1) // 2, f"only {same.sum()} of {m} rows of h match the oracle's exactly"
    gemm_err = assert_gemm_close(gout[same], ref["out"][same], what="fused MLP down_proj stage")
    err = assert_gemm_close(gout, ref["out"], tol=E2E_TOL, what="fused MLP out")
    print(f"mlp_decode m={m} hid={hid} inter={inter} round={round_bf16}: h flips {flips}, sf diffs {sfd}, "
          f"down_proj rel err {gemm_err:.2e} on {same.sum()}/{m} rows, end-to-end rel err {err:.2e}")


SMALL = [  # (m, hidden, inter)
    (4, 256, 512),      # the tiny workload's shape
    (1, 512, 1024),     # down_proj tiles split across four CTAs
    (5, 384, 320),      # ragged K tails in both GEMMs (K/64 = 6 and 5)
    (16, 1024, 2048),
    (17, 512, 512),     # 32-token tile
    (33, 256, 1024),    # 64-token tile
    (64, 768, 1536),
]


@pytest.mark.parametrize("round_bf16", [1, 0])
@pytest.mark.parametrize("m,hid,inter", SMALL)
def test_mlp_decode_small(lib, m, hid, inter, round_bf16):
    xbits, x = synth.activations(0, m, hid)
    wgu = small_weights(2 * inter, hid, 21)
    wdn = small_weights(hid, inter, 22)
    check_all(lib, m, hid, inter, xbits, x, wgu, wdn, round_bf16)


@pytest.mark.parametrize("wid,m,round_bf16", [(1, 1, 1), (1, 16, 1), (2, 8, 0), (2, 64, 0)])
def test_mlp_decode_full_size(lib, wid, m, round_bf16):
    w = synth.WORKLOADS[wid]
    xbits, x = synth.activations(wid, m)
    check_all(lib, m, w.hidden, w.inter, xbits, x, weights(wid, "gate_up"), weights(wid, "down"), round_bf16)


def test_mlp_decode_bounded_wait_gives_up_cleanly(lib):
    """With a wait limit of one poll the pipeline and phase waits run out: the
    kernel records NVFP4_ERR_DEVICE_TIMEOUT and returns; after the workspace
    is zero-filled again the next normal call is correct."""
    m, hid, inter = 4, 512, 1024
    xbits, x = synth.activations(0, m, hid)
    wgu, wdn = small_weights(2 * inter, hid, 21), small_weights(hid, inter, 22)
    ref = oracle_chain(x, wgu, wdn, 1)
    assert lib.nvfp4_get_device_status() == 0
    lib.nvfp4_set_wait_limit(1)
    try:
        run_fused_once_ignoring_result(lib, xbits, m, hid, inter, wgu, wdn, ref)
    finally:
        lib.nvfp4_set_wait_limit(0)
    assert lib.nvfp4_get_device_status() == lib.ERR_DEVICE_TIMEOUT
    assert lib.nvfp4_get_device_status() == 0
    check_all(lib, m, hid, inter, xbits, x, wgu, wdn, 1)


def run_fused_once_ignoring_result(nv, xbits, m, hid, inter, wgu, wdn, ref):
    xq = torch.empty((m, hid // 2), dtype=torch.uint8, device="cuda")
    xs = torch.empty((nv.nvfp4_sf_bytes(m, hid),), dtype=torch.uint8, device="cuda")
    hq = torch.empty((m, inter // 2), dtype=torch.uint8, device="cuda")
    hs = torch.empty((nv.nvfp4_sf_bytes(m, inter),), dtype=torch.uint8, device="cuda")
    out = torch.empty((m, hid), dtype=torch.bfloat16, device="cuda")
    nbytes = nv.nvfp4_mlp_decode_workspace_bytes(m, hid, inter)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    wi, wd = wgu.device_interleaved(nv), wdn.device_prepared(nv)
    nv.nvfp4_mlp_decode(bf16_dev(xbits), scalar(ref["gs_x"]), wi[0], wi[1], scalar(ref["a_gu"]),
                        scalar(ref["gs_h"]), wd[0], wd[1], scalar(ref["a_dn"]), xq, xs, hq, hs, out, m, hid,
                        inter, 1, ws, nbytes)
    torch.cuda.synchronize()


def test_mlp_decode_argument_errors(lib):
    m, hid, inter = 4, 256, 512
    wgu, wdn = small_weights(2 * inter, hid, 21), small_weights(hid, inter, 22)
    wi, wd = wgu.device_interleaved(lib), wdn.device_prepared(lib)
    x = torch.zeros((65, hid), dtype=torch.bfloat16, device="cuda")
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((65, hid), dtype=torch.bfloat16, device="cuda")
    one = scalar(1.0)
    need = lib.nvfp4_mlp_decode_workspace_bytes(m, hid, inter)
    base = [x, one, wi[0], wi[1], one, one, wd[0], wd[1], one, buf, buf, buf, buf, out, m, hid, inter, 1, buf, need]

    def status(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        with pytest.raises(lib.Nvfp4Error) as e:
            lib.nvfp4_mlp_decode(*a)
        return e.value.status

    assert status(a1=None) == lib.ERR_INVALID_ARG                       # missing scale
    assert status(a14=65) == lib.ERR_UNSUPPORTED_SHAPE                  # m > 64
    assert status(a15=200) == lib.ERR_UNSUPPORTED_SHAPE                 # hidden % 128
    assert status(a19=need - 1) == lib.ERR_INVALID_ARG                  # workspace too small
    assert lib.nvfp4_mlp_decode_workspace_bytes(65, hid, inter) == 0
