"""GPU parity of the MLP chain as the bench times it: nvfp4_quantize ->
nvfp4_gemm_swiglu_quant -> nvfp4_gemm captured with the library's
programmatic dependent launches into one CUDA graph (two forwards on two
copies of the weights), replayed several times.

Programmatic launch edges let a kernel start while its predecessor is still
running; every kernel waits for its predecessor's results before reading
them.  A missing wait would show only here, as a replay that reads a stale or
half-written x or h.  Every replay is therefore checked against the oracle's
chain on the same seeded inputs, with the outputs overwritten by garbage
before each replay:
  * x codes and scales bit-exact;
  * h within the requantize tolerance;
  * out: the token rows whose h is bit-identical to the oracle's hold the
    GEMM tolerance (1e-3; their down_proj input is the oracle's), and all
    rows the end-to-end tolerance.
Workloads: decode H5120/I17408 at M = 1 and 16 (weight-streaming kernels)
and prefill H7168/I18432 at M = 1024 (CTA-pair tensor-core kernels; the
oracle checks 64 stratified tokens)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, bf16_host, host, sample_rows, scalar, weights
from tolerance import assert_gemm_close, check_requant

pytestmark = pytest.mark.gpu

E2E_TOL = 5e-3
REPLAYS = 3


def oracle_rows(aq, asf, ws, alpha, round_bf16, chunk=4096):
    parts = [oracle.gemm_w4a4(aq, asf, ws.packed[r:r + chunk], ws.sf[r:r + chunk], alpha, round_bf16=round_bf16)
             for r in range(0, ws.n, chunk)]
    return np.concatenate(parts, axis=1)


@pytest.mark.parametrize("wid,m,sampled", [(1, 1, None), (1, 16, None), (3, 1024, 64)])
def test_graph_chain_replays_match_oracle(lib, wid, m, sampled):
    w = synth.WORKLOADS[wid]
    hid, inter = w.hidden, w.inter
    wgu, wdn = weights(wid, "gate_up"), weights(wid, "down")
    xbits, x = synth.activations(wid, m)
    toks = np.arange(m) if sampled is None else sample_rows(m, sampled, seed=11)

    # the oracle's chain (fused reading: SwiGLU on the unrounded gate_up)
    gs_x = oracle.global_scale(np.abs(x).max())
    xq, xs = oracle.quantize_nvfp4(x, gs_x)
    a_gu = np.float32(1.0) / (gs_x * wgu.gs)
    h = oracle.swiglu_h(oracle_rows(xq[toks], xs[toks], wgu, a_gu, False))
    gs_h = oracle.global_scale(np.abs(h).max())
    hq, hs = oracle.quantize_nvfp4(h, gs_h)
    a_dn = np.float32(1.0) / (gs_h * wdn.gs)
    out_ref = oracle_rows(hq, hs, wdn, a_dn, True)

    # two copies of the prepared weights, as the bench rotates them
    wi0, wd0 = wgu.device_interleaved(lib), wdn.device_prepared(lib)
    copies = [(wi0, wd0), ((wi0[0].clone(), wi0[1].clone()), (wd0[0].clone(), wd0[1].clone()))]
    x_d = bf16_dev(xbits)
    gsx_d, agu_d, gsh_d, adn_d = scalar(gs_x), scalar(a_gu), scalar(gs_h), scalar(a_dn)
    nbytes = max(lib.nvfp4_workspace_bytes(m, 2 * inter, hid), lib.nvfp4_workspace_bytes(m, hid, inter), 16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    bufs = []
    for _ in copies:
        bufs.append(dict(
            xq=torch.empty((m, hid // 2), dtype=torch.uint8, device="cuda"),
            xs=torch.empty((lib.nvfp4_sf_bytes(m, hid),), dtype=torch.uint8, device="cuda"),
            hq=torch.empty((m, inter // 2), dtype=torch.uint8, device="cuda"),
            hs=torch.empty((lib.nvfp4_sf_bytes(m, inter),), dtype=torch.uint8, device="cuda"),
            out=torch.empty((m, hid), dtype=torch.bfloat16, device="cuda")))

    stream = torch.cuda.Stream()
    sh = stream.cuda_stream

    def forward(c):
        (gq, gsf), (dq, dsf) = copies[c]
        b = bufs[c]
        lib.nvfp4_quantize(x_d, m, hid, gsx_d, b["xq"], b["xs"], stream=sh)
        lib.nvfp4_gemm_swiglu_quant(b["xq"], b["xs"], gq, gsf, agu_d, gsh_d, b["hq"], b["hs"], m, 2 * inter, hid,
                                    ws, nbytes, stream=sh)
        lib.nvfp4_gemm(b["hq"], b["hs"], dq, dsf, adn_d, b["out"], m, hid, inter, ws, nbytes, stream=sh)

    with torch.cuda.stream(stream):
        forward(0)                       # warm outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            forward(0)
            forward(1)
    torch.cuda.synchronize()

    sf_swz = oracle.sf_swizzle_128x4(xs)
    for rep in range(REPLAYS):
        with torch.cuda.stream(stream):
            for b in bufs:
                for key in ("xq", "xs", "hq", "hs"):
                    b[key].fill_(0xAB)
                b["out"].fill_(float("nan"))
            graph.replay()
        stream.synchronize()
        for c, b in enumerate(bufs):
            what = f"replay {rep} copy {c}"
            assert np.array_equal(host(b["xq"]), xq), f"{what}: x codes differ"
            assert np.array_equal(host(b["xs"]), sf_swz), f"{what}: x scales differ"
            ghq = host(b["hq"])[toks]
            ghs = oracle.sf_unswizzle_128x4(host(b["hs"]), m, inter // 16)[toks]
            check_requant(ghq, ghs, h, gs_h, what=f"{what} h")
            gout = bf16_host(b["out"])[toks]
            same = np.array([np.array_equal(ghq[t], hq[t]) and np.array_equal(ghs[t], hs[t])
                             for t in range(len(toks))])
            assert same.sum() >= (len(toks) + 1) // 2, f"{what}: only {same.sum()} rows of h match exactly"
            assert_gemm_close(gout[same], out_ref[same], what=f"{what} down_proj stage")
            assert_gemm_close(gout, out_ref, tol=E2E_TOL, what=f"{what} end to end")
