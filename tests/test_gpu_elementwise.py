"""GPU parity of the HBM-bound kernels against the CPU oracle:
nvfp4_quantize (bit-exact), silu_mul_nvfp4_quantize (requant tolerance),
silu_mul_bf16 (<= 1 bf16 ulp) and the weight-prep calls (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, bf16_host, dev, host, quantized_activation, sample_rows, scalar
from tolerance import check_requant

pytestmark = pytest.mark.gpu


def _run_quantize(nv, bits, m, k, gs, layout):
    q = torch.empty((m, k // 2), dtype=torch.uint8, device="cuda")
    s = torch.full((nv.nvfp4_sf_bytes(m, k, layout),), 0xAB, dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize(bf16_dev(bits), m, k, scalar(gs), q, s, layout)
    torch.cuda.synchronize()
    return host(q), host(s)


QUANT_CASES = [  # (workload, m, k or None)
    (0, 4, None), (1, 1, None), (1, 16, None), (2, 64, None), (3, 1024, None), (4, 128, None),
    (0, 130, 320), (0, 1, 16), (0, 3, 48),
]


@pytest.mark.parametrize("layout", [0, 1], ids=["swizzled", "linear"])
@pytest.mark.parametrize("wid,m,k", QUANT_CASES)
def test_quantize_bit_exact(lib, wid, m, k, layout):
    bits, x, gs, ref_q, ref_s = quantized_activation(wid, m, k)
    k = x.shape[1]
    q, s = _run_quantize(lib, bits, m, k, gs, layout)
    assert np.array_equal(q, ref_q)
    if layout == 0:
        assert np.array_equal(s, oracle.sf_swizzle_128x4(ref_s))     # padding bytes are 0
    else:
        assert np.array_equal(s.reshape(m, k // 16), ref_s)


def test_quantize_full_size_prefill_sampled_rows(lib):
    """M=8192 x K=7168 in the launch the prefill chain uses; 256 sampled rows."""
    m = 8192
    bits, x = synth.activations(3, m)
    gs = oracle.global_scale(np.abs(x).max())
    q, s = _run_quantize(lib, bits, m, x.shape[1], gs, 0)
    rows = sample_rows(m, 256, seed=1)
    ref_q, ref_s = oracle.quantize_nvfp4(x[rows], gs)
    assert np.array_equal(q[rows], ref_q)
    assert np.array_equal(oracle.sf_unswizzle_128x4(s, m, x.shape[1] // 16)[rows], ref_s)


def test_quantize_special_blocks(lib):
    """Exact ties, SF == 0 blocks with negative zeros, saturation, outliers."""
    rows = []
    with open(__file__.replace("test_gpu_elementwise.py", "golden/quant_block.txt")) as f:
        lines = f.read().splitlines()
    for line in lines:
        if line.strip() and not line.startswith("#"):
            rows.append(np.array(line.split("|")[2].split(), dtype=np.float32))
    x = np.concatenate(rows)[None, :]                      # the golden blocks side by side
    x = np.concatenate([x, -x, x * np.float32(1e-30), x * np.float32(1e4)], axis=0).astype(np.float32)
    bits, xv = synth.to_bf16_bits(x)
    # gs = fp32(0.3) puts the golden case-4 block's scale on an exact E4M3 tie
    for gs in (np.float32(1.0), np.float32(0.5), np.float32(0.3), oracle.global_scale(np.abs(xv).max())):
        ref_q, ref_s = oracle.quantize_nvfp4(xv, gs)
        q, s = _run_quantize(lib, bits, xv.shape[0], xv.shape[1], gs, 1)
        assert np.array_equal(q, ref_q) and np.array_equal(s.reshape(ref_s.shape), ref_s)


def test_quantize_m_zero_is_a_noop(lib):
    q = torch.full((1, 128), 7, dtype=torch.uint8, device="cuda")
    s = torch.full((512,), 7, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
    lib.nvfp4_quantize(x, 0, 256, scalar(1.0), q, s)
    torch.cuda.synchronize()
    assert int(q.min()) == 7 and int(s.min()) == 7


def _gate_up_input(m, inter, seed):
    """bf16 [m, 2I] shaped like a gate_up GEMM output (N(0, 1.5^2))."""
    g = synth.random_matrix((m, 2 * inter), (11, m, inter, seed), scale=1.5)
    return synth.to_bf16_bits(g)


@pytest.mark.parametrize("m,inter", [(4, 512), (1, 17408), (16, 17408), (130, 320), (64, 18432)])
def test_silu_mul_quantize(lib, m, inter):
    bits, gu = _gate_up_input(m, inter, 0)
    h = oracle.swiglu_h(gu)
    gs = oracle.global_scale(np.abs(h).max())
    q = torch.empty((m, inter // 2), dtype=torch.uint8, device="cuda")
    s = torch.full((lib.nvfp4_sf_bytes(m, inter),), 0xAB, dtype=torch.uint8, device="cuda")
    lib.silu_mul_nvfp4_quantize(bf16_dev(bits), m, inter, scalar(gs), q, s)
    torch.cuda.synchronize()
    s = host(s)
    lin = oracle.sf_unswizzle_128x4(s, m, inter // 16)
    assert np.array_equal(oracle.sf_swizzle_128x4(lin), s), "padding of the scale buffer is not zero"
    nflip, nsf = check_requant(host(q), lin, h, gs, what="silu_mul_nvfp4_quantize")
    print(f"silu_mul_quant m={m} i={inter}: {nflip} boundary flips, {nsf} scale differences")


# (5, 2056): a ragged last block of column groups; (65539, 24): rows past the
# launch grid's y extent, taken in slices
@pytest.mark.parametrize("m,inter", [(1, 17408), (16, 17408), (128, 17408), (3, 520), (5, 2056), (65539, 24)])
def test_silu_mul_bf16_within_one_ulp(lib, m, inter):
    bits, gu = _gate_up_input(m, inter, 1)
    out = torch.empty((m, inter), dtype=torch.bfloat16, device="cuda")
    lib.silu_mul_bf16(bf16_dev(bits), m, inter, out)
    torch.cuda.synchronize()
    got = bf16_host(out)
    ref = oracle.silu_mul_bf16(gu)
    # bf16 keeps 8 significant bits: spacing at |ref| in [2^(e-1), 2^e) is 2^(e-8)
    ulp = np.ldexp(1.0, np.frexp(np.where(ref == 0, 1e-38, ref))[1] - 8)
    assert np.all(np.abs(got - ref) <= ulp), f"max diff {np.max(np.abs(got - ref) / ulp):.2f} ulp"


@pytest.mark.parametrize("n,k", [(1024, 256), (160, 320), (256, 512), (5120, 17408)])
def test_prepare_weights_bit_exact(lib, n, k):
    from gpu_util import small_weights
    ws = small_weights(n, k, 0)
    w_in = dev(ws.packed)
    w_out = torch.empty_like(w_in)
    s = torch.full((lib.nvfp4_sf_bytes(n, k),), 0xAB, dtype=torch.uint8, device="cuda")
    lib.nvfp4_prepare_weights(w_in, dev(ws.sf), n, k, w_out, s)
    torch.cuda.synchronize()
    assert np.array_equal(host(w_out), ws.packed)
    assert np.array_equal(host(s), oracle.sf_swizzle_128x4(ws.sf))
    # in place: w_out == w_fp4 copies nothing and still writes the scales
    s2 = torch.zeros_like(s)
    lib.nvfp4_prepare_weights(w_in, dev(ws.sf), n, k, w_in, s2)
    torch.cuda.synchronize()
    assert np.array_equal(host(w_in), ws.packed) and np.array_equal(host(s2), host(s))


@pytest.mark.parametrize("n,k", [(1024, 256), (256, 320), (36864, 7168)])
def test_prepare_gate_up_interleaved_bit_exact(lib, n, k):
    from gpu_util import small_weights, weights
    ws = weights(2, "gate_up") if n == 36864 else small_weights(n, k, 1)
    w_out = torch.empty((n, k // 2), dtype=torch.uint8, device="cuda")
    s = torch.full((lib.nvfp4_sf_bytes(n, k),), 0xAB, dtype=torch.uint8, device="cuda")
    lib.nvfp4_prepare_gate_up_interleaved(dev(ws.packed), dev(ws.sf), n, k, w_out, s)
    torch.cuda.synchronize()
    assert np.array_equal(host(w_out), oracle.interleave_gate_up(ws.packed))
    assert np.array_equal(host(s), oracle.interleave_gate_up_scales_then_swizzle(ws.sf))


def test_prepare_is_deterministic(lib):
    from gpu_util import small_weights
    ws = small_weights(256, 512, 2)
    outs = []
    for _ in range(2):
        w_out = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        s = torch.empty((lib.nvfp4_sf_bytes(256, 512),), dtype=torch.uint8, device="cuda")
        lib.nvfp4_prepare_gate_up_interleaved(dev(ws.packed), dev(ws.sf), 256, 512, w_out, s)
        outs.append((host(w_out), host(s)))
    assert all(np.array_equal(a, b) for a, b in zip(*outs))


def test_silu_mul_quantize_masked_groups(lib):
    """Three groups of up to 40 rows, masked to 40, 17 and 0 valid rows."""
    groups, m_max, inter = 3, 40, 512
    masked = np.array([40, 17, 0], dtype=np.int32)
    bits, gu = _gate_up_input(groups * m_max, inter, 5)
    gu3 = gu.reshape(groups, m_max, 2 * inter)
    h_all = oracle.swiglu_h(gu)
    gs = oracle.global_scale(np.abs(h_all).max())
    q = torch.full((groups, m_max, inter // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sfb = lib.nvfp4_sf_bytes(m_max, inter)
    s = torch.full((groups * sfb,), 0xAB, dtype=torch.uint8, device="cuda")
    lib.silu_mul_nvfp4_quantize_masked(bf16_dev(bits), dev(masked), groups, m_max, inter, scalar(gs), q, s)
    torch.cuda.synchronize()
    q, s = host(q), host(s)
    ref = oracle.silu_mul_quant_masked(gu3, masked, gs)
    for e in range(groups):
        v = int(masked[e])
        lin = oracle.sf_unswizzle_128x4(s[e * sfb:(e + 1) * sfb], m_max, inter // 16)
        assert np.all(lin[v:] == 0), "scales of masked rows must be zero"
        pad = oracle.sf_swizzle_128x4(lin)
        assert np.array_equal(pad, s[e * sfb:(e + 1) * sfb]), "padding of the scale block is not zero"
        assert np.all(q[e, v:] == 0xAB), "codes of masked rows must be untouched"
        if v:
            check_requant(q[e, :v], lin[:v], oracle.swiglu_h(gu3[e, :v]), gs, what=f"masked group {e}")
            assert ref[e][0].shape == q[e, :v].shape
