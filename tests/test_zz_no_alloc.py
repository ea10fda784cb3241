"""The decode GEMM entry point that allocates nothing.

Some callers cannot give the library a workspace: a host program that only
holds the buffers it was handed, a plugin whose host framework owns all
device memory, or a path that must not allocate.  nvfp4_gemm_decode_noalloc
serves them from a fixed scratch array inside the library.  Its result must
match nvfp4_gemm (weight-streaming tensor-core kernel, caller workspace)
within the GEMM tolerance, on two calls in a row -- the second call finds the
array holding the first call's leftovers and must still be right.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_host, dev, quantized_activation, scalar, small_weights
from tolerance import assert_gemm_close

pytestmark = pytest.mark.gpu

TC_SWAPAB = 3


@pytest.mark.parametrize("m,n,k", [(4, 512, 4096), (16, 2048, 8192), (1, 256, 256), (33, 384, 1024)])
def test_noalloc_matches_workspace_entry_point(lib, m, n, k):
    ws = small_weights(n, k, 13)
    w, w_sf = ws.device_prepared(lib)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = scalar(np.float32(1.0) / (gs_x * ws.gs))
    a, a_sf = dev(xq), dev(oracle.sf_swizzle_128x4(xs))

    nbytes = lib.nvfp4_workspace_bytes(m, n, k, TC_SWAPAB)
    scratch = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    ref = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    lib.nvfp4_gemm_ex(a, a_sf, w, w_sf, alpha, ref, m, n, k, scratch, nbytes, algo=TC_SWAPAB)
    torch.cuda.synchronize()
    ref = bf16_host(ref)
    assert_gemm_close(ref, oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, np.float32(alpha.item())))

    for _ in range(2):
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        lib.nvfp4_gemm_decode_noalloc(a, a_sf, w, w_sf, alpha, out, m, n, k)
        torch.cuda.synchronize()
        assert_gemm_close(bf16_host(out), ref, what="noalloc vs workspace entry point")


def test_noalloc_rejects_too_much_scratch(lib):
    """A split plan larger than the fixed array is refused before launch.
    The operands are real device buffers of the stated shape, so a launch
    that should not happen would compute on valid memory rather than fault."""
    m, n, k = 64, 256, 65536
    need = lib.nvfp4_workspace_bytes(m, n, k, TC_SWAPAB)
    assert need > (8 << 20)
    a = torch.zeros((m, k // 2), dtype=torch.uint8, device="cuda")
    a_sf = torch.zeros((lib.nvfp4_sf_bytes(m, k),), dtype=torch.uint8, device="cuda")
    w = torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda")
    w_sf = torch.zeros((lib.nvfp4_sf_bytes(n, k),), dtype=torch.uint8, device="cuda")
    out = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.Nvfp4Error) as e:
        lib.nvfp4_gemm_decode_noalloc(a, a_sf, w, w_sf, scalar(1.0), out, m, n, k)
    assert e.value.status == lib.ERR_UNSUPPORTED_SHAPE


def test_noalloc_bounded_wait_gives_up_cleanly(lib):
    """The wait limit set through nvfp4_set_wait_limit applies to this entry
    point too: with one poll the kernel gives up, reports the timeout, and the
    next normal call (which clears the array's counters again) is right."""
    m, n, k = 16, 2048, 8192
    ws = small_weights(n, k, 13)
    w, w_sf = ws.device_prepared(lib)
    _, _, gs_x, xq, xs = quantized_activation(0, m, k)
    alpha = np.float32(1.0) / (gs_x * ws.gs)
    a, a_sf = dev(xq), dev(oracle.sf_swizzle_128x4(xs))
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    assert lib.nvfp4_get_device_status() == 0
    lib.nvfp4_set_wait_limit(1)
    try:
        lib.nvfp4_gemm_decode_noalloc(a, a_sf, w, w_sf, scalar(alpha), out, m, n, k)
    finally:
        lib.nvfp4_set_wait_limit(0)
    assert lib.nvfp4_get_device_status() == lib.ERR_DEVICE_TIMEOUT
    lib.nvfp4_gemm_decode_noalloc(a, a_sf, w, w_sf, scalar(alpha), out, m, n, k)
    torch.cuda.synchronize()
    assert lib.nvfp4_get_device_status() == 0
    assert_gemm_close(bf16_host(out), oracle.gemm_w4a4(xq, xs, ws.packed, ws.sf, alpha))
