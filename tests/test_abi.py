"""Host-side checks of the C ABI: the library builds, loads and exports every
function declared in include/nvfp4mlp.h; argument validation answers before
any launch.  No GPU needed (and no compute call is made)."""
import os
import re

import pytest

import nvfp4_quantized_dense_gb300 as nv
import oracle
from nvfp4_quantized_dense_gb300 import build as nvbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "nvfp4mlp.h")


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.load()


def _declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z0-9_]+)\s*\(", text)) - {"sizeof"})


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert "nvfp4_gemm_swiglu_quant" in names and len(names) >= 17
    for name in names:
        assert hasattr(lib, name), f"{name} declared in nvfp4mlp.h but not exported"
    assert sorted(names) == sorted(nv.EXPORTS)


def test_version_and_status_strings(lib):
    assert nv.nvfp4_version() >> 16 == 1
    for s in range(6):
        assert nv.nvfp4_status_string(s)
    assert "sm_103" in nv.nvfp4_status_string(nv.ERR_ARCH)


@pytest.mark.parametrize("rows,k", [(1, 16), (4, 256), (130, 320), (8192, 7168), (0, 64)])
def test_sf_bytes(lib, rows, k):
    assert nv.nvfp4_sf_bytes(rows, k, nv.SF_SWIZZLED_128x4) == oracle.sf_swizzled_bytes(rows, k // 16)
    assert nv.nvfp4_sf_bytes(rows, k, nv.SF_LINEAR) == rows * k // 16
    assert nv.nvfp4_sf_bytes(rows, 24, nv.SF_LINEAR) == 0
    assert nv.nvfp4_workspace_bytes(rows, 1024, k) == 0


FAKE = 1 << 20   # 16-byte aligned address that is never dereferenced


def test_null_pointers_rejected(lib):
    assert lib.nvfp4_quantize(None, 4, 256, FAKE, FAKE, FAKE, 0, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm(FAKE, FAKE, FAKE, None, FAKE, FAKE, 4, 256, 256, None, 0, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm_swiglu_quant(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 4, 256, 256,
                                       None, 0, None) == nv.ERR_INVALID_ARG
    assert lib.bf16_fp4_gemm(None, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None, 0, None) == nv.ERR_INVALID_ARG
    assert lib.silu_mul_nvfp4_quantize(FAKE, 4, 256, None, FAKE, FAKE, None) == nv.ERR_INVALID_ARG
    assert lib.silu_mul_bf16(FAKE, 4, 256, None, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_prepare_weights(FAKE, None, 256, 256, FAKE, FAKE, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_get_device_status(None, None) == nv.ERR_INVALID_ARG


def test_bad_sizes_rejected(lib):
    assert lib.nvfp4_quantize(FAKE, -1, 256, FAKE, FAKE, FAKE, 0, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_quantize(FAKE, 4, 250, FAKE, FAKE, FAKE, 0, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_quantize(FAKE, 4, 256, FAKE, FAKE, FAKE, 7, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_quantize(FAKE + 8, 4, 256, FAKE, FAKE, FAKE, 0, None) == nv.ERR_UNSUPPORTED_SHAPE
    # GEMMs: K % 64, N % 32, fused N % 128
    assert lib.nvfp4_gemm(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 96, None, 0, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemm(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 100, 256, None, 0, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemm(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0, 256, None, 0, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm_swiglu_quant(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 96, 256,
                                       None, 0, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_gemm_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None, 0, 9, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_prepare_gate_up_interleaved(FAKE, FAKE, 192, 256, FAKE + 4096, FAKE, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_prepare_gate_up_interleaved(FAKE, FAKE, 256, 256, FAKE, FAKE, None) == nv.ERR_INVALID_ARG
    assert lib.silu_mul_bf16(FAKE, 4, 12, FAKE, None) == nv.ERR_UNSUPPORTED_SHAPE


def test_binding_raises_on_error(lib):
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_quantize(FAKE, 4, 250, FAKE, FAKE, FAKE, stream=0)
    assert e.value.status == nv.ERR_UNSUPPORTED_SHAPE


def test_valid_call_without_a_gpu_launches_nothing(lib):
    """On a machine without a usable GB300 a well-formed call must come back
    with an error status (ARCH or CUDA), not crash or fall back."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = lib.nvfp4_quantize(FAKE, 4, 256, FAKE, FAKE, FAKE, 0, None)
    assert st in (nv.ERR_ARCH, nv.ERR_CUDA)


def test_missing_library_raises(tmp_path):
    saved = nv._lib
    nv._lib = None
    try:
        with pytest.raises(ImportError):
            nv.load(str(tmp_path / "missing.so"))
    finally:
        nv._lib = saved


def test_awq_prescale_host_checks(lib):
    # workspace: m*k bf16 (rounded up to 256) plus the W4A16 GEMM's scratch on
    # the tensor cores (the TMEM kernel's counters, split-K partials, f16
    # activations and row scales: never empty), none on the GEMV
    r256 = lambda b: (b + 255) // 256 * 256
    for m, n, k in [(1, 256, 512), (65, 256, 512), (16, 34816, 5120), (1024, 34816, 5120)]:
        assert nv.bf16_fp4_gemm_prescaled_workspace_bytes(m, n, k) == \
            r256(m * k * 2) + nv.bf16_fp4_gemm_workspace_bytes(m, n, k)
    assert nv.bf16_fp4_gemm_workspace_bytes(16, 34816, 5120) > 0
    assert nv.bf16_fp4_gemm_workspace_bytes(65, 34816, 5120) >= 64 * 1024 + 65 * 5120 * 2
    assert nv.bf16_fp4_gemm_workspace_bytes(65, 5120, 17408) > 0
    assert nv.bf16_fp4_gemm_workspace_bytes(16, 34816, 5120, nv.ALGO_GEMV) == 0
    assert nv.bf16_fp4_gemm_prescaled_workspace_bytes(0, 256, 512) == 0
    assert nv.bf16_fp4_gemm_prescaled_workspace_bytes(1024, 34816, 5120, nv.ALGO_TC) == \
        1024 * 5120 * 2 + nv.bf16_fp4_gemm_workspace_bytes(1024, 34816, 5120, nv.ALGO_TC)
    assert nv.bf16_fp4_gemm_prescaled_workspace_bytes(1024, 34816, 5120, nv.ALGO_GEMV) == 0
    assert lib.bf16_awq_prescale(None, FAKE, FAKE, 4, 256, None) == nv.ERR_INVALID_ARG
    assert lib.bf16_awq_prescale(FAKE, FAKE, FAKE, 4, 100, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.bf16_awq_prescale(FAKE, FAKE + 2, FAKE, 4, 256, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.bf16_fp4_gemm_prescaled(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None, 0, 0,
                                       None) == nv.ERR_INVALID_ARG
    assert lib.bf16_fp4_gemm_prescaled(FAKE, FAKE + 8, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None, 0, 0,
                                       None) == nv.ERR_UNSUPPORTED_SHAPE


def test_mlp_decode_host_checks(lib):
    args = [FAKE] * 14 + [4, 256, 512, 1, FAKE, 1 << 30, None]
    bad = list(args)
    bad[1] = None                                    # no x global scale
    assert lib.nvfp4_mlp_decode(*bad) == nv.ERR_INVALID_ARG
    bad = list(args)
    bad[14] = 65                                     # more tokens than the kernel takes
    assert lib.nvfp4_mlp_decode(*bad) == nv.ERR_UNSUPPORTED_SHAPE
    bad = list(args)
    bad[15] = 320                                    # hidden % 128
    assert lib.nvfp4_mlp_decode(*bad) == nv.ERR_UNSUPPORTED_SHAPE
    bad = list(args)
    bad[19] = 16                                     # workspace too small
    assert lib.nvfp4_mlp_decode(*bad) == nv.ERR_INVALID_ARG
    bad = list(args)
    bad[14] = 0                                      # no tokens: nothing to do
    assert lib.nvfp4_mlp_decode(*bad) == nv.OK
    assert nv.nvfp4_mlp_decode_workspace_bytes(4, 256, 512) > 0
    assert nv.nvfp4_mlp_decode_workspace_bytes(65, 256, 512) == 0


def test_per_token_and_masked_host_checks(lib):
    # per-token quantize: the row-scale output is required, K % 16, layout enum
    assert lib.nvfp4_quantize_per_token(FAKE, 4, 256, FAKE, FAKE, 0, None, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token(FAKE, 4, 100, FAKE, FAKE, 0, FAKE, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_quantize_per_token(FAKE, 4, 256, FAKE, FAKE, 5, FAKE, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_per_token(FAKE, -1, 256, FAKE, FAKE, 0, FAKE, None) == nv.ERR_INVALID_ARG
    # per-token GEMMs: the row factor is required
    assert lib.nvfp4_gemm_per_token(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None, 0, 0,
                                    None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm_swiglu_quant_per_token(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256,
                                                 256, None, 0, 0, None) == nv.ERR_INVALID_ARG
    # masked groups: masked_m required, I % 16, at most 65535 groups
    assert lib.silu_mul_nvfp4_quantize_masked(FAKE, None, 2, 4, 256, FAKE, FAKE, FAKE,
                                              None) == nv.ERR_INVALID_ARG
    assert lib.silu_mul_nvfp4_quantize_masked(FAKE, FAKE, -1, 4, 256, FAKE, FAKE, FAKE,
                                              None) == nv.ERR_INVALID_ARG
    assert lib.silu_mul_nvfp4_quantize_masked(FAKE, FAKE, 2, 4, 24, FAKE, FAKE, FAKE,
                                              None) == nv.ERR_UNSUPPORTED_SHAPE
    assert lib.silu_mul_nvfp4_quantize_masked(FAKE, FAKE, 65536, 4, 256, FAKE, FAKE, FAKE,
                                              None) == nv.ERR_UNSUPPORTED_SHAPE


def _declared_params():
    """{function: [C parameter type, ...]} parsed from the header."""
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(?:nvfp4_status|size_t|int|const char \*)\s+([a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = [re.sub(r"([\s*])[a-z0-9_]+$", r"\1", p).strip() for p in params]
    return out


def _ctype_kind(c_type):
    t = c_type.replace("const ", "").strip()
    if "*" in t or t == "nvfp4_stream_t":
        return "ptr"
    return {"int64_t": "i64", "size_t": "size", "uint32_t": "u32", "int": "int",
            "nvfp4_sf_layout": "int", "nvfp4_algo": "int"}[t]


def test_binding_signatures_match_the_header():
    import ctypes
    kind = {ctypes.c_void_p: "ptr", ctypes.c_int64: "i64", ctypes.c_size_t: "size", ctypes.c_int: "int",
            ctypes.c_uint32: "u32"}
    declared = _declared_params()
    for fn, argtypes in nv._SIGS.items():
        assert fn in declared, fn
        got = ["ptr" if isinstance(a, type) and issubclass(a, ctypes._Pointer) else kind[a] for a in argtypes]
        assert got == [_ctype_kind(t) for t in declared[fn]], fn
