"""Python binding of the NVFP4 dense-MLP C ABI (``include/nvfp4mlp.h``).

Argument marshalling only: every function has the C name and argument
order; pointer arguments accept a torch tensor (its data pointer), a plain
integer address or None (NULL), and ``stream`` defaults to the current torch
CUDA stream.  Every computation runs in the CUDA library; if the library is
not built this module raises instead of falling back to anything else.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libnvfp4mlp.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_ARCH, ERR_CUDA, ERR_DEVICE_TIMEOUT = range(6)
SF_SWIZZLED_128x4, SF_LINEAR = 0, 1
ALGO_AUTO, ALGO_GEMV, ALGO_TC, ALGO_TC_SWAPAB, ALGO_TC_1SM = 0, 1, 2, 3, 4

_lib = None


class Nvfp4Error(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: status {status} ({msg})")
        self.status = status


_P, _I64, _SZ, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int

_SIGS = {
    "nvfp4_quantize": [_P, _I64, _I64, _P, _P, _P, _I, _P],
    "silu_mul_nvfp4_quantize": [_P, _I64, _I64, _P, _P, _P, _P],
    "silu_mul_nvfp4_quantize_masked": [_P, _P, _I64, _I64, _I64, _P, _P, _P, _P],
    "nvfp4_quantize_per_token": [_P, _I64, _I64, _P, _P, _I, _P, _P],
    "nvfp4_gemm_per_token": [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _I, _P],
    "nvfp4_gemm_swiglu_quant_per_token": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ,
                                          _I, _P],
    "silu_mul_bf16": [_P, _I64, _I64, _P, _P],
    "nvfp4_gemm": [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P],
    "nvfp4_gemm_ex": [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _I, _P],
    "nvfp4_gemm_swiglu_quant": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P],
    "nvfp4_gemm_swiglu_quant_ex": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _I, _P],
    "nvfp4_quantize_gemm_swiglu_quant": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P],
    "bf16_fp4_gemm": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P],
    "bf16_fp4_gemm_ex": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _I, _P],
    "bf16_fp4_gemm_prescaled": [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _I, _P],
    "bf16_awq_prescale": [_P, _P, _P, _I64, _I64, _P],
    "nvfp4_mlp_decode": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _P, _SZ,
                         _P],
    "nvfp4_prepare_weights": [_P, _P, _I64, _I64, _P, _P, _P],
    "nvfp4_prepare_gate_up_interleaved": [_P, _P, _I64, _I64, _P, _P, _P],
    "nvfp4_gemm_decode_noalloc": [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P],
    "nvfp4_get_device_status": [ctypes.POINTER(_I), _P],
    "nvfp4_set_wait_limit": [ctypes.c_uint32],
}
EXPORTS = sorted(list(_SIGS) + ["nvfp4_status_string", "nvfp4_version", "nvfp4_sf_bytes",
                                "nvfp4_workspace_bytes", "bf16_fp4_gemm_prescaled_workspace_bytes",
                                "bf16_fp4_gemm_workspace_bytes",
                                "nvfp4_mlp_decode_workspace_bytes",
                                "nvfp4_quantize_gemm_swiglu_quant_workspace_bytes"])


def load(path=LIB_PATH):
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"NVFP4 CUDA library not built: {path} is missing "
                          "(run `python -m nvfp4_quantized_dense_gb300.build`)")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, _I
    lib.nvfp4_status_string.argtypes, lib.nvfp4_status_string.restype = [_I], ctypes.c_char_p
    lib.nvfp4_version.argtypes, lib.nvfp4_version.restype = [], _I
    lib.nvfp4_sf_bytes.argtypes, lib.nvfp4_sf_bytes.restype = [_I64, _I64, _I], _SZ
    lib.nvfp4_workspace_bytes.argtypes, lib.nvfp4_workspace_bytes.restype = [_I64, _I64, _I64, _I], _SZ
    lib.bf16_fp4_gemm_prescaled_workspace_bytes.argtypes = [_I64, _I64, _I64, _I]
    lib.bf16_fp4_gemm_prescaled_workspace_bytes.restype = _SZ
    lib.bf16_fp4_gemm_workspace_bytes.argtypes = [_I64, _I64, _I64, _I]
    lib.bf16_fp4_gemm_workspace_bytes.restype = _SZ
    lib.nvfp4_mlp_decode_workspace_bytes.argtypes = [_I64, _I64, _I64]
    lib.nvfp4_mlp_decode_workspace_bytes.restype = _SZ
    lib.nvfp4_quantize_gemm_swiglu_quant_workspace_bytes.argtypes = [_I64, _I64, _I64]
    lib.nvfp4_quantize_gemm_swiglu_quant_workspace_bytes.restype = _SZ
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


_torch = None


def _stream(s):
    if s is None:
        global _torch
        if _torch is None:
            import torch
            _torch = torch
        return _torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _call(name, *args):
    st = getattr(load(), name)(*args)
    if st != OK:
        raise Nvfp4Error(name, st, load().nvfp4_status_string(st).decode())


def nvfp4_status_string(status):
    return load().nvfp4_status_string(status).decode()


def nvfp4_version():
    return load().nvfp4_version()


def nvfp4_sf_bytes(rows, k, layout=SF_SWIZZLED_128x4):
    return load().nvfp4_sf_bytes(rows, k, layout)


def nvfp4_workspace_bytes(m, n, k, algo=ALGO_AUTO):
    return load().nvfp4_workspace_bytes(m, n, k, algo)


def bf16_fp4_gemm_workspace_bytes(m, n, k, algo=ALGO_AUTO):
    return load().bf16_fp4_gemm_workspace_bytes(m, n, k, algo)


def bf16_fp4_gemm_prescaled_workspace_bytes(m, n, k, algo=ALGO_AUTO):
    return load().bf16_fp4_gemm_prescaled_workspace_bytes(m, n, k, algo)


def nvfp4_mlp_decode_workspace_bytes(m, hidden, inter):
    return load().nvfp4_mlp_decode_workspace_bytes(m, hidden, inter)


def nvfp4_mlp_decode(x, x_global_scale, w_gate_up_int, w_gate_up_int_sf, alpha_gate_up, h_global_scale,
                     w_down, w_down_sf, alpha_down, x_fp4, x_sf, h_fp4, h_sf, out, m, hidden, inter,
                     round_gate_up_bf16, workspace, ws_bytes, stream=None):
    _call("nvfp4_mlp_decode", _ptr(x), _ptr(x_global_scale), _ptr(w_gate_up_int), _ptr(w_gate_up_int_sf),
          _ptr(alpha_gate_up), _ptr(h_global_scale), _ptr(w_down), _ptr(w_down_sf), _ptr(alpha_down),
          _ptr(x_fp4), _ptr(x_sf), _ptr(h_fp4), _ptr(h_sf), _ptr(out), m, hidden, inter,
          1 if round_gate_up_bf16 else 0, _ptr(workspace), ws_bytes, _stream(stream))


def bf16_awq_prescale(x, pre_quant_scale, out, m, k, stream=None):
    _call("bf16_awq_prescale", _ptr(x), _ptr(pre_quant_scale), _ptr(out), m, k, _stream(stream))


def nvfp4_quantize(x, m, k, global_scale, out_fp4, out_sf, sf_layout=SF_SWIZZLED_128x4, stream=None):
    _call("nvfp4_quantize", _ptr(x), m, k, _ptr(global_scale), _ptr(out_fp4), _ptr(out_sf),
          sf_layout, _stream(stream))


def silu_mul_nvfp4_quantize(gate_up, m, i, global_scale, out_fp4, out_sf, stream=None):
    _call("silu_mul_nvfp4_quantize", _ptr(gate_up), m, i, _ptr(global_scale), _ptr(out_fp4),
          _ptr(out_sf), _stream(stream))


def silu_mul_nvfp4_quantize_masked(gate_up, masked_m, g, m_max, i, global_scale, out_fp4, out_sf,
                                   stream=None):
    _call("silu_mul_nvfp4_quantize_masked", _ptr(gate_up), _ptr(masked_m), g, m_max, i, _ptr(global_scale),
          _ptr(out_fp4), _ptr(out_sf), _stream(stream))


def nvfp4_quantize_per_token(x, m, k, out_fp4, out_sf, sf_layout, out_row_scale, stream=None):
    _call("nvfp4_quantize_per_token", _ptr(x), m, k, _ptr(out_fp4), _ptr(out_sf), sf_layout,
          _ptr(out_row_scale), _stream(stream))


def nvfp4_gemm_per_token(a_fp4, a_sf, a_row_scale, b_fp4, b_sf, alpha, d, m, n, k, workspace=None,
                         ws_bytes=0, algo=ALGO_AUTO, stream=None):
    _call("nvfp4_gemm_per_token", _ptr(a_fp4), _ptr(a_sf), _ptr(a_row_scale), _ptr(b_fp4), _ptr(b_sf),
          _ptr(alpha), _ptr(d), m, n, k, _ptr(workspace), ws_bytes, algo, _stream(stream))


def nvfp4_gemm_swiglu_quant_per_token(a_fp4, a_sf, a_row_scale, w_int_fp4, w_int_sf, alpha,
                                      out_global_scale, out_fp4, out_sf, m, n, k, workspace=None,
                                      ws_bytes=0, algo=ALGO_AUTO, stream=None):
    _call("nvfp4_gemm_swiglu_quant_per_token", _ptr(a_fp4), _ptr(a_sf), _ptr(a_row_scale), _ptr(w_int_fp4),
          _ptr(w_int_sf), _ptr(alpha), _ptr(out_global_scale), _ptr(out_fp4), _ptr(out_sf), m, n, k,
          _ptr(workspace), ws_bytes, algo, _stream(stream))


def silu_mul_bf16(gate_up, m, i, out, stream=None):
    _call("silu_mul_bf16", _ptr(gate_up), m, i, _ptr(out), _stream(stream))


def nvfp4_gemm(a_fp4, a_sf, b_fp4, b_sf, alpha, d, m, n, k, workspace=None, ws_bytes=0, stream=None):
    _call("nvfp4_gemm", _ptr(a_fp4), _ptr(a_sf), _ptr(b_fp4), _ptr(b_sf), _ptr(alpha), _ptr(d),
          m, n, k, _ptr(workspace), ws_bytes, _stream(stream))


def nvfp4_gemm_ex(a_fp4, a_sf, b_fp4, b_sf, alpha, d, m, n, k, workspace=None, ws_bytes=0,
                  algo=ALGO_AUTO, stream=None):
    _call("nvfp4_gemm_ex", _ptr(a_fp4), _ptr(a_sf), _ptr(b_fp4), _ptr(b_sf), _ptr(alpha), _ptr(d),
          m, n, k, _ptr(workspace), ws_bytes, algo, _stream(stream))


def nvfp4_gemm_swiglu_quant(a_fp4, a_sf, w_int_fp4, w_int_sf, alpha, out_global_scale, out_fp4,
                            out_sf, m, n, k, workspace=None, ws_bytes=0, stream=None):
    _call("nvfp4_gemm_swiglu_quant", _ptr(a_fp4), _ptr(a_sf), _ptr(w_int_fp4), _ptr(w_int_sf),
          _ptr(alpha), _ptr(out_global_scale), _ptr(out_fp4), _ptr(out_sf), m, n, k,
          _ptr(workspace), ws_bytes, _stream(stream))


def nvfp4_quantize_gemm_swiglu_quant_workspace_bytes(m, n, k):
    return load().nvfp4_quantize_gemm_swiglu_quant_workspace_bytes(m, n, k)


def nvfp4_quantize_gemm_swiglu_quant(x, x_global_scale, x_fp4, x_sf, w_int_fp4, w_int_sf, alpha,
                                     out_global_scale, out_fp4, out_sf, m, n, k, workspace=None, ws_bytes=0,
                                     stream=None):
    _call("nvfp4_quantize_gemm_swiglu_quant", _ptr(x), _ptr(x_global_scale), _ptr(x_fp4), _ptr(x_sf),
          _ptr(w_int_fp4), _ptr(w_int_sf), _ptr(alpha), _ptr(out_global_scale), _ptr(out_fp4), _ptr(out_sf),
          m, n, k, _ptr(workspace), ws_bytes, _stream(stream))


def nvfp4_gemm_swiglu_quant_ex(a_fp4, a_sf, w_int_fp4, w_int_sf, alpha, out_global_scale, out_fp4,
                               out_sf, m, n, k, workspace=None, ws_bytes=0, algo=ALGO_AUTO,
                               stream=None):
    _call("nvfp4_gemm_swiglu_quant_ex", _ptr(a_fp4), _ptr(a_sf), _ptr(w_int_fp4), _ptr(w_int_sf),
          _ptr(alpha), _ptr(out_global_scale), _ptr(out_fp4), _ptr(out_sf), m, n, k,
          _ptr(workspace), ws_bytes, algo, _stream(stream))


def bf16_fp4_gemm(a, b_fp4, b_sf, alpha, d, m, n, k, workspace=None, ws_bytes=0, stream=None):
    _call("bf16_fp4_gemm", _ptr(a), _ptr(b_fp4), _ptr(b_sf), _ptr(alpha), _ptr(d), m, n, k,
          _ptr(workspace), ws_bytes, _stream(stream))


def bf16_fp4_gemm_ex(a, b_fp4, b_sf, alpha, d, m, n, k, workspace=None, ws_bytes=0, algo=ALGO_AUTO,
                     stream=None):
    _call("bf16_fp4_gemm_ex", _ptr(a), _ptr(b_fp4), _ptr(b_sf), _ptr(alpha), _ptr(d), m, n, k,
          _ptr(workspace), ws_bytes, algo, _stream(stream))


def bf16_fp4_gemm_prescaled(a, pre_quant_scale, b_fp4, b_sf, alpha, d, m, n, k, workspace=None, ws_bytes=0,
                            algo=ALGO_AUTO, stream=None):
    _call("bf16_fp4_gemm_prescaled", _ptr(a), _ptr(pre_quant_scale), _ptr(b_fp4), _ptr(b_sf), _ptr(alpha),
          _ptr(d), m, n, k, _ptr(workspace), ws_bytes, algo, _stream(stream))


def nvfp4_prepare_weights(w_fp4, sf_linear, n, k, w_out, sf_out, stream=None):
    _call("nvfp4_prepare_weights", _ptr(w_fp4), _ptr(sf_linear), n, k, _ptr(w_out), _ptr(sf_out),
          _stream(stream))


def nvfp4_prepare_gate_up_interleaved(w_fp4, sf_linear, n, k, w_out, sf_out, stream=None):
    _call("nvfp4_prepare_gate_up_interleaved", _ptr(w_fp4), _ptr(sf_linear), n, k, _ptr(w_out),
          _ptr(sf_out), _stream(stream))


def nvfp4_gemm_decode_noalloc(a_fp4, a_sf, b_fp4, b_sf, alpha, d, m, n, k, stream=None):
    """Decode GEMM whose split-K scratch lives inside the library (for
    callers that cannot provide a workspace)."""
    _call("nvfp4_gemm_decode_noalloc", _ptr(a_fp4), _ptr(a_sf), _ptr(b_fp4), _ptr(b_sf), _ptr(alpha),
          _ptr(d), m, n, k, _stream(stream))


def nvfp4_get_device_status(stream=None):
    v = ctypes.c_int(0)
    _call("nvfp4_get_device_status", ctypes.byref(v), _stream(stream))
    return v.value


def nvfp4_set_wait_limit(spins):
    _call("nvfp4_set_wait_limit", spins)
