"""ctypes binding of librnl.so (include/rnl.h).

Argument marshalling only: tensors are checked for device, dtype and
layout, outputs and workspace are allocated with torch when the caller
passes none, and the raw pointers plus the current CUDA stream are handed to
the C entry point of the same name.  Every step of the computation runs in
the library's CUDA kernels; there is no other code path.  If the library
has not been built, every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "librnl.so")
DEBUG_LIB_PATH = os.path.join(PKG, "librnl_debug.so")

NORM_RSQRT, NORM_SQRT_DIV = 0, 1
OUT_BF16, OUT_FP32 = 0, 1
OP_BF16, OP_W8A8, OP_MLA, OP_GEMM_S8, OP_QKV_ROPE, OP_QMRS, OP_MXFP8, OP_W8A8_PREPARED = range(8)

STATUS = {
    0: "RNL_OK", 1: "RNL_ERR_NULL", 2: "RNL_ERR_SHAPE", 3: "RNL_ERR_ALIGN", 4: "RNL_ERR_ARG",
    5: "RNL_ERR_WORKSPACE", 6: "RNL_ERR_LAUNCH", 7: "RNL_ERR_TIMEOUT", 8: "RNL_ERR_UNSUPPORTED",
    9: "RNL_ERR_DEVICE", 10: "RNL_ERR_BOUNDS",
}

EXPORTS = ("rnl_version", "rnl_debug_build", "rnl_selftest_bounds_check", "rnl_status_string", "rnl_workspace_size", "rmsnorm_linear_bf16",
           "rmsnorm_linear_w8a8", "mla_q_chain", "rnl_gemm_s8s8s32", "rnl_check_device_error",
           "rnl_trace_enable", "rnl_trace_read", "rmsnorm_linear_skinny_noalloc",
           "rnl_selftest_wait_timeout", "rnl_pipeline_create", "rnl_pipeline_submit_bf16",
           "rnl_pipeline_submit_w8a8", "rnl_pipeline_submit_mla", "rnl_pipeline_wait",
           "rnl_pipeline_destroy", "rmsnorm_linear_bf16_ex", "rnl_qkv_rope",
           "rmsnorm_linear_qkv_rope", "quant_matmul_reduce_sum", "rmsnorm_linear_mxfp8",
           "mxfp8_scaled_mm", "rnl_head_rmsnorm", "mla_q_chain_head_norm", "rnl_w8a8_prepare_weight",
           "rmsnorm_linear_w8a8_prepared")


class RnlError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


_lock = threading.Lock()
_lib = None


def _declare(lib):
    P, I64, F, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
    sig = {
        "rnl_version": (I, []),
        "rnl_debug_build": (I, []),
        "rnl_selftest_bounds_check": (I, [P]),
        "rnl_status_string": (ctypes.c_char_p, [I]),
        "rnl_workspace_size": (SZ, [I, I64, I64, I64, I64]),
        "rmsnorm_linear_bf16": (I, [P, P, P, I64, I64, I64, F, I, P, I, P, SZ, P]),
        "rmsnorm_linear_w8a8": (I, [P, P, P, P, I64, I64, I64, F, I, P, P, P, P, SZ, P]),
        "rmsnorm_linear_w8a8_prepared": (I, [P, P, P, P, I64, I64, I64, F, I, P, P, P, P, SZ, P]),
        "rnl_w8a8_prepare_weight": (I, [P, I64, I64, P, P]),
        "mla_q_chain": (I, [P, P, P, P, I64, I64, I64, I64, F, I, P, P, P, SZ, P]),
        "rnl_gemm_s8s8s32": (I, [P, P, P, I64, I64, I64, P, SZ, P]),
        "rnl_check_device_error": (I, [P, ctypes.POINTER(I)]),
        "rnl_trace_enable": (I, [I]),
        "rnl_trace_read": (I, [P, ctypes.POINTER(F), I]),
        "rmsnorm_linear_skinny_noalloc": (I, [P, P, I64, I64, I64, F, I, P, P]),
        "rnl_selftest_wait_timeout": (I, [P]),
        "rnl_pipeline_create": (I, [I, I64, I64, I64, I64, ctypes.POINTER(P)]),
        "rnl_pipeline_submit_bf16": (I, [P, P, P, P, F, I, P, ctypes.POINTER(I64)]),
        "rnl_pipeline_submit_w8a8": (I, [P, P, P, P, P, F, I, P, ctypes.POINTER(I64)]),
        "rnl_pipeline_submit_mla": (I, [P, P, P, P, P, F, I, P, ctypes.POINTER(I64)]),
        "rnl_pipeline_wait": (I, [P, I64, ctypes.POINTER(I)]),
        "rnl_pipeline_destroy": (I, [P]),
        "rmsnorm_linear_bf16_ex": (I, [P, P, P, P, P, P, P, I64, I64, I64, F, I, P, P, P, SZ, P]),
        "rnl_qkv_rope": (I, [P, I64, I64, I64, I64, P, P, F, P, P, I64, P, P, P, P]),
        "quant_matmul_reduce_sum": (I, [P, P, P, P, I64, I64, I64, I64, P, P, SZ, P]),
        "rmsnorm_linear_mxfp8": (I, [P, P, P, P, I64, I64, I64, F, I, I64, P, I, P, P, P, SZ, P]),
        "mxfp8_scaled_mm": (I, [P, P, P, P, I64, I64, I64, I64, P, I, P, SZ, P]),
        "rnl_head_rmsnorm": (I, [P, I64, I64, I64, P, F, I, P, P]),
        "mla_q_chain_head_norm": (I, [P, P, P, P, I64, I64, I64, I64, F, I, I64, P, F, P, P, P, SZ, P]),
        "rmsnorm_linear_qkv_rope": (I, [P, P, P, I64, I64, I64, I64, I64, F, I, P, P, F, P, P, I64,
                                        P, P, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None):
    """Load librnl.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with "
                                   "`python -m rmsnorm_linear_projection_gb300.build`")
            lib = _declare(ctypes.CDLL(p))
            if path is not None:
                return lib
            _lib = lib
    return _lib


@contextlib.contextmanager
def debug_library():
    """Route every call of this module through librnl_debug.so (the build with
    device-side bounds checks, ``python -m rmsnorm_linear_projection_gb300.build
    --debug``) while the context is open; yields that library."""
    global _lib
    dbg = load(DEBUG_LIB_PATH)
    with _lock:
        prev, _lib = _lib, dbg
    try:
        yield dbg
    finally:
        with _lock:
            _lib = prev


def rnl_debug_build() -> bool:
    """Whether the library in use is the debug build (bounds-checked kernels)."""
    return bool(load().rnl_debug_build())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream):
    """The stream handle for a call on `device`.  The C entry points work on the
    current CUDA device (its kernels, its cached set-up), so tensors on
    another device are refused here rather than handed over."""
    if device.type != "cuda":
        raise ValueError(f"tensors must be on a CUDA device, got {device}")
    cur = torch.cuda.current_device()
    if device.index is not None and device.index != cur:
        raise ValueError(f"tensors are on {device} but the current CUDA device is cuda:{cur}; "
                         f"make the call under torch.cuda.device({device})")
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != 0:
        raise RnlError(status, what)


def _need(t, name, dtype, shape, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def workspace_size(op: int, T: int, K: int, N: int, N2: int = 0) -> int:
    v = load().rnl_workspace_size(op, T, K, N, N2)
    if v == ctypes.c_size_t(-1).value:
        raise RnlError(2, "rnl_workspace_size")
    return int(v)


def _workspace(nbytes, device, given):
    if given is not None:
        return given
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def rmsnorm_linear_bf16(x, gamma, W, eps=1e-6, norm_mode=NORM_RSQRT, out=None,
                        out_dtype=OUT_BF16, workspace=None, stream=None):
    """AT-10 RMSNorm + Linear (bf16 out), or the mhc_pre FP32 form (fp32 out)."""
    T, K = x.shape
    N = W.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(W, "W", torch.bfloat16, (N, K), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (K,), dev)
    odt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if out is None:
        out = torch.empty((T, N), dtype=odt, device=dev)
    _need(out, "out", odt, (T, N), dev)
    ws = _workspace(workspace_size(OP_BF16, T, K, N, out_dtype), dev, workspace)
    _check(load().rmsnorm_linear_bf16(_ptr(x), _ptr(gamma), _ptr(W), T, K, N, float(eps),
                                      int(norm_mode), _ptr(out), int(out_dtype), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(dev, stream)),
           "rmsnorm_linear_bf16")
    return out


def rmsnorm_linear_bf16_ex(x, gamma, W, residual=None, x_sum_out=None, beta=None, bias=None,
                           eps=1e-6, norm_mode=NORM_RSQRT, out=None, rstd_out=None,
                           workspace=None, stream=None):
    """AT-10 with the residual add (x_add = bf16(x + residual)), the AT-03
    norm bias beta and output_rstd, and the AT-09 projection bias; bf16 out.
    x_sum_out may be x or residual (in-place add)."""
    T, K = x.shape
    N = W.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(W, "W", torch.bfloat16, (N, K), dev)
    for t, name, shape in ((residual, "residual", (T, K)), (x_sum_out, "x_sum_out", (T, K)),
                           (gamma, "gamma", (K,)), (beta, "beta", (K,)), (bias, "bias", (N,))):
        if t is not None:
            _need(t, name, torch.bfloat16, shape, dev)
    if rstd_out is not None:
        _need(rstd_out, "rstd_out", torch.float32, (T,), dev)
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (T, N), dev)
    ws = _workspace(workspace_size(OP_BF16, T, K, N, OUT_BF16), dev, workspace)
    _check(load().rmsnorm_linear_bf16_ex(_ptr(x), _ptr(residual), _ptr(x_sum_out), _ptr(gamma),
                                         _ptr(beta), _ptr(W), _ptr(bias), T, K, N, float(eps),
                                         int(norm_mode), _ptr(out), _ptr(rstd_out), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream(dev, stream)),
           "rmsnorm_linear_bf16_ex")
    return out


def _qkv_outputs(T, Hq, Hkv, D, dev, q_out, k_out, v_out):
    q_out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev) if q_out is None else q_out
    k_out = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev) if k_out is None else k_out
    v_out = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev) if v_out is None else v_out
    _need(q_out, "q_out", torch.bfloat16, (T, Hq, D), dev)
    _need(k_out, "k_out", torch.bfloat16, (T, Hkv, D), dev)
    _need(v_out, "v_out", torch.bfloat16, (T, Hkv, D), dev)
    return q_out, k_out, v_out


def rnl_qkv_rope(y, n_q_heads, n_kv_heads, head_dim, q_gamma, k_gamma, positions, cos_sin,
                 eps=1e-6, q_out=None, k_out=None, v_out=None, stream=None):
    """QKV split + per-head RMSNorm + RoPE of a bf16 projection output y
    [T, (Hq + 2 Hkv) * D]; returns (q, k, v)."""
    T = y.shape[0]
    Hq, Hkv, D = n_q_heads, n_kv_heads, head_dim
    dev = y.device
    _need(y, "y", torch.bfloat16, (T, (Hq + 2 * Hkv) * D), dev)
    _need(q_gamma, "q_gamma", torch.bfloat16, (D,), dev)
    _need(k_gamma, "k_gamma", torch.bfloat16, (D,), dev)
    _need(positions, "positions", torch.int32, (T,), dev)
    P = cos_sin.shape[0]
    _need(cos_sin, "cos_sin", torch.float32, (P, D), dev)
    q_out, k_out, v_out = _qkv_outputs(T, Hq, Hkv, D, dev, q_out, k_out, v_out)
    _check(load().rnl_qkv_rope(_ptr(y), T, Hq, Hkv, D, _ptr(q_gamma), _ptr(k_gamma), float(eps),
                               _ptr(positions), _ptr(cos_sin), P, _ptr(q_out), _ptr(k_out),
                               _ptr(v_out), _stream(dev, stream)), "rnl_qkv_rope")
    return q_out, k_out, v_out


def rmsnorm_linear_qkv_rope(x, gamma, W, n_q_heads, n_kv_heads, head_dim, q_gamma, k_gamma,
                            positions, cos_sin, eps=1e-6, norm_mode=NORM_RSQRT, head_eps=1e-6,
                            q_out=None, k_out=None, v_out=None, workspace=None, stream=None):
    """AT-10 RMSNorm + Linear into the qkv projection, then the QKV split +
    per-head RMSNorm + RoPE stage; returns (q, k, v)."""
    T, K = x.shape
    Hq, Hkv, D = n_q_heads, n_kv_heads, head_dim
    N = (Hq + 2 * Hkv) * D
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(W, "W", torch.bfloat16, (N, K), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (K,), dev)
    _need(q_gamma, "q_gamma", torch.bfloat16, (D,), dev)
    _need(k_gamma, "k_gamma", torch.bfloat16, (D,), dev)
    _need(positions, "positions", torch.int32, (T,), dev)
    P = cos_sin.shape[0]
    _need(cos_sin, "cos_sin", torch.float32, (P, D), dev)
    q_out, k_out, v_out = _qkv_outputs(T, Hq, Hkv, D, dev, q_out, k_out, v_out)
    ws = _workspace(workspace_size(OP_QKV_ROPE, T, K, N), dev, workspace)
    _check(load().rmsnorm_linear_qkv_rope(_ptr(x), _ptr(gamma), _ptr(W), T, K, Hq, Hkv, D,
                                          float(eps), int(norm_mode), _ptr(q_gamma), _ptr(k_gamma),
                                          float(head_eps), _ptr(positions), _ptr(cos_sin), P,
                                          _ptr(q_out), _ptr(k_out), _ptr(v_out), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(dev, stream)),
           "rmsnorm_linear_qkv_rope")
    return q_out, k_out, v_out


def quant_matmul_reduce_sum(x1, x2, x1_scale, x2_scale, out=None, workspace=None, stream=None):
    """QuantMatMulReduceSum: exact int8 matmuls x1[b] @ x2[b] (x1 [B,M,K],
    x2 [B,K,N]), dequantised with x1_scale [B,M] (fp32) and x2_scale [N]
    (bf16) and summed over the batch in FP32; bf16 out [M, N]."""
    B, M, K = x1.shape
    N = x2.shape[2]
    dev = x1.device
    _need(x1, "x1", torch.int8, (B, M, K), dev)
    _need(x2, "x2", torch.int8, (B, K, N), dev)
    _need(x1_scale, "x1_scale", torch.float32, (B, M), dev)
    _need(x2_scale, "x2_scale", torch.bfloat16, (N,), dev)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (M, N), dev)
    ws = _workspace(workspace_size(OP_QMRS, M, K, N, B), dev, workspace)
    _check(load().quant_matmul_reduce_sum(_ptr(x1), _ptr(x2), _ptr(x1_scale), _ptr(x2_scale), B, M, K, N,
                                          _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(dev, stream)),
           "quant_matmul_reduce_sum")
    return out


def rmsnorm_linear_w8a8(x, gamma, Wq, w_scale, eps=1e-6, norm_mode=NORM_RSQRT, out=None,
                        q_out=None, x_scale_out=None, workspace=None, stream=None):
    """AT-11 RMSNorm + per-token INT8 quant + exact INT8 matmul + dequant (bf16 out)."""
    T, K = x.shape
    N = Wq.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(Wq, "Wq", torch.int8, (N, K), dev)
    _need(w_scale, "w_scale", torch.float32, (N,), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (K,), dev)
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (T, N), dev)
    if q_out is not None:
        _need(q_out, "q_out", torch.int8, (T, K), dev)
    if x_scale_out is not None:
        _need(x_scale_out, "x_scale_out", torch.float32, (T,), dev)
    ws = _workspace(workspace_size(OP_W8A8, T, K, N), dev, workspace)
    _check(load().rmsnorm_linear_w8a8(_ptr(x), _ptr(gamma), _ptr(Wq), _ptr(w_scale), T, K, N,
                                      float(eps), int(norm_mode), _ptr(out), _ptr(q_out),
                                      _ptr(x_scale_out), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(dev, stream)),
           "rmsnorm_linear_w8a8")
    return out


def rnl_w8a8_prepare_weight(Wq, out=None, stream=None):
    """The W8A8 weight prepared once: int8 Wq [N, K] widened exactly to the
    bf16 operand [N, K] that rmsnorm_linear_w8a8_prepared reads."""
    N, K = Wq.shape
    dev = Wq.device
    _need(Wq, "Wq", torch.int8, (N, K), dev)
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    _need(out, "Wb", torch.bfloat16, (N, K), dev)
    _check(load().rnl_w8a8_prepare_weight(_ptr(Wq), N, K, _ptr(out), _stream(dev, stream)),
           "rnl_w8a8_prepare_weight")
    return out


def rmsnorm_linear_w8a8_prepared(x, gamma, Wb, w_scale, eps=1e-6, norm_mode=NORM_RSQRT, out=None,
                                 q_out=None, x_scale_out=None, workspace=None, stream=None):
    """rmsnorm_linear_w8a8 with the weight from rnl_w8a8_prepare_weight (bf16 [N, K])."""
    T, K = x.shape
    N = Wb.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(Wb, "Wb", torch.bfloat16, (N, K), dev)
    _need(w_scale, "w_scale", torch.float32, (N,), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (K,), dev)
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (T, N), dev)
    if q_out is not None:
        _need(q_out, "q_out", torch.int8, (T, K), dev)
    if x_scale_out is not None:
        _need(x_scale_out, "x_scale_out", torch.float32, (T,), dev)
    ws = _workspace(workspace_size(OP_W8A8_PREPARED, T, K, N), dev, workspace)
    _check(load().rmsnorm_linear_w8a8_prepared(_ptr(x), _ptr(gamma), _ptr(Wb), _ptr(w_scale), T, K, N,
                                               float(eps), int(norm_mode), _ptr(out), _ptr(q_out),
                                               _ptr(x_scale_out), _ptr(ws), ws.numel() * ws.element_size(),
                                               _stream(dev, stream)),
           "rmsnorm_linear_w8a8_prepared")
    return out


def rmsnorm_linear_mxfp8(x, gamma, w_codes, w_scale, eps=1e-6, norm_mode=NORM_RSQRT, block=64,
                         out=None, out_dtype=OUT_BF16, x_codes_out=None, x_scale_out=None,
                         workspace=None, stream=None):
    """AT-11 in MXFP8 mode: RMSNorm, MX quantisation of the rows, scaled_mm
    against E4M3 weight codes [N, K] with E8M0 scale bytes [N, K / block]."""
    T, K = x.shape
    N = w_codes.shape[0]
    dev = x.device
    nb = K // block if block else 0
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(w_codes, "w_codes", torch.uint8, (N, K), dev)
    _need(w_scale, "w_scale", torch.uint8, (N, nb), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (K,), dev)
    odt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if out is None:
        out = torch.empty((T, N), dtype=odt, device=dev)
    _need(out, "out", odt, (T, N), dev)
    if x_codes_out is not None:
        _need(x_codes_out, "x_codes_out", torch.uint8, (T, K), dev)
    if x_scale_out is not None:
        _need(x_scale_out, "x_scale_out", torch.uint8, (T, nb), dev)
    ws = _workspace(workspace_size(OP_MXFP8, T, K, N), dev, workspace)
    _check(load().rmsnorm_linear_mxfp8(_ptr(x), _ptr(gamma), _ptr(w_codes), _ptr(w_scale), T, K, N,
                                       float(eps), int(norm_mode), int(block), _ptr(out), int(out_dtype),
                                       _ptr(x_codes_out), _ptr(x_scale_out), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(dev, stream)),
           "rmsnorm_linear_mxfp8")
    return out


def mxfp8_scaled_mm(x_codes, x_scale, w_codes, w_scale, block=64, out=None, out_dtype=OUT_BF16,
                    workspace=None, stream=None):
    """scaled_mm(x_fp8, w_fp8, FP32, x_scale, w_scale) on MXFP8 operands."""
    T, K = x_codes.shape
    N = w_codes.shape[0]
    dev = x_codes.device
    nb = K // block if block else 0
    _need(x_codes, "x_codes", torch.uint8, (T, K), dev)
    _need(x_scale, "x_scale", torch.uint8, (T, nb), dev)
    _need(w_codes, "w_codes", torch.uint8, (N, K), dev)
    _need(w_scale, "w_scale", torch.uint8, (N, nb), dev)
    odt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if out is None:
        out = torch.empty((T, N), dtype=odt, device=dev)
    _need(out, "out", odt, (T, N), dev)
    ws = _workspace(workspace_size(OP_MXFP8, T, K, N), dev, workspace)
    _check(load().mxfp8_scaled_mm(_ptr(x_codes), _ptr(x_scale), _ptr(w_codes), _ptr(w_scale), T, K, N,
                                  int(block), _ptr(out), int(out_dtype), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(dev, stream)),
           "mxfp8_scaled_mm")
    return out


def rnl_head_rmsnorm(y, n_heads, head_dim, gamma=None, eps=1e-6, norm_mode=NORM_RSQRT, out=None,
                     stream=None):
    """Per-head RMSNorm of y [T, n_heads * head_dim] (bf16); out may be y (in place)."""
    T = y.shape[0]
    dev = y.device
    _need(y, "y", torch.bfloat16, (T, n_heads * head_dim), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (head_dim,), dev)
    if out is None:
        out = torch.empty_like(y)
    _need(out, "out", torch.bfloat16, (T, n_heads * head_dim), dev)
    _check(load().rnl_head_rmsnorm(_ptr(y), T, n_heads, head_dim, _ptr(gamma), float(eps), int(norm_mode),
                                   _ptr(out), _stream(dev, stream)),
           "rnl_head_rmsnorm")
    return out


def mla_q_chain_head_norm(x, W_qa, gamma_cq, W_qb, head_dim, head_gamma=None, eps=1e-6,
                          norm_mode=NORM_SQRT_DIV, head_eps=1e-6, out=None, qa_out=None,
                          workspace=None, stream=None):
    """MLA q chain, then the per-head RMSNorm of its output (in place)."""
    T, K = x.shape
    N1, N2 = W_qa.shape[0], W_qb.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(W_qa, "W_qa", torch.bfloat16, (N1, K), dev)
    _need(gamma_cq, "gamma_cq", torch.bfloat16, (N1,), dev)
    _need(W_qb, "W_qb", torch.bfloat16, (N2, N1), dev)
    if head_gamma is not None:
        _need(head_gamma, "head_gamma", torch.bfloat16, (head_dim,), dev)
    if out is None:
        out = torch.empty((T, N2), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (T, N2), dev)
    if qa_out is not None:
        _need(qa_out, "qa_out", torch.bfloat16, (T, N1), dev)
    ws = _workspace(workspace_size(OP_MLA, T, K, N1, N2), dev, workspace)
    _check(load().mla_q_chain_head_norm(_ptr(x), _ptr(W_qa), _ptr(gamma_cq), _ptr(W_qb), T, K, N1, N2,
                                        float(eps), int(norm_mode), int(head_dim), _ptr(head_gamma),
                                        float(head_eps), _ptr(out), _ptr(qa_out), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(dev, stream)),
           "mla_q_chain_head_norm")
    return out


def mla_q_chain(x, W_qa, gamma_cq, W_qb, eps=1e-6, norm_mode=NORM_SQRT_DIV, out=None,
                qa_out=None, workspace=None, stream=None):
    """MLA two-stage q chain: q_a projection -> RMSNorm * gamma_cq -> q_b projection."""
    T, K = x.shape
    N1, N2 = W_qa.shape[0], W_qb.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(W_qa, "W_qa", torch.bfloat16, (N1, K), dev)
    _need(gamma_cq, "gamma_cq", torch.bfloat16, (N1,), dev)
    _need(W_qb, "W_qb", torch.bfloat16, (N2, N1), dev)
    if out is None:
        out = torch.empty((T, N2), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (T, N2), dev)
    if qa_out is not None:
        _need(qa_out, "qa_out", torch.bfloat16, (T, N1), dev)
    ws = _workspace(workspace_size(OP_MLA, T, K, N1, N2), dev, workspace)
    _check(load().mla_q_chain(_ptr(x), _ptr(W_qa), _ptr(gamma_cq), _ptr(W_qb), T, K, N1, N2,
                              float(eps), int(norm_mode), _ptr(out), _ptr(qa_out), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(dev, stream)),
           "mla_q_chain")
    return out


def rmsnorm_linear_skinny_noalloc(x, W, eps=1e-6, norm_mode=NORM_RSQRT, out=None, stream=None):
    """mhc_pre FP32 form (no gamma, N <= 64) with no workspace: for callers that
    cannot allocate device memory.  The scratch is an array built into the
    library, shared by every call on the device (overlapping calls race)."""
    T, K = x.shape
    N = W.shape[0]
    dev = x.device
    _need(x, "x", torch.bfloat16, (T, K), dev)
    _need(W, "W", torch.bfloat16, (N, K), dev)
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, (T, N), dev)
    _check(load().rmsnorm_linear_skinny_noalloc(_ptr(x), _ptr(W), T, K, N, float(eps),
                                                int(norm_mode), _ptr(out), _stream(dev, stream)),
           "rmsnorm_linear_skinny_noalloc")
    return out


def rnl_gemm_s8s8s32(A, B, out=None, workspace=None, stream=None):
    """Exact int8 x int8 -> int32 matmul C = A @ B^T (the W8A8 matmul on its own)."""
    M, K = A.shape
    N = B.shape[0]
    dev = A.device
    _need(A, "A", torch.int8, (M, K), dev)
    _need(B, "B", torch.int8, (N, K), dev)
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=dev)
    _need(out, "C", torch.int32, (M, N), dev)
    ws = _workspace(workspace_size(OP_GEMM_S8, M, K, N), dev, workspace)
    _check(load().rnl_gemm_s8s8s32(_ptr(A), _ptr(B), _ptr(out), M, N, K, _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(dev, stream)),
           "rnl_gemm_s8s8s32")
    return out


def rnl_selftest_wait_timeout(stream=None, device=None):
    """Enqueue the failure-detection self-test (a 1 ms bounded wait that must give up)."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    _check(load().rnl_selftest_wait_timeout(_stream(dev, stream)), "rnl_selftest_wait_timeout")


def rnl_selftest_bounds_check(stream=None, device=None):
    """Enqueue the debug build's bounds-check self-test (a check that must fail
    on an index that still lies inside the kernel's own array); raises
    RnlError(RNL_ERR_UNSUPPORTED) on a release build."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    _check(load().rnl_selftest_bounds_check(_stream(dev, stream)), "rnl_selftest_bounds_check")


def rnl_check_device_error(stream=None, device=None):
    """Synchronise and read the device error words; raises RnlError on a timeout."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    site = ctypes.c_int(0)
    st = load().rnl_check_device_error(_stream(dev, stream), ctypes.byref(site))
    if st != 0:
        raise RnlError(st, f"device error (site {site.value})")


def rnl_trace_enable(on: bool = True):
    _check(load().rnl_trace_enable(1 if on else 0), "rnl_trace_enable")


def rnl_trace_read(max_records: int = 16384):
    """[(kernel name, milliseconds)] of the launches traced since the last read."""
    names = (ctypes.c_char * 32 * max_records)()
    ms = (ctypes.c_float * max_records)()
    n = load().rnl_trace_read(ctypes.cast(names, ctypes.c_void_p), ms, max_records)
    return [(bytes(names[i]).split(b"\0", 1)[0].decode(), float(ms[i])) for i in range(n)]


# ---------------------------------------------------------------- host-buffer pipeline
class PipelineHandle:
    """An rnl_pipeline* plus the sizes it was created for."""

    def __init__(self, ptr, op, T, K, N, N2, device):
        self.ptr, self.op, self.T, self.K, self.N, self.N2, self.device = ptr, op, T, K, N, N2, device

    def out_shape_dtype(self):
        if self.op == OP_MLA:
            return (self.T, self.N2), torch.bfloat16
        if self.op == OP_BF16 and self.N2 == OUT_FP32:
            return (self.T, self.N), torch.float32
        return (self.T, self.N), torch.bfloat16


def _host(t, name, dtype, shape):
    if t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned (page-locked) CPU tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")


def rnl_pipeline_create(op, T, K, N, N2=0, device=None):
    """Create a host-buffer pipeline on `device` (default: current) for calls of
    one op and size; N2 = out_dtype for OP_BF16, the stage-2 width for OP_MLA."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    ptr = ctypes.c_void_p(None)
    with torch.cuda.device(dev):
        _check(load().rnl_pipeline_create(int(op), T, K, N, N2, ctypes.byref(ptr)),
               "rnl_pipeline_create")
    return PipelineHandle(ptr, op, T, K, N, N2, dev)


def _submit(pipe, name, x_host, out_host, call):
    _host(x_host, "x_host", torch.bfloat16, (pipe.T, pipe.K))
    shape, dt = pipe.out_shape_dtype()
    _host(out_host, "out_host", dt, shape)
    ticket = ctypes.c_int64(-1)
    _check(call(ctypes.byref(ticket)), name)
    return ticket.value


def rnl_pipeline_submit_bf16(pipe, x_host, gamma, W, out_host, eps=1e-6, norm_mode=NORM_RSQRT):
    """Enqueue one rmsnorm_linear_bf16 call fed from pinned host x_host into
    pinned host out_host; returns its ticket."""
    dev = pipe.device
    _need(W, "W", torch.bfloat16, (pipe.N, pipe.K), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (pipe.K,), dev)
    return _submit(pipe, "rnl_pipeline_submit_bf16", x_host, out_host, lambda t: load().rnl_pipeline_submit_bf16(
        pipe.ptr, _ptr(x_host), _ptr(gamma), _ptr(W), float(eps), int(norm_mode), _ptr(out_host), t))


def rnl_pipeline_submit_w8a8(pipe, x_host, gamma, Wq, w_scale, out_host, eps=1e-6, norm_mode=NORM_RSQRT):
    """Enqueue one rmsnorm_linear_w8a8 call (host x_host -> host out_host)."""
    dev = pipe.device
    _need(Wq, "Wq", torch.int8, (pipe.N, pipe.K), dev)
    _need(w_scale, "w_scale", torch.float32, (pipe.N,), dev)
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (pipe.K,), dev)
    return _submit(pipe, "rnl_pipeline_submit_w8a8", x_host, out_host, lambda t: load().rnl_pipeline_submit_w8a8(
        pipe.ptr, _ptr(x_host), _ptr(gamma), _ptr(Wq), _ptr(w_scale), float(eps), int(norm_mode),
        _ptr(out_host), t))


def rnl_pipeline_submit_mla(pipe, x_host, W_qa, gamma_cq, W_qb, out_host, eps=1e-6, norm_mode=NORM_SQRT_DIV):
    """Enqueue one mla_q_chain call (host x_host -> host out_host)."""
    dev = pipe.device
    _need(W_qa, "W_qa", torch.bfloat16, (pipe.N, pipe.K), dev)
    _need(gamma_cq, "gamma_cq", torch.bfloat16, (pipe.N,), dev)
    _need(W_qb, "W_qb", torch.bfloat16, (pipe.N2, pipe.N), dev)
    return _submit(pipe, "rnl_pipeline_submit_mla", x_host, out_host, lambda t: load().rnl_pipeline_submit_mla(
        pipe.ptr, _ptr(x_host), _ptr(W_qa), _ptr(gamma_cq), _ptr(W_qb), float(eps), int(norm_mode),
        _ptr(out_host), t))


def rnl_pipeline_wait(pipe, ticket):
    """Block until call `ticket` has written its host output; raises RnlError on a
    device timeout."""
    site = ctypes.c_int(0)
    st = load().rnl_pipeline_wait(pipe.ptr, int(ticket), ctypes.byref(site))
    if st != 0:
        raise RnlError(st, f"rnl_pipeline_wait (wait site {site.value})")


def rnl_pipeline_destroy(pipe):
    """Wait for all submitted calls and free the pipeline."""
    if pipe.ptr:
        _check(load().rnl_pipeline_destroy(pipe.ptr), "rnl_pipeline_destroy")
        pipe.ptr = ctypes.c_void_p(None)
