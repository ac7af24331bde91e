"""CPU oracle for the fused RMSNorm -> Linear projection (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never does.  The arithmetic lives in ``oracle.c`` (plain
loops, binary64; the W8A8 front end in binary32); this module compiles it
with gcc and marshals numpy arrays through ctypes.

Each wrapper cites the passage it follows in the docstring of the C function
it calls (``oracle.c``).  bf16 tensors are passed as uint16 bit patterns.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force in exact rational / integer
arithmetic, and library cross-checks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False, out_path: str | None = None, defines=()) -> str:
    """Compile oracle.c with gcc (about a second).  Returns the .so path."""
    path = out_path or _LIB_PATH
    os.makedirs(os.path.dirname(path), exist_ok=True)
    if (not force and not defines and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, *["-D" + d for d in defines], _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _declare(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    D = ctypes.c_double
    F = ctypes.c_float
    C = ctypes.c_int
    sigs = {
        "orc_bf16_rne": (ctypes.c_uint16, [D]),
        "orc_bf16_value": (D, [ctypes.c_uint16]),
        "orc_bf16_rne_array": (None, [P, I64, P]),
        "orc_threads": (C, []),
        "orc_set_threads": (None, [C]),
        "orc_rmsnorm_f64": (C, [P, P, I64, I64, D, C, P, P]),
        "orc_rmsnorm_linear": (C, [P, P, P, I64, I64, I64, D, C, C, P, P]),
        "orc_mla_q_chain": (C, [P, P, P, P, I64, I64, I64, I64, D, C, P, P, P]),
        "orc_rmsnorm_linear_ex": (C, [P, P, P, P, P, P, I64, I64, I64, D, C, P, P, P, P]),
        "orc_qkv_rope": (C, [P, I64, I64, I64, I64, P, P, D, P, P, I64, P, P, P]),
        "orc_quant_matmul_reduce_sum": (C, [P, P, P, P, I64, I64, I64, I64, P, P]),
        "orc_head_rmsnorm": (C, [P, I64, I64, I64, P, D, C, P]),
        "orc_e4m3_value": (D, [ctypes.c_uint8]),
        "orc_e4m3_rne_sat": (ctypes.c_uint8, [D]),
        "orc_e8m0_value": (D, [ctypes.c_uint8]),
        "orc_mxfp8_quant_rows": (C, [P, P, I64, I64, ctypes.c_float, C, I64, P, P]),
        "orc_mxfp8_scaled_mm": (C, [P, P, P, P, I64, I64, I64, I64, C, P, P]),
        "orc_quant_rows_f32": (C, [P, P, I64, I64, F, C, P, P, P, P]),
        "orc_gemm_s8": (C, [P, P, I64, I64, I64, P]),
        "orc_dequant_bf16": (C, [P, P, P, I64, I64, P, P]),
        "orc_rmsnorm_linear_w8a8": (C, [P, P, P, P, I64, I64, I64, F, C, P, P, P, P, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  ``path`` loads a variant."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(st, what):
    if st < 0:
        raise RuntimeError(f"oracle {what} failed with status {st}")
    return st


class Oracle:
    """Thin marshalling layer over one loaded copy of the C oracle."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    # -- bf16 codec ---------------------------------------------------------
    def bf16_rne(self, values) -> np.ndarray:
        v = _c(np.atleast_1d(values), np.float64)
        out = np.empty(v.shape, np.uint16)
        self.lib.orc_bf16_rne_array(_ptr(v), v.size, _ptr(out))
        return out

    def bf16_value(self, bits) -> np.ndarray:
        b = np.atleast_1d(np.asarray(bits, dtype=np.uint16))
        return np.array([self.lib.orc_bf16_value(int(h)) for h in b.ravel()]).reshape(b.shape)

    def threads(self) -> int:
        return int(self.lib.orc_threads())

    def set_threads(self, n: int) -> None:
        self.lib.orc_set_threads(int(n))

    # -- AT-03 --------------------------------------------------------------
    def rmsnorm_f64(self, x, gamma, eps, variant):
        x = _c(x, np.uint16)
        T, K = x.shape
        y = np.empty((T, K), np.float64)
        rstd = np.empty(T, np.float64)
        _check(self.lib.orc_rmsnorm_f64(_ptr(x), _ptr(_c(gamma, np.uint16)), T, K, float(eps),
                                        int(variant), _ptr(y), _ptr(rstd)), "rmsnorm")
        return y, rstd

    # -- AT-10 (form 0) and the mhc_pre FP32 form (form 1) --------------------
    def rmsnorm_linear(self, x, gamma, W, eps, variant, form):
        """Returns (ref, out): binary64 sums and the rounded output."""
        x, W = _c(x, np.uint16), _c(W, np.uint16)
        T, K = x.shape
        N = W.shape[0]
        assert W.shape[1] == K
        ref = np.empty((T, N), np.float64)
        out = np.empty((T, N), np.uint16 if form == 0 else np.float32)
        _check(self.lib.orc_rmsnorm_linear(_ptr(x), _ptr(_c(gamma, np.uint16)), _ptr(W), T, K, N,
                                           float(eps), int(variant), int(form), _ptr(ref),
                                           _ptr(out)), "rmsnorm_linear")
        return ref, out

    def rmsnorm_linear_ex(self, x, residual, gamma, beta, W, bias, eps, variant):
        """AT-10 with residual add, norm bias, projection bias; returns
        (ref, out, x_sum, rstd)."""
        x, W = _c(x, np.uint16), _c(W, np.uint16)
        T, K = x.shape
        N = W.shape[0]
        assert W.shape[1] == K
        res = _c(residual, np.uint16)
        assert res is None or res.shape == (T, K)
        ref = np.empty((T, N), np.float64)
        out = np.empty((T, N), np.uint16)
        x_sum = np.empty((T, K), np.uint16)
        rstd = np.empty((T,), np.float64)
        _check(self.lib.orc_rmsnorm_linear_ex(
            _ptr(x), _ptr(res), _ptr(_c(gamma, np.uint16)), _ptr(_c(beta, np.uint16)), _ptr(W),
            _ptr(_c(bias, np.uint16)), T, K, N, float(eps), int(variant), _ptr(ref), _ptr(out),
            _ptr(x_sum), _ptr(rstd)), "rmsnorm_linear_ex")
        return ref, out, x_sum, rstd

    def qkv_rope(self, y, Hq, Hkv, D, q_gamma, k_gamma, eps, pos, cs):
        """QKV split + per-head RMSNorm + RoPE of a projection output y (bf16
        bits [T, (Hq + 2 Hkv) D]); cs: fp32 [P, D] cos | sin table.  Returns
        (q, k, v) bf16 bits [T, H, D]."""
        y = _c(y, np.uint16)
        T = y.shape[0]
        assert y.shape[1] == (Hq + 2 * Hkv) * D
        pos = _c(pos, np.int32)
        cs = _c(cs, np.float32)
        q = np.empty((T, Hq, D), np.uint16)
        k = np.empty((T, Hkv, D), np.uint16)
        v = np.empty((T, Hkv, D), np.uint16)
        _check(self.lib.orc_qkv_rope(_ptr(y), T, Hq, Hkv, D, _ptr(_c(q_gamma, np.uint16)),
                                     _ptr(_c(k_gamma, np.uint16)), float(eps), _ptr(pos), _ptr(cs),
                                     cs.shape[0], _ptr(q), _ptr(k), _ptr(v)), "qkv_rope")
        return q, k, v

    def quant_matmul_reduce_sum(self, x1, x2, x1_scale, x2_scale):
        """QuantMatMulReduceSum: x1 int8 [B,M,K], x2 int8 [B,K,N], x1_scale fp32
        [B,M], x2_scale bf16 bits [N].  Returns (ref fp32 [M,N], out bf16 bits)."""
        x1, x2 = _c(x1, np.int8), _c(x2, np.int8)
        B, M, K = x1.shape
        N = x2.shape[2]
        assert x2.shape == (B, K, N)
        xs, ws = _c(x1_scale, np.float32), _c(x2_scale, np.uint16)
        assert xs.shape == (B, M) and ws.shape == (N,)
        ref = np.empty((M, N), np.float32)
        out = np.empty((M, N), np.uint16)
        st = self.lib.orc_quant_matmul_reduce_sum(_ptr(x1), _ptr(x2), _ptr(xs), _ptr(ws), B, M, K, N,
                                                  _ptr(ref), _ptr(out))
        _check(st, "quant_matmul_reduce_sum")
        if st == 1:
            raise OverflowError("int32 accumulator overflow")
        return ref, out

    # -- MXFP8 ----------------------------------------------------------------
    def e4m3_value(self, c):
        return self.lib.orc_e4m3_value(int(c))

    def e4m3_rne_sat(self, v):
        return int(self.lib.orc_e4m3_rne_sat(float(v)))

    def e8m0_value(self, s):
        return self.lib.orc_e8m0_value(int(s))

    def mxfp8_quant_rows(self, x, gamma, eps, variant, block=64):
        """E4M3 codes [T,K] (uint8) and E8M0 scale bytes [T, K/block]."""
        x = _c(x, np.uint16)
        T, K = x.shape
        codes = np.empty((T, K), np.uint8)
        scales = np.empty((T, K // block), np.uint8)
        _check(self.lib.orc_mxfp8_quant_rows(_ptr(x), _ptr(_c(gamma, np.uint16)), T, K, float(eps),
                                             int(variant), int(block), _ptr(codes), _ptr(scales)),
               "mxfp8_quant_rows")
        return codes, scales

    def mxfp8_scaled_mm(self, xq, xs, wq, ws, out_dtype=0, block=64):
        """(ref binary64 [T,N], out bf16 bits or fp32 [T,N])."""
        xq, xs, wq, ws = _c(xq, np.uint8), _c(xs, np.uint8), _c(wq, np.uint8), _c(ws, np.uint8)
        T, K = xq.shape
        N = wq.shape[0]
        ref = np.empty((T, N), np.float64)
        out = np.empty((T, N), np.uint16 if out_dtype == 0 else np.float32)
        _check(self.lib.orc_mxfp8_scaled_mm(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), T, K, N, int(block),
                                            int(out_dtype), _ptr(ref), _ptr(out)), "mxfp8_scaled_mm")
        return ref, out

    # -- MLA q chain ----------------------------------------------------------
    def head_rmsnorm(self, y, H, D, gamma, eps, variant):
        """Per-head RMSNorm of y (bf16 bits [T, H*D]): bf16 bits [T, H*D]."""
        y = _c(y, np.uint16)
        T = y.shape[0]
        assert y.shape[1] == H * D
        out = np.empty((T, H * D), np.uint16)
        _check(self.lib.orc_head_rmsnorm(_ptr(y), T, H, D, _ptr(_c(gamma, np.uint16)), float(eps),
                                         int(variant), _ptr(out)), "head_rmsnorm")
        return out

    def mla_q_chain(self, x, W_qa, gamma_cq, W_qb, eps, variant):
        """Returns (qa, ref, out)."""
        x, W_qa, W_qb = _c(x, np.uint16), _c(W_qa, np.uint16), _c(W_qb, np.uint16)
        g = _c(gamma_cq, np.uint16)
        T, K = x.shape
        N1, N2 = W_qa.shape[0], W_qb.shape[0]
        assert W_qa.shape[1] == K and W_qb.shape[1] == N1 and g.shape == (N1,)
        qa = np.empty((T, N1), np.uint16)
        ref = np.empty((T, N2), np.float64)
        out = np.empty((T, N2), np.uint16)
        _check(self.lib.orc_mla_q_chain(_ptr(x), _ptr(W_qa), _ptr(g), _ptr(W_qb), T, K, N1, N2,
                                        float(eps), int(variant), _ptr(qa), _ptr(ref), _ptr(out)),
               "mla_q_chain")
        return qa, ref, out

    # -- W8A8 ---------------------------------------------------------------
    def quant_rows_f32(self, x, gamma, eps, variant):
        """Returns (q int8 [T,K], x_scale fp32 [T], rstd fp32 [T], v fp32 [T,K]).

        v is y*qs before rounding (for checking near-tie codes)."""
        x = _c(x, np.uint16)
        T, K = x.shape
        q = np.empty((T, K), np.int8)
        xs = np.empty(T, np.float32)
        rstd = np.empty(T, np.float32)
        v = np.empty((T, K), np.float32)
        _check(self.lib.orc_quant_rows_f32(_ptr(x), _ptr(_c(gamma, np.uint16)), T, K,
                                           ctypes.c_float(eps), int(variant), _ptr(q), _ptr(xs),
                                           _ptr(rstd), _ptr(v)), "quant_rows_f32")
        return q, xs, rstd, v

    def gemm_s8(self, A, B):
        """Returns (C int32 [M,N], overflowed: bool)."""
        A, B = _c(A, np.int8), _c(B, np.int8)
        M, K = A.shape
        N = B.shape[0]
        assert B.shape[1] == K
        C = np.empty((M, N), np.int32)
        st = _check(self.lib.orc_gemm_s8(_ptr(A), _ptr(B), M, N, K, _ptr(C)), "gemm_s8")
        return C, st == 1

    def dequant_bf16(self, acc, x_scale, w_scale):
        acc = _c(acc, np.int32)
        M, N = acc.shape
        ref = np.empty((M, N), np.float64)
        out = np.empty((M, N), np.uint16)
        _check(self.lib.orc_dequant_bf16(_ptr(acc), _ptr(_c(x_scale, np.float32)),
                                         _ptr(_c(w_scale, np.float32)), M, N, _ptr(ref),
                                         _ptr(out)), "dequant_bf16")
        return ref, out

    def rmsnorm_linear_w8a8(self, x, gamma, Wq, w_scale, eps, variant):
        """Returns dict(q, x_scale, acc, ref, out, overflowed)."""
        x, Wq = _c(x, np.uint16), _c(Wq, np.int8)
        T, K = x.shape
        N = Wq.shape[0]
        q = np.empty((T, K), np.int8)
        xs = np.empty(T, np.float32)
        acc = np.empty((T, N), np.int32)
        ref = np.empty((T, N), np.float64)
        out = np.empty((T, N), np.uint16)
        st = _check(self.lib.orc_rmsnorm_linear_w8a8(
            _ptr(x), _ptr(_c(gamma, np.uint16)), _ptr(Wq), _ptr(_c(w_scale, np.float32)), T, K, N,
            ctypes.c_float(eps), int(variant), _ptr(q), _ptr(xs), _ptr(acc), _ptr(ref), _ptr(out)),
            "rmsnorm_linear_w8a8")
        return dict(q=q, x_scale=xs, acc=acc, ref=ref, out=out, overflowed=(st == 1))


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode bf16 bit patterns with numpy (bits << 16 reinterpreted as binary32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
