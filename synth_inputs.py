"""Seeded synthetic inputs for the fused RMSNorm -> Linear projection.

This module is the one thing the CPU oracle (``oracle/``) and the CUDA path
(``rmsnorm_linear_projection_gb300``) have in common: both are fed the bytes
it produces.  It holds none of the method's arithmetic (no norm, no
quantisation, no matmul); it only draws numbers and stores them in the
formats the operators take (bf16 bit patterns as ``uint16``, int8, fp32).

Every value is a pure function of ``(seed, tensor name, flat index)``: a
counter-based generator (the SplitMix64 output function applied to a Weyl
sequence, Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014).  So any subset of rows can be drawn without the
rest, the same bytes come out on x86 and on Arm, and nothing depends on a
library's RNG version.

Workload recipes (shapes and distributions of the five projection cases):

* ``tiny``   x[16,256] ~N(0,1), gamma[256] ~U(0.5,1.5), W[128,256] ~N(0,0.02),
             eps 1e-6, rsqrt form, bf16 out.
* ``qkv``    x[4096,4096] ~N(0,1), gamma ~U(0.5,1.5), W[6144,4096] ~N(0,0.02),
             eps 1e-6, rsqrt form, bf16 out (pre-attention fused QKV).
* ``mla``    x[2048,7168] ~N(0,1), W_qa[1536,7168], gamma_cq[1536] ~U(0.5,1.5),
             W_qb[24576,1536], weights ~N(0,0.02), eps 1e-6, sqrt+div form.
* ``w8a8``   x[8192,4096] ~N(0,1) with each entry independently (p=0.01)
             multiplied by 20, gamma ~U(0.5,1.5), Wq[4096,4096] int8 uniform
             on [-127,127], w_scale[4096] fp32 ~U(1e-3,1e-2), eps 1e-6.
* ``skinny`` x[16384,28672] ~N(0,1), no gamma, W[24,28672] ~N(0,0.02),
             eps 1e-6, rsqrt form, fp32 out (mhc_pre-style).
* ``decode`` x[4,4096] ~N(0,1), gamma ~U(0.5,1.5), W[6144,4096] ~N(0,0.02): a decode
             step of 4 tokens through the qkv weight, eps 1e-6, rsqrt form, bf16 out.
* ``mxfp8``  x[4096,4096] ~N(0,1), gamma ~U(0.5,1.5), an MXFP8 weight [6144,4096]
             drawn directly as bytes: E4M3 codes with uniform sign, exponent
             field uniform on [10, 15] and mantissa uniform (the NaN pattern
             replaced by the largest finite magnitude), E8M0 scale bytes
             uniform on [113, 114] per block of 64 (|w| mostly 2^-10 .. 0.05),
             eps 1e-6, rsqrt form, bf16 out.
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO_POW_M53 = 1.0 / 9007199254740992.0

CONFIGS = {
    "tiny": dict(T=16, K=256, N=128, eps=1e-6, norm_mode=0, has_gamma=True,
                 out_dtype="bf16", seed=1000),
    "qkv": dict(T=4096, K=4096, N=6144, eps=1e-6, norm_mode=0, has_gamma=True,
                out_dtype="bf16", seed=1001),
    "mla": dict(T=2048, K=7168, N1=1536, N2=24576, eps=1e-6, norm_mode=1,
                seed=1002),
    "w8a8": dict(T=8192, K=4096, N=4096, eps=1e-6, norm_mode=0, has_gamma=True,
                 seed=1003),
    "skinny": dict(T=16384, K=28672, N=24, eps=1e-6, norm_mode=0,
                   has_gamma=False, out_dtype="fp32", seed=1004),
    # QuantMatMulReduceSum: a batch of 4 exact int8 matmuls, summed (the
    # pages give no sizes; 275 GOP like the W8A8 workload)
    "qmrs": dict(B=4, M=2048, K=4096, N=4096, seed=1005),
    # the qkv projection followed by the QKV split + per-head RMSNorm + RoPE
    # stage (Qwen3 layout: 32 query heads and 8 key/value heads of 128)
    # a decode step: 4 tokens through the qkv weight (bound by reading W once)
    "decode": dict(T=4, K=4096, N=6144, eps=1e-6, norm_mode=0, has_gamma=True,
                   out_dtype="bf16", seed=1007),
    # the qkv projection shape in MXFP8 mode (one E8M0 scale per 64 elements)
    "mxfp8": dict(T=4096, K=4096, N=6144, eps=1e-6, norm_mode=0, has_gamma=True,
                  out_dtype="bf16", block=64, seed=1006),
    "qkv_rope": dict(T=4096, K=4096, N=6144, eps=1e-6, norm_mode=0, has_gamma=True,
                     out_dtype="bf16", seed=1001, n_q_heads=32, n_kv_heads=8, head_dim=128,
                     head_eps=1e-6, max_pos=4096, rope_base=1.0e6),
}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, name: str) -> np.uint64:
    with np.errstate(over="ignore"):
        base = (np.uint64(seed) * _GOLDEN) ^ np.uint64(zlib.crc32(name.encode()))
        return _mix(np.array([base], dtype=np.uint64))[0]


def _bits(key: np.uint64, idx: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return _mix(key + (idx.astype(np.uint64) + np.uint64(1)) * _GOLDEN)


def _unit(key: np.uint64, idx: np.ndarray) -> np.ndarray:
    """Uniform doubles in the open interval (0, 1)."""
    return ((_bits(key, idx) >> np.uint64(11)).astype(np.float64) + 0.5) * _TWO_POW_M53


def _flat_index(rows: np.ndarray, cols: int) -> np.ndarray:
    return (rows.astype(np.int64)[:, None] * cols + np.arange(cols, dtype=np.int64)[None, :])


def _f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Store float32 values as bf16 bit patterns, round to nearest even.

    The synthetic values are finite and far from the bf16 overflow threshold.
    """
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _rows_arg(nrows: int, rows) -> np.ndarray:
    if rows is None:
        return np.arange(nrows, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= nrows):
        raise IndexError("row index out of range")
    return rows


def _chunked(fn, rows: np.ndarray, cols: int, dtype) -> np.ndarray:
    """Evaluate fn(row_block) -> [len(block), cols] over row blocks in threads."""
    out = np.empty((rows.size, cols), dtype=dtype)
    if rows.size == 0:
        return out
    per = max(1, (1 << 22) // max(cols, 1))
    blocks = [(s, min(s + per, rows.size)) for s in range(0, rows.size, per)]

    def run(b):
        s, e = b
        out[s:e] = fn(rows[s:e])

    if len(blocks) == 1:
        run(blocks[0])
    else:
        with ThreadPoolExecutor(max_workers=min(len(blocks), os.cpu_count() or 4)) as ex:
            list(ex.map(run, blocks))
    return out


def normal_bf16(seed: int, name: str, shape, sigma: float = 1.0, rows=None,
                outlier_p: float = 0.0, outlier_scale: float = 1.0) -> np.ndarray:
    """N(0, sigma^2) values (Box-Muller on two counter draws) as bf16 bits.

    With ``outlier_p`` > 0 each entry is independently, with that
    probability, multiplied by ``outlier_scale`` before the bf16 rounding.
    ``rows`` selects a subset of the rows of a 2-D tensor; the values are the
    same as in the full tensor.
    """
    shape = tuple(shape)
    nrows, cols = (shape[0], shape[1]) if len(shape) == 2 else (1, shape[0])
    r = _rows_arg(nrows, rows)
    k_u1, k_u2, k_o = _key(seed, name + "/u1"), _key(seed, name + "/u2"), _key(seed, name + "/outlier")

    def fn(rb):
        idx = _flat_index(rb, cols)
        u1, u2 = _unit(k_u1, idx), _unit(k_u2, idx)
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2) * sigma
        if outlier_p > 0.0:
            z = np.where(_unit(k_o, idx) < outlier_p, z * outlier_scale, z)
        return _f32_to_bf16_bits(z.astype(np.float32))

    out = _chunked(fn, r, cols, np.uint16)
    return out if len(shape) == 2 or rows is not None else out.reshape(shape)


def uniform_bf16(seed: int, name: str, shape, lo: float, hi: float) -> np.ndarray:
    shape = tuple(shape)
    n = int(np.prod(shape))
    u = _unit(_key(seed, name), np.arange(n, dtype=np.int64))
    return _f32_to_bf16_bits((lo + (hi - lo) * u).astype(np.float32)).reshape(shape)


def uniform_f32(seed: int, name: str, shape, lo: float, hi: float) -> np.ndarray:
    shape = tuple(shape)
    n = int(np.prod(shape))
    u = _unit(_key(seed, name), np.arange(n, dtype=np.int64))
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def uniform_int8(seed: int, name: str, shape, lo: int = -127, hi: int = 127, rows=None) -> np.ndarray:
    """Integers uniform on [lo, hi] as int8."""
    shape = tuple(shape)
    nrows, cols = shape
    r = _rows_arg(nrows, rows)
    key = _key(seed, name)
    span = hi - lo + 1

    def fn(rb):
        u = _unit(key, _flat_index(rb, cols))
        return (np.floor(u * span).astype(np.int64) + lo).clip(lo, hi).astype(np.int8)

    return _chunked(fn, r, cols, np.int8)


def uniform_u8(seed: int, name: str, shape, lo: int, hi: int, rows=None) -> np.ndarray:
    """Integers uniform on [lo, hi] as uint8."""
    shape = tuple(shape)
    nrows, cols = shape
    r = _rows_arg(nrows, rows)
    key = _key(seed, name)
    span = hi - lo + 1

    def fn(rb):
        u = _unit(key, _flat_index(rb, cols))
        return (np.floor(u * span).astype(np.int64) + lo).clip(lo, hi).astype(np.uint8)

    return _chunked(fn, r, cols, np.uint8)


def e4m3_codes(seed: int, name: str, shape, e_lo: int = 10, rows=None) -> np.ndarray:
    """E4M3FN bytes drawn field by field: sign uniform, exponent field uniform
    on [e_lo, 15], mantissa uniform on [0, 7]; the NaN pattern (exponent 15,
    mantissa 7) becomes mantissa 6 (the largest finite magnitude)."""
    shape = tuple(shape)
    nrows, cols = shape
    r = _rows_arg(nrows, rows)
    key = _key(seed, name)
    span = np.uint64(16 - e_lo)

    def fn(rb):
        b = _bits(key, _flat_index(rb, cols))
        sign = (b & np.uint64(1)).astype(np.uint8)
        mant = ((b >> np.uint64(1)) & np.uint64(7)).astype(np.uint8)
        e = ((b >> np.uint64(4)) % span).astype(np.uint8) + np.uint8(e_lo)
        mant = np.where((e == 15) & (mant == 7), np.uint8(6), mant)
        return (sign << np.uint8(7)) | (e << np.uint8(3)) | mant

    return _chunked(fn, r, cols, np.uint8)


# ---------------------------------------------------------------------------
# The five workloads.  Each returns a dict of numpy arrays; ``rows`` (optional)
# restricts the activation to a subset of its rows (weights are always full).
# ---------------------------------------------------------------------------

def make_projection(cfg: dict, rows=None, with_x: bool = True) -> dict:
    """x, gamma (or None), W for the bf16 / fp32-out projection workloads."""
    s, T, K, N = cfg["seed"], cfg["T"], cfg["K"], cfg["N"]
    d = {}
    if with_x:
        d["x"] = normal_bf16(s, "x", (T, K), 1.0, rows=rows)
    d["gamma"] = uniform_bf16(s, "gamma", (K,), 0.5, 1.5) if cfg.get("has_gamma", True) else None
    d["W"] = normal_bf16(s, "W", (N, K), 0.02)
    return d


def make_mla(cfg: dict, rows=None, with_x: bool = True) -> dict:
    s, T, K, N1, N2 = cfg["seed"], cfg["T"], cfg["K"], cfg["N1"], cfg["N2"]
    d = {}
    if with_x:
        d["x"] = normal_bf16(s, "x", (T, K), 1.0, rows=rows)
    d["W_qa"] = normal_bf16(s, "W_qa", (N1, K), 0.02)
    d["gamma_cq"] = uniform_bf16(s, "gamma_cq", (N1,), 0.5, 1.5)
    d["W_qb"] = normal_bf16(s, "W_qb", (N2, N1), 0.02)
    return d


def make_w8a8(cfg: dict, rows=None, with_x: bool = True) -> dict:
    s, T, K, N = cfg["seed"], cfg["T"], cfg["K"], cfg["N"]
    d = {}
    if with_x:
        d["x"] = normal_bf16(s, "x", (T, K), 1.0, rows=rows, outlier_p=0.01, outlier_scale=20.0)
    d["gamma"] = uniform_bf16(s, "gamma", (K,), 0.5, 1.5)
    d["Wq"] = uniform_int8(s, "Wq", (N, K), -127, 127)
    d["w_scale"] = uniform_f32(s, "w_scale", (N,), 1e-3, 1e-2)
    return d


def make_mxfp8(cfg: dict, rows=None, with_x: bool = True) -> dict:
    """x, gamma and the MXFP8 weight (codes [N, K], scale bytes [N, K/block])."""
    s, T, K, N, blk = cfg["seed"], cfg["T"], cfg["K"], cfg["N"], cfg.get("block", 64)
    d = {}
    if with_x:
        d["x"] = normal_bf16(s, "x", (T, K), 1.0, rows=rows)
    d["gamma"] = uniform_bf16(s, "gamma", (K,), 0.5, 1.5) if cfg.get("has_gamma", True) else None
    d["w_codes"] = e4m3_codes(s, "w_codes", (N, K))
    d["w_scale"] = uniform_u8(s, "w_scale", (N, K // blk), 113, 114)
    return d


def rope_table(P: int, D: int, base: float = 1.0e6) -> np.ndarray:
    """A rotary-embedding angle table, as a model precomputes it: fp32 [P, D],
    row p = [cos(p * f_0) .. cos(p * f_{D/2-1}), sin(p * f_0) .. sin(p * f_{D/2-1})]
    with f_i = base^(-2i/D) (base 1e6 as in Qwen3).  Computed in binary64 and
    rounded to fp32; both the oracle and the GPU path receive the same table."""
    i = np.arange(D // 2, dtype=np.float64)
    f = base ** (-2.0 * i / D)
    ang = np.arange(P, dtype=np.float64)[:, None] * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def make_qkv_rope(cfg: dict) -> dict:
    """Per-head norm weights, positions and angle table for the QKV split +
    per-head RMSNorm + RoPE stage after the qkv projection (Hq query heads,
    Hkv key/value heads of D; tokens of one sequence at positions 0..T-1)."""
    s, T, D = cfg["seed"], cfg["T"], cfg["head_dim"]
    return {
        "q_gamma": uniform_bf16(s, "q_gamma", (D,), 0.5, 1.5),
        "k_gamma": uniform_bf16(s, "k_gamma", (D,), 0.5, 1.5),
        "positions": (np.arange(T, dtype=np.int64) % cfg["max_pos"]).astype(np.int32),
        "cos_sin": rope_table(cfg["max_pos"], D, cfg.get("rope_base", 1.0e6)),
    }


def make_qmrs(cfg: dict, rows=None) -> dict:
    """QuantMatMulReduceSum operands: x1 int8 [B, M, K], x2 int8 [B, K, N]
    (uniform integers in [-127, 127]), x1_scale fp32 [B, M], x2_scale bf16 [N]
    (uniform in [1e-3, 1e-2]).  ``rows`` restricts x1 and x1_scale to a subset
    of M (the values are those of the full tensors)."""
    s, B, M, K, N = cfg["seed"], cfg["B"], cfg["M"], cfg["K"], cfg["N"]
    x1 = uniform_int8(s, "x1", (B * M, K), -127, 127).reshape(B, M, K)
    xs = uniform_f32(s, "x1_scale", (B, M), 1e-3, 1e-2)
    if rows is not None:
        x1, xs = x1[:, rows, :], xs[:, rows]
    return {
        "x1": x1,
        "x2": uniform_int8(s, "x2", (B * K, N), -127, 127).reshape(B, K, N),
        "x1_scale": xs,
        "x2_scale": uniform_bf16(s, "x2_scale", (N,), 1e-3, 1e-2),
    }


def scaled(cfg: dict, **over) -> dict:
    """A copy of a workload recipe with some sizes replaced (parity cases)."""
    c = dict(cfg)
    c.update(over)
    return c
