"""Helpers shared by the GPU parity tests: moving the generator's numpy
arrays to the device, the acceptance bounds, and row sampling."""
from __future__ import annotations

import numpy as np
import torch

from oracle import bf16_bits_to_f64

# Acceptance bound for bf16 outputs: |gpu - oracle| <= 1e-2 * max(1, |oracle|).
BF16_REL = 1e-2


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 device tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_bf16_close(gpu_bits: np.ndarray, oracle_bits: np.ndarray, what=""):
    g = bf16_bits_to_f64(gpu_bits)
    o = bf16_bits_to_f64(oracle_bits)
    assert g.shape == o.shape
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - o)
    bound = BF16_REL * np.maximum(1.0, np.abs(o))
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside bound; first at {tuple(i)}:"
                             f" gpu {g[tuple(i)]} oracle {o[tuple(i)]}; max err {err.max()}")
    return float(err.max())


def assert_fp32_close(gpu: np.ndarray, oracle_ref: np.ndarray, abs_sum: np.ndarray, what=""):
    """FP32-output bound derived from fp32 accumulation of K products:
    |gpu - ref| <= 2^-16 * sum_k |y_k w_k| + 2^-20 * |ref|."""
    g = gpu.astype(np.float64)
    err = np.abs(g - oracle_ref)
    bound = 2.0**-16 * abs_sum + 2.0**-20 * np.abs(oracle_ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outside bound; first at {tuple(i)}: gpu {g[tuple(i)]}"
                             f" oracle {oracle_ref[tuple(i)]} bound {bound[tuple(i)]}")
    return float((err / np.maximum(abs_sum, 1e-30)).max())


def sample_rows(T: int, n: int, seed: int = 0) -> np.ndarray:
    """First/last rows, tile edges and random rows (sorted, unique)."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, T // 2, T - 129, T - 128, T - 2, T - 1]
    rows = set(r for r in fixed if 0 <= r < T)
    while len(rows) < min(n, T):
        rows.add(int(rng.integers(0, T)))
    return np.array(sorted(rows), dtype=np.int64)
