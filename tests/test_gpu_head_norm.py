"""Per-head RMSNorm (rnl_head_rmsnorm) and the MLA chain with it
(mla_q_chain_head_norm) against the oracle.

Bounds, from the arithmetic.  The stage alone: the GPU's FP32 rstd differs
from the oracle's binary64 one by a few FP32 ulps, so a normalised value can
land on the other side of a bf16 rounding boundary: at most one bf16 ulp
apart when both sides see the same input.  The chain: the stage-2 output y
differs from the oracle's by the projection's error (FP32 accumulation, then
one bf16 rounding: at most one bf16 ulp of y where |y| is not tiny, an
absolute error of the accumulation where y is near zero after
cancellation); normalising scales that by rstd, and the final rounding adds
one ulp.  So each element is within the acceptance bound
1e-2 * max(1, |oracle|) (which covers the near-zero elements) or within two
bf16 ulps (which covers the larger normalised values, where two ulps can
exceed 1 % near the bottom of a binade).
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_bf16_close, dev_bf16, host_bits, sample_rows
from oracle import bf16_bits_to_f64

pytestmark = pytest.mark.gpu

rnl = pytest.importorskip("rmsnorm_linear_projection_gb300")


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_linear_projection_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    yield
    rnl.rnl_check_device_error()


def _ordered(bits):
    """bf16 bit patterns -> integers in the order of their values."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - b, b)


def assert_ulps(got, want, n, what):
    d = np.abs(_ordered(got) - _ordered(want))
    assert d.max() <= n, f"{what}: {int((d > n).sum())} elements more than {n} ulp apart (max {d.max()})"


def assert_chain_close(got, want, what):
    g, o = bf16_bits_to_f64(got), bf16_bits_to_f64(want)
    ok = (np.abs(g - o) <= 1e-2 * np.maximum(1.0, np.abs(o))) | (np.abs(_ordered(got) - _ordered(want)) <= 2)
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} outside both bounds"


@pytest.mark.parametrize("T,H,D,gamma,mode", [
    (37, 16, 192, False, 1),   # the MLA head width
    (50, 3, 64, True, 0),
    (9, 5, 512, True, 1),
    (1, 1, 128, False, 0),
    (130, 7, 320, True, 1),    # a group of 8 heads with a ragged tail, 5 words a lane
    (64, 9, 448, False, 0),
])
def test_head_norm_stage(orc, T, H, D, gamma, mode):
    y = si.normal_bf16(T + D, "y", (T, H * D), 1.5)
    y[0, :D] = si.normal_bf16(T + D, "quiet", (1, D), 1e-3)  # a quiet head beside loud ones
    g = si.uniform_bf16(D, "g", (D,), 0.5, 1.5) if gamma else None
    out = rnl.rnl_head_rmsnorm(dev_bf16(y), H, D, dev_bf16(g) if gamma else None, eps=1e-6, norm_mode=mode)
    want = orc.head_rmsnorm(y, H, D, g, 1e-6, mode)
    got = host_bits(out)
    assert_bf16_close(got, want, "head norm")
    assert_ulps(got, want, 1, "head norm")


def test_head_norm_in_place(orc):
    T, H, D = 40, 12, 192
    y = si.normal_bf16(5, "y", (T, H * D), 1.0)
    t = dev_bf16(y)
    out = rnl.rnl_head_rmsnorm(t, H, D, eps=1e-6, norm_mode=1, out=t)
    assert out.data_ptr() == t.data_ptr()
    assert_ulps(host_bits(t), orc.head_rmsnorm(y, H, D, None, 1e-6, 1), 1, "in place")


def test_mla_chain_head_norm_small(orc):
    T, K, N1, H, D = 300, 520, 128, 4, 192
    d = si.make_mla(dict(seed=51, T=T, K=K, N1=N1, N2=H * D))
    out = rnl.mla_q_chain_head_norm(dev_bf16(d["x"]), dev_bf16(d["W_qa"]), dev_bf16(d["gamma_cq"]),
                                    dev_bf16(d["W_qb"]), D, eps=1e-6, norm_mode=1)
    _, _, y = orc.mla_q_chain(d["x"], d["W_qa"], d["gamma_cq"], d["W_qb"], 1e-6, 1)
    want = orc.head_rmsnorm(y, H, D, None, 1e-6, 1)
    assert_chain_close(host_bits(out), want, "chain")


def test_mla_chain_head_norm_full_size_sampled(orc):
    """The MLA workload (2048 x 7168 -> 1536 -> 128 heads of 192) with the
    per-head norm, sampled rows against the oracle chain."""
    c = si.CONFIGS["mla"]
    d = si.make_mla(c)
    H, D = c["N2"] // 192, 192
    out = rnl.mla_q_chain_head_norm(dev_bf16(d["x"]), dev_bf16(d["W_qa"]), dev_bf16(d["gamma_cq"]),
                                    dev_bf16(d["W_qb"]), D, eps=c["eps"], norm_mode=c["norm_mode"])
    rows = sample_rows(c["T"], 12, seed=9)
    _, _, y = orc.mla_q_chain(d["x"][rows], d["W_qa"], d["gamma_cq"], d["W_qb"], c["eps"], c["norm_mode"])
    want = orc.head_rmsnorm(y, H, D, None, c["eps"], c["norm_mode"])
    got = host_bits(out)[rows]
    assert_chain_close(got, want, "full size")
    z = bf16_bits_to_f64(got).reshape(len(rows), H, D)
    assert np.allclose(np.sqrt((z * z).mean(axis=2)), 1.0, atol=0.01)  # every head normalised
