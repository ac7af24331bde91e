"""The GEMM on CTA pairs (tcgen05 cta_group::2, RNL_GEMM_PAIR=1) against the
oracle: bf16, fp32 row-scaled, exact int32 and dequant epilogues, ragged
tails, every output tile width, and a full-size sampled check."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_bf16_close, assert_fp32_close, dev, dev_bf16, host_bits, sample_rows
from oracle import bf16_bits_to_f64

pytestmark = pytest.mark.gpu

rnl = pytest.importorskip("rmsnorm_linear_projection_gb300")


@pytest.fixture(autouse=True)
def pair_mode(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("RNL_GEMM_PAIR", "1")
    yield
    rnl.rnl_check_device_error()


def _case(seed, T, K, N, gamma=True):
    return si.make_projection(dict(seed=seed, T=T, K=K, N=N, has_gamma=gamma))


@pytest.mark.parametrize("T,K,N", [(256, 64, 256), (300, 520, 600), (129, 4096, 256),
                                   (1000, 1024, 700), (16, 256, 128),
                                   (600, 3000, 1000)])  # 12 tiles in 5 k ranges: split-K pieces
def test_pair_bf16(orc, T, K, N):
    d = _case(T + K + N, T, K, N)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    assert_bf16_close(host_bits(out), want, f"pair bf16 {T}x{K}x{N}")


@pytest.mark.parametrize("bn", [128, 192, 256])
def test_pair_bf16_each_width(orc, monkeypatch, bn):
    monkeypatch.setenv("RNL_GEMM_BN", str(bn))
    d = _case(bn, 520, 1032, 777)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    assert_bf16_close(host_bits(out), want, f"pair bf16 BN={bn}")


def test_pair_fp32_rowscale(orc):
    d = _case(5, 500, 1024, 200, gamma=False)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), None, dev_bf16(d["W"]), out_dtype=rnl.OUT_FP32)
    ref, _ = orc.rmsnorm_linear(d["x"], None, d["W"], 1e-6, 0, 1)
    y, _ = orc.rmsnorm_f64(d["x"], None, 1e-6, 0)
    assert_fp32_close(out.cpu().numpy(), ref, np.abs(y) @ np.abs(bf16_bits_to_f64(d["W"])).T)


@pytest.mark.parametrize("bn", [128, 192, 256])
def test_pair_s8_bit_exact(orc, monkeypatch, bn):
    monkeypatch.setenv("RNL_GEMM_BN", str(bn))
    rng = np.random.default_rng(bn)
    A = rng.integers(-127, 128, (300, 4096)).astype(np.int8)
    B = rng.integers(-127, 128, (520, 4096)).astype(np.int8)
    C = rnl.rnl_gemm_s8s8s32(dev(A), dev(B)).cpu().numpy()
    want, _ = orc.gemm_s8(A, B)
    assert np.array_equal(C, want)


def test_pair_s8_worst_case(orc):
    M, N, K = 260, 260, 4096
    A = np.full((M, K), 127, np.int8)
    A[1::2] = -127
    B = np.full((N, K), 127, np.int8)
    B[::3] = -127
    C = rnl.rnl_gemm_s8s8s32(dev(A), dev(B)).cpu().numpy()
    want, _ = orc.gemm_s8(A, B)
    assert np.array_equal(C, want)


def test_pair_w8a8(orc):
    d = si.make_w8a8(dict(seed=9, T=300, K=2048, N=520))
    q = torch.empty((300, 2048), dtype=torch.int8, device="cuda")
    out = rnl.rmsnorm_linear_w8a8(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev(d["Wq"]),
                                  dev(d["w_scale"]), q_out=q)
    r = orc.rmsnorm_linear_w8a8(d["x"], d["gamma"], d["Wq"], d["w_scale"], 1e-6, 0)
    assert np.array_equal(q.cpu().numpy(), r["q"])
    assert_bf16_close(host_bits(out), r["out"], "pair w8a8")


def test_pair_mla(orc):
    d = si.make_mla(dict(seed=4, T=300, K=1024, N1=512, N2=1000))
    out = rnl.mla_q_chain(dev_bf16(d["x"]), dev_bf16(d["W_qa"]), dev_bf16(d["gamma_cq"]),
                          dev_bf16(d["W_qb"]))
    _, _, want = orc.mla_q_chain(d["x"], d["W_qa"], d["gamma_cq"], d["W_qb"], 1e-6, 1)
    assert_bf16_close(host_bits(out), want, "pair mla")


def test_pair_qkv_full_sampled(orc):
    c = si.CONFIGS["qkv"]
    d = si.make_projection(c)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    rows = sample_rows(c["T"], 32)
    _, want = orc.rmsnorm_linear(d["x"][rows], d["gamma"], d["W"], c["eps"], 0, 0)
    assert_bf16_close(host_bits(out)[rows], want, "pair qkv sampled")
