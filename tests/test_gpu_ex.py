"""AT-10 with the residual add, the AT-03 norm bias and output_rstd, and the
AT-09 projection bias (rmsnorm_linear_bf16_ex) against the oracle.

Bounds: out as every bf16 output, |gpu - oracle| <= 1e-2 * max(1, |oracle|);
x_sum (the bf16 residual sum) bit-exact; rstd (FP32 on the GPU, binary64 in
the oracle) within (K/64 + 8) * 2^-23 relative -- FP32 sums of K exact
squares over per-lane chains of K/32 terms and a 5-level tree, the 1/K
scale, the eps add and the reciprocal square root."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_bf16_close, dev_bf16, host_bits, sample_rows

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


def _case(seed, T, K, N):
    d = si.make_projection(dict(seed=seed, T=T, K=K, N=N, has_gamma=True))
    d["residual"] = si.normal_bf16(seed, "residual", (T, K), 1.0)
    d["beta"] = si.normal_bf16(seed, "beta", (K,), 0.1)
    d["bias"] = si.normal_bf16(seed, "bias", (N,), 0.5)
    return d


def _rstd_ok(gpu, ref, K):
    bound = (K / 64 + 8) * 2.0**-23
    rel = np.abs(gpu.astype(np.float64) - ref) / ref
    assert rel.max() <= bound, (rel.max(), bound)


@pytest.mark.parametrize("T,K,N,mode", [
    (130, 72, 300, 0),      # K tail (9 vectors), N tail
    (700, 1024, 520, 1),    # sqrt+div form
    (1000, 4096, 768, 0),   # longest row of the streamed pass
    (90, 8200, 300, 0),     # row beyond the streamed pass (warp-per-row kernel)
])
def test_ex_all_options(orc, T, K, N, mode):
    d = _case(T + K + N, T, K, N)
    x, res = dev_bf16(d["x"]), dev_bf16(d["residual"])
    xs_out = torch.empty_like(x)
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    out = rnl.rmsnorm_linear_bf16_ex(x, dev_bf16(d["gamma"]), dev_bf16(d["W"]), residual=res,
                                     x_sum_out=xs_out, beta=dev_bf16(d["beta"]),
                                     bias=dev_bf16(d["bias"]), norm_mode=mode, rstd_out=rstd)
    _, want, want_xs, want_r = orc.rmsnorm_linear_ex(d["x"], d["residual"], d["gamma"], d["beta"],
                                                      d["W"], d["bias"], 1e-6, mode)
    assert np.array_equal(host_bits(xs_out), want_xs)
    _rstd_ok(rstd.cpu().numpy(), want_r, K)
    assert_bf16_close(host_bits(out), want, f"ex {T}x{K}x{N}")


@pytest.mark.parametrize("K", [1024, 8200])
def test_ex_in_place_add(orc, K):
    """x_sum_out = residual and x_sum_out = x give the same output as a
    separate buffer, and leave the sum in the aliased input."""
    T, N = 300, 256
    d = _case(K, T, K, N)
    g, W = dev_bf16(d["gamma"]), dev_bf16(d["W"])
    ref_out = rnl.rmsnorm_linear_bf16_ex(dev_bf16(d["x"]), g, W, residual=dev_bf16(d["residual"]),
                                         x_sum_out=torch.empty(T, K, dtype=torch.bfloat16, device="cuda"))
    _, _, want_xs, _ = orc.rmsnorm_linear_ex(d["x"], d["residual"], d["gamma"], None, d["W"], None,
                                             1e-6, 0)
    for alias in ("residual", "x"):
        x, res = dev_bf16(d["x"]), dev_bf16(d["residual"])
        target = res if alias == "residual" else x
        out = rnl.rmsnorm_linear_bf16_ex(x, g, W, residual=res, x_sum_out=target)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), alias
        assert np.array_equal(host_bits(target), want_xs), alias


def test_ex_options_off_equals_plain_call():
    T, K, N = 500, 2048, 640
    d = _case(3, T, K, N)
    x, g, W = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"])
    a = rnl.rmsnorm_linear_bf16_ex(x, g, W)
    b = rnl.rmsnorm_linear_bf16(x, g, W)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("pair", ["0", "1"])
def test_ex_projection_bias_each_gemm(orc, monkeypatch, pair):
    """Bias alone (streamed norm pass), on the one-CTA GEMM and on CTA pairs
    with the K-split tail and its fix-up (2048 x 2560: 80 pair tiles on 76
    pairs)."""
    monkeypatch.setenv("RNL_GEMM_PAIR", pair)
    T, K, N = 2048, 512, 2560
    d = _case(11, T, K, N)
    out = rnl.rmsnorm_linear_bf16_ex(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                     bias=dev_bf16(d["bias"]))
    _, want, _, _ = orc.rmsnorm_linear_ex(d["x"], None, d["gamma"], None, d["W"], d["bias"], 1e-6, 0)
    assert_bf16_close(host_bits(out), want, f"bias pair={pair}")


def test_ex_rstd_only_and_beta_only(orc):
    T, K, N = 257, 3072, 384
    d = _case(12, T, K, N)
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    out = rnl.rmsnorm_linear_bf16_ex(dev_bf16(d["x"]), None, dev_bf16(d["W"]), beta=dev_bf16(d["beta"]),
                                     norm_mode=1, rstd_out=rstd)
    _, want, _, want_r = orc.rmsnorm_linear_ex(d["x"], None, None, d["beta"], d["W"], None, 1e-6, 1)
    assert_bf16_close(host_bits(out), want, "beta only")
    _rstd_ok(rstd.cpu().numpy(), want_r, K)


def test_ex_qkv_size_sampled(orc):
    """The qkv workload's size with every option on, sampled rows."""
    c = si.CONFIGS["qkv"]
    T, K, N = c["T"], c["K"], c["N"]
    d = _case(c["seed"], T, K, N)
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    out = rnl.rmsnorm_linear_bf16_ex(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                     residual=dev_bf16(d["residual"]), beta=dev_bf16(d["beta"]),
                                     bias=dev_bf16(d["bias"]), rstd_out=rstd)
    rows = sample_rows(T, 48, seed=5)
    _, want, _, want_r = orc.rmsnorm_linear_ex(d["x"][rows], d["residual"][rows], d["gamma"], d["beta"],
                                               d["W"], d["bias"], 1e-6, 0)
    assert_bf16_close(host_bits(out)[rows], want, "ex qkv")
    _rstd_ok(rstd.cpu().numpy()[rows], want_r, K)
