"""MXFP8 mode (rmsnorm_linear_mxfp8, mxfp8_scaled_mm) against the oracle.

Codes and scale bytes: bit for bit.  The front end's FP32 steps are those of
the W8A8 front end (the FP32 sum of squares is the rounding of the exact sum,
every later step one correctly rounded operation), the block exponent is read
from the FP32 block maximum, and y * 2^-X is exact, so the E4M3 rounding sees
the same value on both sides.

Products, on both routes (the block-scaled tensor cores fed the E4M3 codes
and their scales, and the exact emulation with RNL_MXFP8_NATIVE=0 that
multiplies the dequantised operands with the bf16 GEMM), both with FP32
accumulation: fp32 out is held to the FP32 accumulation bound
|gpu - ref| <= 2^-16 sum_k |a_k w_k| + 2^-20 |ref| (ref the oracle's binary64
sum), bf16 out to the acceptance bound 1e-2 * max(1, |oracle|).
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_bf16_close, assert_fp32_close, dev, dev_bf16, host_bits, sample_rows

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


@pytest.fixture(autouse=True, params=["native", "native_pair", "emulated"])
def route(request, monkeypatch):
    """Every test on the block-scaled route (the default one-CTA kernel, and
    the CTA-pair form forced) and on the emulation route."""
    monkeypatch.setenv("RNL_MXFP8_NATIVE", "0" if request.param == "emulated" else "1")
    if request.param == "native_pair":
        monkeypatch.setenv("RNL_MXFP8_PAIR", "1")
    else:
        monkeypatch.delenv("RNL_MXFP8_PAIR", raising=False)
    yield request.param
    rnl.rnl_check_device_error()


def _dequant(codes, scales, block):
    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()
    return v * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), block, axis=1)


def _abs_sum(xq, xs, wq, ws, block):
    return np.abs(_dequant(xq, xs, block)) @ np.abs(_dequant(wq, ws, block)).T


def _run(d, block, eps, mode, out_dtype):
    T, K = d["x"].shape
    codes = torch.empty((T, K), dtype=torch.uint8, device="cuda")
    scales = torch.empty((T, K // block), dtype=torch.uint8, device="cuda")
    g = dev_bf16(d["gamma"]) if d["gamma"] is not None else None
    out = rnl.rmsnorm_linear_mxfp8(dev_bf16(d["x"]), g, dev(d["w_codes"]), dev(d["w_scale"]), eps=eps,
                                   norm_mode=mode, block=block, out_dtype=out_dtype, x_codes_out=codes,
                                   x_scale_out=scales)
    o = host_bits(out) if out_dtype == rnl.OUT_BF16 else out.cpu().numpy()
    return codes.cpu().numpy(), scales.cpu().numpy(), o


@pytest.mark.parametrize("T,K,N,block,mode,gamma,out_dtype", [
    (37, 256, 72, 64, 0, True, 0),
    (130, 4096, 200, 64, 0, True, 0),     # registers form at the workload's K, ragged T
    (64, 6144, 136, 64, 1, True, 1),      # rows longer than 4096: the two-read form
    (50, 192, 64, 32, 0, False, 1),       # the OCP block of 32
    (9, 64, 16, 64, 1, True, 0),          # one block per row
    (300, 1024, 264, 32, 1, False, 0),
    (257, 2048, 384, 64, 0, True, 1),
])
def test_mxfp8_front_and_product(orc, T, K, N, block, mode, gamma, out_dtype):
    cfg = dict(seed=T + K + N + block, T=T, K=K, N=N, block=block, has_gamma=gamma)
    d = si.make_mxfp8(cfg)
    xq, xs, out = _run(d, block, 1e-6, mode, out_dtype)
    wq, wsc = orc.mxfp8_quant_rows(d["x"], d["gamma"], 1e-6, mode, block=block)
    assert np.array_equal(xs, wsc), f"scales: {(xs != wsc).sum()} differ"
    assert np.array_equal(xq, wq), f"codes: {(xq != wq).sum()} differ"
    ref, want = orc.mxfp8_scaled_mm(wq, wsc, d["w_codes"], d["w_scale"], out_dtype, block=block)
    if out_dtype == 0:
        assert_bf16_close(out, want, "bf16 out")
    else:
        assert_fp32_close(out, ref, _abs_sum(wq, wsc, d["w_codes"], d["w_scale"], block), "fp32 out")


def test_mxfp8_constructed_ties_and_saturation(orc):
    """Rows whose normed values land on E4M3 ties, the subnormal range,
    negative values that round to zero and (row 1) saturation; rstd = 1/64
    exactly, block maximum 1.5 or 1.90625, X = -8."""
    base = [96.0, 17 / 64, 19 / 64, -17 / 64, 2.0**-12, 3 * 2.0**-12, 7.5 * 2.0**-11, -2.0**-12,
            -0.0, -3 * 2.0**-12]
    rows = np.array([base + [0.0] * 54, [122.0] + base[1:] + [0.0] * 54], np.float32)
    bits = rows.view(np.uint32) >> np.uint32(16)  # exact: every value has <= 8 significant bits
    x = bits.astype(np.uint16)
    for r in range(2):
        ms = float(np.sum(rows[r].astype(np.float64) ** 2)) / 64
        eps = float(np.float32(4096.0 - ms))
        d = {"x": x[r:r + 1], "gamma": None, "w_codes": si.e4m3_codes(7, "w", (16, 64)),
             "w_scale": np.full((16, 1), 120, np.uint8)}
        for mode in (0, 1):
            xq, xs, out = _run(d, 64, eps, mode, 1)
            wq, wsc = orc.mxfp8_quant_rows(d["x"], None, eps, mode)
            assert xs.tolist() == [[119]] and wsc.tolist() == [[119]]
            assert np.array_equal(xq, wq), (r, mode, xq[0, :10], wq[0, :10])
            assert xq[0, 0] == (0x7C if r == 0 else 0x7E)
            assert xq[0, 7] == 0x80 and xq[0, 8] == 0x80 and xq[0, 9] == 0x82


def test_mxfp8_zero_rows_and_blocks(orc):
    T, K, N = 20, 512, 48
    d = si.make_mxfp8(dict(seed=77, T=T, K=K, N=N, block=64, has_gamma=True))
    d["x"][3] = 0                 # an all-zero row
    d["x"][5, 128:192] = 0        # a zero block
    xq, xs, out = _run(d, 64, 1e-6, 0, 1)
    wq, wsc = orc.mxfp8_quant_rows(d["x"], d["gamma"], 1e-6, 0)
    assert np.array_equal(xq, wq) and np.array_equal(xs, wsc)
    assert not xq[3].any() and (xs[3] == 0).all() and (out[3] == 0).all()
    assert not xq[5, 128:192].any() and xs[5, 2] == 0


@pytest.mark.parametrize("T,K,N,block", [(33, 320, 80, 64), (200, 2048, 256, 32), (1, 64, 16, 64)])
def test_mxfp8_scaled_mm_oracle_operands(orc, T, K, N, block):
    """scaled_mm fed the same codes and scales on both sides."""
    xq = si.e4m3_codes(T, "xq", (T, K), e_lo=0)
    xs = si.uniform_u8(T, "xs", (T, K // block), 117, 130)
    wq = si.e4m3_codes(T, "wq", (N, K), e_lo=0)
    ws = si.uniform_u8(T, "ws", (N, K // block), 110, 120)
    for od in (0, 1):
        out = rnl.mxfp8_scaled_mm(dev(xq), dev(xs), dev(wq), dev(ws), block=block, out_dtype=od)
        ref, want = orc.mxfp8_scaled_mm(xq, xs, wq, ws, od, block=block)
        if od == 0:
            assert_bf16_close(host_bits(out), want, "bf16 out")
        else:
            assert_fp32_close(out.cpu().numpy(), ref, _abs_sum(xq, xs, wq, ws, block), "fp32 out")


def test_mxfp8_empty_batch():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((16, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((16, 2), dtype=torch.uint8, device="cuda")
    out = rnl.rmsnorm_linear_mxfp8(x, None, w, s)
    assert out.shape == (0, 16)


def test_mxfp8_full_size_sampled(orc):
    """The mxfp8 workload's size (4096 x 4096 -> 6144, block 64), in the
    launch configuration the benchmark times: every row's codes and scales
    bit for bit, sampled rows' outputs against the oracle."""
    c = si.CONFIGS["mxfp8"]
    d = si.make_mxfp8(c)
    xq, xs, out = _run(d, 64, c["eps"], c["norm_mode"], 0)
    wq, wsc = orc.mxfp8_quant_rows(d["x"], d["gamma"], c["eps"], c["norm_mode"])
    assert np.array_equal(xs, wsc), f"scales: {(xs != wsc).sum()} differ"
    assert np.array_equal(xq, wq), f"codes: {(xq != wq).sum()} differ"
    rows = sample_rows(c["T"], 32, seed=11)
    _, want = orc.mxfp8_scaled_mm(wq[rows], wsc[rows], d["w_codes"], d["w_scale"], 0)
    assert_bf16_close(out[rows], want, "full size")
