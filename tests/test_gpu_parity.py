"""CUDA path against the CPU oracle, element by element, through the C ABI.

Small shapes span several 128x256 tiles with ragged tails in T, N and K and
are compared in full; the five workload sizes are run in the configuration
the benchmark times and compared on sampled rows (rows are independent, so
a sampled row is checked exactly as in a full comparison).

Bounds: bf16 outputs |gpu - oracle| <= 1e-2 * max(1, |oracle|); fp32
outputs (mhc_pre form) the fp32-accumulation bound of gpu_util; the INT8
matmul and the INT8 codes bit-exact.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import (assert_bf16_close, assert_fp32_close, dev, dev_bf16, host_bits,
                      sample_rows)
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


def _rand_case(seed, T, K, N, gamma=True):
    c = dict(seed=seed, T=T, K=K, N=N, has_gamma=gamma)
    return si.make_projection(c)


# ----------------------------------------------------------------- AT-10
@pytest.mark.parametrize("T,K,N,mode,gamma", [
    (16, 256, 128, 0, True),     # the tiny workload's shape
    (1, 8, 1, 0, True),          # smallest everything
    (130, 72, 300, 0, True),     # T, K (64 + 8) and N (256 + 44) tails
    (300, 520, 520, 1, True),    # sqrt+div form, N not a multiple of 8
    (257, 1024, 768, 0, False),  # no gamma, three N tiles
    (1000, 256, 100, 1, True),
    (640, 4096, 512, 0, True),   # long K
    (100, 8200, 300, 0, True),   # K beyond the streamed norm pass (row-loop kernel)
    (3000, 1536, 256, 1, True),  # many row groups per CTA in the streamed norm pass
])
def test_bf16_small(orc, T, K, N, mode, gamma):
    d = _rand_case(7 + T + K + N, T, K, N, gamma)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]) if gamma else None,
                                  dev_bf16(d["W"]), eps=1e-6, norm_mode=mode)
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, mode, 0)
    assert_bf16_close(host_bits(out), want, f"bf16 {T}x{K}x{N}")


@pytest.mark.parametrize("T,K,N,mode,gamma", [
    (1, 4096, 6144, 0, True),   # one decode token through the qkv weight
    (4, 4096, 1024, 1, False),  # the token limit
    (4, 12288, 2048, 0, True),  # 96 KB of normalised rows
    (3, 2056, 2000, 0, True),   # rows of 257 vectors: a ragged last lane stride
    (2, 2048, 1025, 1, True),   # a ragged weight
    (2, 7168, 1536, 1, True),   # the MLA q_a weight: 3.5 chunks a row
    (2, 2056, 5000, 0, True),   # several rows a warp, each row's second chunk one vector
    (5, 4096, 1024, 0, True),   # beyond the token limit: the tensor-core path either way
])
@pytest.mark.parametrize("decode", ["mma", "0", "rows1", "rows2"])
def test_bf16_decode_sized_both_paths(orc, monkeypatch, decode, T, K, N, mode, gamma):
    """Up to 4 tokens against a wide weight run as a matrix-vector product
    over every SM: on the tensor cores with the K ranges split over several
    CTAs (mma), or on the CUDA cores with one or two weight rows per warp
    group (rows1 / rows2); RNL_DECODE=0 sends them to the GEMM path.  All
    against the oracle."""
    monkeypatch.setenv("RNL_DECODE", "0" if decode == "0" else "1")
    monkeypatch.setenv("RNL_DECODE_MMA", "1" if decode == "mma" else "0")
    if decode.startswith("rows"):
        monkeypatch.setenv("RNL_DECODE_ROWS", decode[-1])
    d = _rand_case(13 + T + K + N, T, K, N, gamma)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]) if gamma else None,
                                  dev_bf16(d["W"]), eps=1e-6, norm_mode=mode)
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, mode, 0)
    assert_bf16_close(host_bits(out), want, f"decode={decode} {T}x{K}x{N}")


@pytest.mark.parametrize("rewrite_weight", [False, True])
def test_decode_chain_reads_what_the_kernel_before_wrote(orc, monkeypatch, rewrite_weight):
    """Decode calls back to back, each taking the previous call's output as
    its tokens (square weights).  The decode kernel is launched as a
    programmatic dependent of the kernel before it, so it may start before
    that kernel's writes are visible: the tokens (written by the previous
    decode call) and, with rewrite_weight, the weight (written by a copy
    kernel just before the call) must still be read as written.  Each call
    against the oracle on the inputs it was given."""
    monkeypatch.setenv("RNL_DECODE", "1")
    monkeypatch.setenv("RNL_DECODE_MMA", "0")
    T, K, layers = 4, 4096, 4
    ds = [_rand_case(211 + i, T, K, K, True) for i in range(layers)]
    gamma = dev_bf16(ds[0]["gamma"])
    staged = [dev_bf16(d["W"]) for d in ds]
    W_one = torch.empty_like(staged[0])
    x, outs = dev_bf16(ds[0]["x"]), []
    for i in range(layers):
        if rewrite_weight:
            W_one.copy_(staged[i])
        out = rnl.rmsnorm_linear_bf16(x, gamma, W_one if rewrite_weight else staged[i], eps=1e-6, norm_mode=0)
        outs.append(out)
        x = out
    torch.cuda.synchronize()
    x_bits = ds[0]["x"]
    for i in range(layers):
        _, want = orc.rmsnorm_linear(x_bits, ds[0]["gamma"], ds[i]["W"], 1e-6, 0, 0)
        got = host_bits(outs[i])
        assert_bf16_close(got, want, f"decode chain call {i} rewrite_weight={rewrite_weight}")
        x_bits = got


@pytest.mark.parametrize("bn", [128, 192, 256])
@pytest.mark.parametrize("T,K,N", [(300, 520, 600), (129, 4096, 256)])
def test_bf16_each_tile_width(orc, monkeypatch, bn, T, K, N):
    """The one-CTA GEMM (RNL_GEMM_PAIR=0) at each output tile width."""
    monkeypatch.setenv("RNL_GEMM_PAIR", "0")
    monkeypatch.setenv("RNL_GEMM_BN", str(bn))
    d = _rand_case(bn + T + N, T, K, N, True)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    assert_bf16_close(host_bits(out), want, f"bf16 BN={bn} {T}x{K}x{N}")


@pytest.mark.parametrize("bn", [128, 192, 256])
def test_gemm_s8_each_tile_width(orc, monkeypatch, bn):
    monkeypatch.setenv("RNL_GEMM_PAIR", "0")
    monkeypatch.setenv("RNL_GEMM_BN", str(bn))
    rng = np.random.default_rng(bn)
    A = rng.integers(-127, 128, (260, 2064)).astype(np.int8)
    B = rng.integers(-127, 128, (520, 2064)).astype(np.int8)
    C = rnl.rnl_gemm_s8s8s32(dev(A), dev(B)).cpu().numpy()
    want, _ = orc.gemm_s8(A, B)
    assert np.array_equal(C, want)


# 40 x 4 = 160 tiles of 128 x 256: more tiles than one wave of CTAs, N
# ragged (the last tile column straddles N), K two exact-integer chunks, the
# second partial.
def test_gemm_s8_past_one_wave(orc, monkeypatch):
    monkeypatch.setenv("RNL_GEMM_PAIR", "0")
    monkeypatch.setenv("RNL_GEMM_BN", "256")
    rng = np.random.default_rng(160)
    A = rng.integers(-127, 128, (5120, 1040)).astype(np.int8)  # two chunks, the second partial
    B = rng.integers(-127, 128, (1000, 1040)).astype(np.int8)
    C = rnl.rnl_gemm_s8s8s32(dev(A), dev(B)).cpu().numpy()
    want, _ = orc.gemm_s8(A, B)
    assert np.array_equal(C, want)


def test_bf16_past_one_wave(orc, monkeypatch):
    monkeypatch.setenv("RNL_GEMM_PAIR", "0")
    monkeypatch.setenv("RNL_GEMM_BN", "256")
    d = _rand_case(161, 5120, 520, 1000, True)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    assert_bf16_close(host_bits(out), want, "bf16 one-CTA 5120x520x1000")


# The one-CTA kernel with one partial wave of tiles (3200 x 1024 at BN = 256:
# 100 tiles) and with a whole wave and then a partial one (8064 x 1024: 252);
# K ragged, 2096 spanning three exact-int32 chunks.
@pytest.mark.parametrize("M", [3200, 8064])
def test_gemm_s8_partial_wave(orc, monkeypatch, M):
    monkeypatch.setenv("RNL_GEMM_PAIR", "0")
    monkeypatch.setenv("RNL_GEMM_BN", "256")
    rng = np.random.default_rng(M)
    A = rng.integers(-127, 128, (M, 2096)).astype(np.int8)
    B = rng.integers(-127, 128, (1024, 2096)).astype(np.int8)
    C = rnl.rnl_gemm_s8s8s32(dev(A), dev(B)).cpu().numpy()
    rows = sample_rows(M, 64, seed=M)
    want, _ = orc.gemm_s8(A[rows], B)
    assert np.array_equal(C[rows], want)


@pytest.mark.parametrize("T", [3200, 8064])
def test_bf16_partial_wave(orc, monkeypatch, T):
    monkeypatch.setenv("RNL_GEMM_PAIR", "0")
    monkeypatch.setenv("RNL_GEMM_BN", "256")
    d = _rand_case(T + 7, T, 1000, 1024, True)
    out = host_bits(rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"])))
    rows = sample_rows(T, 64, seed=T)
    _, want = orc.rmsnorm_linear(d["x"][rows], d["gamma"], d["W"], 1e-6, 0, 0)
    assert_bf16_close(out[rows], want, f"bf16 one-CTA {T}x1000x1024")


@pytest.mark.parametrize("T,K,N,mode,gamma", [(130, 72, 300, 0, True), (640, 4096, 512, 1, False)])
def test_bf16_fused_norm_form(orc, monkeypatch, T, K, N, mode, gamma):
    """RNL_FUSED_NORM=1: transform warps normalise the A stages inside the GEMM."""
    monkeypatch.setenv("RNL_FUSED_NORM", "1")
    d = _rand_case(3 + T + K + N, T, K, N, gamma)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]) if gamma else None,
                                  dev_bf16(d["W"]), eps=1e-6, norm_mode=mode)
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, mode, 0)
    assert_bf16_close(host_bits(out), want, f"fused-norm bf16 {T}x{K}x{N}")


def test_fused_and_two_kernel_forms_agree(monkeypatch):
    """Both forms compute bf16((x * rstd) * gamma) with the same arithmetic.
    Both run on the one-CTA GEMM (the fused form's only GEMM), so the K sums
    are taken in the same order and the outputs agree bit for bit."""
    monkeypatch.setenv("RNL_GEMM_PAIR", "0")
    d = _rand_case(99, 520, 2048, 700, True)
    args = (dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    monkeypatch.setenv("RNL_FUSED_NORM", "1")
    a = host_bits(rnl.rmsnorm_linear_bf16(*args))
    monkeypatch.setenv("RNL_FUSED_NORM", "0")
    b = host_bits(rnl.rmsnorm_linear_bf16(*args))
    assert np.array_equal(a, b)


def test_tiny_workload_and_golden(orc):
    c = si.CONFIGS["tiny"]
    d = si.make_projection(c)
    out = host_bits(rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                            eps=c["eps"], norm_mode=c["norm_mode"]))
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], c["eps"], c["norm_mode"], 0)
    assert_bf16_close(out, want, "tiny")
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_rmsnorm_linear_bf16.txt")
    stored = np.array([[int(v, 16) for v in ln.split()] for ln in open(path) if not ln.startswith("#")],
                      np.uint16)
    assert_bf16_close(out, stored, "tiny vs stored oracle output")


@pytest.mark.parametrize("pair", ["0", "1"])
def test_one_cta_and_pair_gemm_agree_qkv(monkeypatch, pair):
    """Full qkv size through both GEMM kernels: identical bf16 results are not
    required (different accumulation splits), closeness to each other is."""
    c = si.CONFIGS["qkv"]
    d = si.make_projection(c)
    args = (dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    monkeypatch.setenv("RNL_GEMM_PAIR", pair)
    a = host_bits(rnl.rmsnorm_linear_bf16(*args))
    monkeypatch.setenv("RNL_GEMM_PAIR", "1" if pair == "0" else "0")
    b = host_bits(rnl.rmsnorm_linear_bf16(*args))
    assert_bf16_close(a, b, "one-CTA vs pair GEMM")


def test_qkv_full_sampled(orc):
    c = si.CONFIGS["qkv"]
    d = si.make_projection(c)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                  eps=c["eps"], norm_mode=c["norm_mode"])
    rows = sample_rows(c["T"], 48)
    got = host_bits(out)[rows]
    _, want = orc.rmsnorm_linear(d["x"][rows], d["gamma"], d["W"], c["eps"], c["norm_mode"], 0)
    assert_bf16_close(got, want, "qkv sampled rows")


# ------------------------------------------------------- mhc_pre FP32 form
def _fp32_check(orc, d, mode, out, rows=None):
    x = d["x"] if rows is None else d["x"][rows]
    got = out.cpu().numpy() if rows is None else out.cpu().numpy()[rows]
    ref, _ = orc.rmsnorm_linear(x, None, d["W"], 1e-6, mode, 1)
    y, _ = orc.rmsnorm_f64(x, None, 1e-6, mode)
    abs_sum = np.abs(y) @ np.abs(bf16_bits_to_f64(d["W"])).T
    return assert_fp32_close(got, ref, abs_sum, "fp32 form")


@pytest.mark.parametrize("T,K,N,mode", [
    (300, 20480, 24, 0),   # skinny kernel: 3 row tiles (ragged), split across CTAs
    (129, 16384, 64, 1),   # N = 64, sqrt+div form
    (1, 512, 1, 0),        # one row, one output
    (700, 4160, 33, 0),    # N just above 32 (64-wide MMA), K tail
    (500, 1024, 200, 0),   # N > 64: row rstd pass + GEMM with row-scale epilogue
    (200, 2048, 600, 1),
])
def test_fp32_form_small(orc, T, K, N, mode):
    d = _rand_case(11 + T + K + N, T, K, N, gamma=False)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), None, dev_bf16(d["W"]), eps=1e-6,
                                  norm_mode=mode, out_dtype=rnl.OUT_FP32)
    _fp32_check(orc, d, mode, out)


def test_skinny_full_sampled(orc):
    c = si.CONFIGS["skinny"]
    d = si.make_projection(c)
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), None, dev_bf16(d["W"]), eps=c["eps"],
                                  norm_mode=c["norm_mode"], out_dtype=rnl.OUT_FP32)
    rows = sample_rows(c["T"], 64)
    _fp32_check(orc, d, c["norm_mode"], out, rows)


# -------------------------------------------------------------- MLA chain
@pytest.mark.parametrize("fused", ["1", "0"])
@pytest.mark.parametrize("T,K,N1,N2,mode", [
    (200, 1024, 512, 1000, 1),
    (129, 520, 136, 264, 0),
])
def test_mla_small(orc, monkeypatch, fused, T, K, N1, N2, mode):
    monkeypatch.setenv("RNL_FUSED_NORM", fused)
    c = dict(seed=T + K, T=T, K=K, N1=N1, N2=N2)
    d = si.make_mla(c)
    qa = torch.empty((T, N1), dtype=torch.bfloat16, device="cuda")
    out = rnl.mla_q_chain(dev_bf16(d["x"]), dev_bf16(d["W_qa"]), dev_bf16(d["gamma_cq"]),
                          dev_bf16(d["W_qb"]), eps=1e-6, norm_mode=mode, qa_out=qa)
    want_qa, _, want = orc.mla_q_chain(d["x"], d["W_qa"], d["gamma_cq"], d["W_qb"], 1e-6, mode)
    assert_bf16_close(host_bits(qa), want_qa, "mla stage 1")
    assert_bf16_close(host_bits(out), want, "mla out")


def test_mla_full_sampled(orc):
    c = si.CONFIGS["mla"]
    d = si.make_mla(c)
    out = rnl.mla_q_chain(dev_bf16(d["x"]), dev_bf16(d["W_qa"]), dev_bf16(d["gamma_cq"]),
                          dev_bf16(d["W_qb"]), eps=c["eps"], norm_mode=c["norm_mode"])
    rows = sample_rows(c["T"], 24)
    _, _, want = orc.mla_q_chain(d["x"][rows], d["W_qa"], d["gamma_cq"], d["W_qb"], c["eps"],
                                 c["norm_mode"])
    assert_bf16_close(host_bits(out)[rows], want, "mla sampled rows")


# ------------------------------------------------------------------ W8A8
@pytest.mark.parametrize("M,N,K", [(300, 300, 4096), (1, 1, 16), (129, 257, 1040)])
def test_gemm_s8_bit_exact_random(orc, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-127, 128, (M, K)).astype(np.int8)
    B = rng.integers(-127, 128, (N, K)).astype(np.int8)
    C = rnl.rnl_gemm_s8s8s32(dev(A), dev(B)).cpu().numpy()
    want, ovf = orc.gemm_s8(A, B)
    assert not ovf
    assert np.array_equal(C, want)


def test_gemm_s8_bit_exact_worst_case(orc):
    # all entries +-127: partial sums reach 127*127*K = 66,064,384 > 2^24 for
    # K = 4096, which fp32 accumulation without the exact 1024-chunks would round
    M, N, K = 130, 260, 4096
    A = np.full((M, K), 127, np.int8)
    A[1::2] = -127
    B = np.full((N, K), 127, np.int8)
    B[::3] = -127
    B[5, ::2] = -127  # mixed signs in one row
    C = rnl.rnl_gemm_s8s8s32(dev(A), dev(B)).cpu().numpy()
    want, ovf = orc.gemm_s8(A, B)
    assert not ovf
    assert int(np.abs(want).max()) == 127 * 127 * K
    assert np.array_equal(C, want)


# ------------------------------------------------------------- edge cases
def test_empty_T_is_noop():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    out = rnl.rmsnorm_linear_bf16(x, None, W)
    assert out.shape == (0, 8)


def test_misaligned_pointer_rejected():
    buf = torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda")
    x = buf.view(-1)[1:1 + 16 * 64].view(16, 64)  # 2-byte offset
    W = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rnl.RnlError) as e:
        rnl.rmsnorm_linear_bf16(x, None, W)
    assert e.value.status == 3


def test_device_error_word_clean():
    rnl.rnl_check_device_error()
