"""Cross-CTA hand-offs under repetition, against the oracle.

Two kernels pass partial results between CTAs through flags in the caller's
workspace: the CTA-pair GEMM's stream-K tiles (a finisher pair adds the
partial sums its partners published) and QuantMatMulReduceSum's batch sum
(item (b, tile) adds to the running sum item (b - 1, tile) published).

* Replay: a call captured in a CUDA graph keeps its launch arguments,
  including the flags' epoch, on every replay; each replay runs on new
  activations and must give the uncaptured call's bits on them (and agree
  with the oracle), so no replay may consume the previous replay's flags.
* Determinism: the hand-offs add partial sums in a fixed order, so repeated
  calls on the same inputs give identical bits; a race on a flag shows up as
  a difference between runs.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_bf16_close, dev, dev_bf16, host_bits, sample_rows

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


def _capture(fn):
    """Warm the call up on a side stream (one-time set-up stays outside the
    capture), then capture it into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("shape,force_pair", [
    ((4096, 4096, 6144), None),  # the qkv size: 4 data-parallel waves + stream-K tail
    ((600, 3000, 1000), "1"),    # 12 tiles on CTA pairs: every tile split
    ((3200, 1000, 1024), "0"),   # 100 one-CTA tiles of 128 x 256 (no hand-off: the baseline)
])
def test_graph_replay_bf16_stream_k(orc, monkeypatch, shape, force_pair):
    if force_pair is not None:
        monkeypatch.setenv("RNL_GEMM_PAIR", force_pair)
    if force_pair == "0":
        monkeypatch.setenv("RNL_GEMM_BN", "256")
    T, K, N = shape
    d = si.make_projection(dict(seed=31 + T, T=T, K=K, N=N))
    xs = [d["x"], si.make_projection(dict(seed=32 + T, T=T, K=K, N=N))["x"]]
    gamma, W = dev_bf16(d["gamma"]), dev_bf16(d["W"])
    ws = torch.empty(rnl.workspace_size(rnl.OP_BF16, T, K, N, rnl.OUT_BF16), dtype=torch.uint8,
                     device="cuda")
    # uncaptured reference results on each input (same workspace)
    direct = [host_bits(rnl.rmsnorm_linear_bf16(dev_bf16(x), gamma, W, workspace=ws)) for x in xs]
    x_static = dev_bf16(xs[0]).clone()
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    g = _capture(lambda: rnl.rmsnorm_linear_bf16(x_static, gamma, W, out=out, workspace=ws))
    rows = sample_rows(T, 24, seed=T)
    for i in (0, 1, 0, 1):
        x_static.copy_(dev_bf16(xs[i]))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = host_bits(out)
        assert np.array_equal(got, direct[i]), f"replay on input {i}: {(got != direct[i]).sum()} differ"
        _, want = orc.rmsnorm_linear(xs[i][rows], d["gamma"], d["W"], 1e-6, 0, 0)
        assert_bf16_close(got[rows], want, f"replay on input {i}")
    rnl.rnl_check_device_error()


def test_graph_replay_qmrs_batch_flags(orc):
    B, M, K, N = 4, 300, 1024, 528
    c = dict(seed=41, B=B, M=M, K=K, N=N)
    d = si.make_qmrs(c)
    d2 = si.make_qmrs(dict(c, seed=42))
    x2, x1s, x2s = dev(d["x2"]), dev(d["x1_scale"]), dev_bf16(d["x2_scale"])
    ws = torch.empty(rnl.workspace_size(rnl.OP_QMRS, M, K, N, B), dtype=torch.uint8, device="cuda")
    x1_inputs = [d["x1"], d2["x1"]]
    x1_static = dev(d["x1"]).clone()
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g = _capture(lambda: rnl.quant_matmul_reduce_sum(x1_static, x2, x1s, x2s, out=out, workspace=ws))
    for i in (0, 1, 0, 1):
        x1_static.copy_(dev(x1_inputs[i]))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        _, want = orc.quant_matmul_reduce_sum(x1_inputs[i], d["x2"], d["x1_scale"], d["x2_scale"])
        got = host_bits(out)
        assert np.array_equal(got, want), f"replay on input {i}: {(got != want).sum()} differ"
    rnl.rnl_check_device_error()


def _repeat_identical(call, n):
    first = call()
    for r in range(1, n):
        again = call()
        assert np.array_equal(first, again), f"run {r}: {(first != again).sum()} of {first.size} differ"
    return first


def test_deterministic_qkv_full():
    c = si.CONFIGS["qkv"]
    d = si.make_projection(c)
    x, gamma, W = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"])
    ws = torch.empty(rnl.workspace_size(rnl.OP_BF16, c["T"], c["K"], c["N"]), dtype=torch.uint8,
                     device="cuda")
    _repeat_identical(lambda: host_bits(rnl.rmsnorm_linear_bf16(x, gamma, W, workspace=ws)), 5)


def test_deterministic_stream_k_split_small(monkeypatch):
    monkeypatch.setenv("RNL_GEMM_PAIR", "1")
    d = si.make_projection(dict(seed=7, T=600, K=3000, N=1000))
    x, gamma, W = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"])
    _repeat_identical(lambda: host_bits(rnl.rmsnorm_linear_bf16(x, gamma, W)), 8)


def test_deterministic_w8a8_full():
    """W8A8 at full size: the streamed quantiser and the exact-integer GEMM."""
    c = si.CONFIGS["w8a8"]
    d = si.make_w8a8(c)
    x, g, Wq, ws_ = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev(d["Wq"]), dev(d["w_scale"])
    Wb = rnl.rnl_w8a8_prepare_weight(Wq)
    _repeat_identical(lambda: host_bits(rnl.rmsnorm_linear_w8a8_prepared(x, g, Wb, ws_)), 3)


def test_deterministic_qmrs_full():
    c = si.CONFIGS["qmrs"]
    d = si.make_qmrs(c)
    args = (dev(d["x1"]), dev(d["x2"]), dev(d["x1_scale"]), dev_bf16(d["x2_scale"]))
    ws = torch.empty(rnl.workspace_size(rnl.OP_QMRS, c["M"], c["K"], c["N"], c["B"]),
                     dtype=torch.uint8, device="cuda")
    _repeat_identical(lambda: host_bits(rnl.quant_matmul_reduce_sum(*args, workspace=ws)), 3)
