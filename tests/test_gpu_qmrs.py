"""QuantMatMulReduceSum (quant_matmul_reduce_sum) against the oracle, bit
for bit: the integer matmul is exact on both sides, and every later step
(int32 -> FP32, the FP32 scale product, the product, the FP32 sum over the
batch in increasing b, the bf16 cast) is one correctly rounded operation in
the same order on both sides."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import dev, dev_bf16, host_bits, sample_rows

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


def _run(d):
    return host_bits(rnl.quant_matmul_reduce_sum(dev(d["x1"]), dev(d["x2"]), dev(d["x1_scale"]),
                                                 dev_bf16(d["x2_scale"])))


@pytest.mark.parametrize("B,M,K,N", [
    (1, 64, 64, 64),
    (3, 130, 272, 208),    # ragged M, K and N of several tiles
    (4, 300, 1024, 528),
    (2, 1, 16, 16),        # smallest
    (5, 257, 2048, 1024),  # K of two exact-integer chunks
])
def test_qmrs_bit_exact(orc, B, M, K, N):
    d = si.make_qmrs(dict(seed=B * 1000 + M + K + N, B=B, M=M, K=K, N=N))
    _, want = orc.quant_matmul_reduce_sum(d["x1"], d["x2"], d["x1_scale"], d["x2_scale"])
    got = _run(d)
    assert np.array_equal(got, want), f"{(got != want).sum()} of {got.size} differ"


def test_qmrs_worst_case_integers(orc):
    """All codes +-127 with K = 4096: per-batch sums reach 66,064,384 > 2^24,
    beyond exact FP32, so the exact-integer path is what makes this pass."""
    B, M, K, N = 2, 200, 4096, 256
    rng = np.random.default_rng(5)
    d = {
        "x1": (rng.integers(0, 2, (B, M, K)) * 254 - 127).astype(np.int8),
        "x2": (rng.integers(0, 2, (B, K, N)) * 254 - 127).astype(np.int8),
        "x1_scale": rng.uniform(1e-3, 1e-2, (B, M)).astype(np.float32),
        "x2_scale": si.uniform_bf16(5, "x2_scale", (N,), 1e-3, 1e-2),
    }
    d["x1"][:, :4, :] = 127  # rows whose sums are all +-127 * 127 * K
    d["x2"][:, :, :4] = 127
    _, want = orc.quant_matmul_reduce_sum(d["x1"], d["x2"], d["x1_scale"], d["x2_scale"])
    assert np.array_equal(_run(d), want)


def test_qmrs_full_size_sampled(orc):
    """The qmrs workload's size (B = 4, M = 2048, K = N = 4096), sampled rows."""
    c = si.CONFIGS["qmrs"]
    d = si.make_qmrs(c)
    got = _run(d)
    rows = sample_rows(c["M"], 24, seed=9)
    ds = si.make_qmrs(c, rows=rows)
    _, want = orc.quant_matmul_reduce_sum(ds["x1"], ds["x2"], ds["x1_scale"], ds["x2_scale"])
    assert np.array_equal(got[rows], want)
