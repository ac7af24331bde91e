"""The allocation-free entry point (rmsnorm_linear_skinny_noalloc), through the
C ABI, against the CPU oracle and against the regular entry point
(rmsnorm_linear_bf16, fp32 form).

That entry point serves callers that cannot allocate device memory (code
inside a host program that owns all device allocations); its scratch is an
array built into the library and shared by every call.  So the calls here
come in a row, with a call on different activations in between: the scratch
then holds values that are wrong for the next call, and that call must still
match.  This file is collected last, so a run that stops at the first failure
has run everything else first; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_fp32_close, dev_bf16, sample_rows
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


def _abs_sum(orc, x_bits, W_bits, mode):
    """sum_k |y_k| |w_k| per output, the scale of the fp32 accumulation bound."""
    y, _ = orc.rmsnorm_f64(x_bits, None, 1e-6, mode)
    return np.abs(y) @ np.abs(bf16_bits_to_f64(W_bits)).T


def _noalloc(x, W, mode):
    out = torch.full((x.shape[0], W.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    rnl.rmsnorm_linear_skinny_noalloc(x, W, eps=1e-6, norm_mode=mode, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("T,K,N,mode", [(1000, 16384, 24, 0), (300, 4160, 64, 1)])
def test_noalloc_matches_oracle_and_regular(orc, T, K, N, mode):
    d = si.make_projection(dict(seed=77 + N, T=T, K=K, N=N, has_gamma=False))
    d2 = si.make_projection(dict(seed=177 + N, T=T, K=K, N=N, has_gamma=False))
    x, W, x2 = dev_bf16(d["x"]), dev_bf16(d["W"]), dev_bf16(d2["x"])
    rows = sample_rows(T, 96, seed=N)
    want, _ = orc.rmsnorm_linear(d["x"][rows], None, d["W"], 1e-6, mode, 1)
    want_scale = _abs_sum(orc, d["x"][rows], d["W"], mode)
    reg = rnl.rmsnorm_linear_bf16(x, None, W, eps=1e-6, norm_mode=mode,
                                  out_dtype=rnl.OUT_FP32).cpu().numpy().astype(np.float64)
    reg2 = rnl.rmsnorm_linear_bf16(x2, None, W, eps=1e-6, norm_mode=mode,
                                   out_dtype=rnl.OUT_FP32).cpu().numpy().astype(np.float64)
    reg_scale = _abs_sum(orc, d["x"], d["W"], mode)
    reg2_scale = _abs_sum(orc, d2["x"], d["W"], mode)
    # first call: against the oracle on sampled rows and the regular path on all rows
    got = _noalloc(x, W, mode)
    assert_fp32_close(got[rows], want, want_scale, "noalloc call 1 vs oracle")
    assert_fp32_close(got, reg, reg_scale, "noalloc call 1 vs regular")
    # a call on other activations leaves scratch values that are wrong for x
    got2 = _noalloc(x2, W, mode)
    assert_fp32_close(got2, reg2, reg2_scale, "noalloc call 2 (other x) vs regular")
    # the next call on x must not see them
    got3 = _noalloc(x, W, mode)
    assert_fp32_close(got3[rows], want, want_scale, "noalloc call 3 vs oracle")
    assert_fp32_close(got3, reg, reg_scale, "noalloc call 3 vs regular")
    rnl.rnl_check_device_error()


def test_noalloc_rejects_oversize_without_launching():
    # T beyond what the built-in scratch holds for N <= 64 (45,056 rows on 152 SMs)
    T, K, N = 200_000, 64, 48
    x = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    out = torch.full((T, N), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(rnl.RnlError) as e:
        rnl.rmsnorm_linear_skinny_noalloc(x, W, out=out)
    assert e.value.status == 5  # RNL_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
