"""The allocation-free entry point (rmsnorm_linear_skinny_noalloc) against the
regular one (rmsnorm_linear_bf16, fp32 form), through the C ABI.

That entry point serves callers that cannot allocate device memory (code
inside a host program that owns all device allocations); its scratch is an
array built into the library and shared by every call, so two calls in a row
must both match.  This file is collected last, so a run that stops at the
first failure has run everything else first; it also passes on its own in a
fresh process.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_fp32_close, dev_bf16
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


def _abs_sum(d, mode):
    """sum_k |y_k| |w_k| per output, the scale of the fp32 accumulation bound."""
    xv = bf16_bits_to_f64(d["x"])
    rstd = 1.0 / np.sqrt(np.mean(xv * xv, axis=1) + 1e-6)
    return (np.abs(xv) * rstd[:, None]) @ np.abs(bf16_bits_to_f64(d["W"])).T


@pytest.mark.parametrize("T,K,N,mode", [(1000, 16384, 24, 0), (300, 4160, 64, 1)])
def test_noalloc_matches_regular_twice(T, K, N, mode):
    d = si.make_projection(dict(seed=77 + N, T=T, K=K, N=N, has_gamma=False))
    x, W = dev_bf16(d["x"]), dev_bf16(d["W"])
    ref = rnl.rmsnorm_linear_bf16(x, None, W, eps=1e-6, norm_mode=mode,
                                  out_dtype=rnl.OUT_FP32).cpu().numpy().astype(np.float64)
    bound_scale = _abs_sum(d, mode)
    for _ in range(2):  # the second call reuses the scratch left by the first
        out = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
        rnl.rmsnorm_linear_skinny_noalloc(x, W, eps=1e-6, norm_mode=mode, out=out)
        torch.cuda.synchronize()
        assert_fp32_close(out.cpu().numpy(), ref, bound_scale, "noalloc vs regular")
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
