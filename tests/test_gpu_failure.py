"""Failure detection on the GPU without a fault: a kernel's bounded wait on a
barrier that nothing arrives on gives up after 1 ms, the host reads
RNL_ERR_TIMEOUT (wait site 99) and the context keeps working."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_bf16_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

rnl = pytest.importorskip("rmsnorm_linear_projection_gb300")


def test_wait_timeout_is_reported_and_context_survives(orc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rnl.rnl_check_device_error()  # start clean
    rnl.rnl_selftest_wait_timeout()
    with pytest.raises(rnl.RnlError) as e:
        rnl.rnl_check_device_error()
    assert e.value.status == 7 and "site 99" in str(e.value)
    rnl.rnl_check_device_error()  # the word was cleared
    d = si.make_projection(dict(seed=21, T=200, K=512, N=300, has_gamma=True))
    out = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]))
    _, want = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    assert_bf16_close(host_bits(out), want, "after the self-test")
    rnl.rnl_check_device_error()
