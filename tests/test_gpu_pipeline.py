"""The host-buffer pipeline (rnl_pipeline_*) against the device-pointer entry
points and the oracle.

Several calls are submitted before any is waited on, each with its own
pinned input and output, so that both staging slots are reused while other
calls are in flight; every output must equal, bit for bit, what the
device-pointer call computes for the same input (same kernels, same
order), and a sample of rows is checked against the oracle."""
import ctypes

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


def pinned_bf16(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory()


def pinned_empty(shape, dtype):
    return torch.empty(shape, dtype=dtype).pin_memory()


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


CALLS = 5  # > 2 slots: every slot is reused while the other is busy


@pytest.mark.parametrize("T,K,N,out_dtype,gamma", [
    (1000, 1024, 1536, 0, True),   # several tiles, ragged T
    (300, 520, 600, 0, False),
    (1100, 16384, 24, 1, False),   # mhc_pre fp32 form (skinny kernel)
])
def test_pipeline_bf16_equals_device_call(orc, T, K, N, out_dtype, gamma):
    base = si.make_projection(dict(seed=77 + T, T=T, K=K, N=N, has_gamma=gamma))
    W = dev_bf16(base["W"])
    g = dev_bf16(base["gamma"]) if gamma else None
    odt = torch.float32 if out_dtype == 1 else torch.bfloat16
    xs = [si.make_projection(dict(seed=500 + i, T=T, K=K, N=1, has_gamma=False))["x"] for i in range(CALLS)]
    hx = [pinned_bf16(x) for x in xs]
    ho = [pinned_empty((T, N), odt) for _ in range(CALLS)]
    p = rnl.rnl_pipeline_create(rnl.OP_BF16, T, K, N, out_dtype)
    try:
        tickets = [rnl.rnl_pipeline_submit_bf16(p, hx[i], g, W, ho[i]) for i in range(CALLS)]
        assert tickets == list(range(CALLS))
        for t in reversed(tickets):
            rnl.rnl_pipeline_wait(p, t)
    finally:
        rnl.rnl_pipeline_destroy(p)
    for i in range(CALLS):
        want = rnl.rmsnorm_linear_bf16(dev_bf16(xs[i]), g, W, out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert torch.equal(ho[i].view(torch.int16 if odt == torch.bfloat16 else torch.int32),
                           want.cpu().view(torch.int16 if odt == torch.bfloat16 else torch.int32)), i
    if out_dtype == 0:
        rows = sample_rows(T, 24, seed=T)
        _, ref = orc.rmsnorm_linear(xs[0][rows], base["gamma"] if gamma else None, base["W"], 1e-6, 0, 0)
        assert_bf16_close(_bits(ho[0])[rows], ref, "pipeline bf16 vs oracle")


def test_pipeline_w8a8_equals_device_call():
    T, K, N = 700, 1024, 520
    c = dict(seed=91, T=T, K=K, N=N)
    base = si.make_w8a8(c)
    Wq, ws, g = dev(base["Wq"]), dev(base["w_scale"]), dev_bf16(base["gamma"])
    xs = [si.make_w8a8(dict(c, seed=300 + i))["x"] for i in range(CALLS)]
    hx = [pinned_bf16(x) for x in xs]
    ho = [pinned_empty((T, N), torch.bfloat16) for _ in range(CALLS)]
    p = rnl.rnl_pipeline_create(rnl.OP_W8A8, T, K, N)
    try:
        tickets = [rnl.rnl_pipeline_submit_w8a8(p, hx[i], g, Wq, ws, ho[i]) for i in range(CALLS)]
        rnl.rnl_pipeline_wait(p, tickets[-1])
        rnl.rnl_pipeline_wait(p, tickets[0])
    finally:
        rnl.rnl_pipeline_destroy(p)
    for i in range(CALLS):
        want = rnl.rmsnorm_linear_w8a8(dev_bf16(xs[i]), g, Wq, ws)
        assert np.array_equal(_bits(ho[i]), host_bits(want)), i


def test_pipeline_mla_equals_device_call():
    T, K, N1, N2 = 300, 1024, 256, 1100
    c = dict(seed=92, T=T, K=K, N1=N1, N2=N2)
    base = si.make_mla(c)
    Wa, gq, Wb = dev_bf16(base["W_qa"]), dev_bf16(base["gamma_cq"]), dev_bf16(base["W_qb"])
    xs = [si.make_mla(dict(c, seed=400 + i))["x"] for i in range(CALLS)]
    hx = [pinned_bf16(x) for x in xs]
    ho = [pinned_empty((T, N2), torch.bfloat16) for _ in range(CALLS)]
    p = rnl.rnl_pipeline_create(rnl.OP_MLA, T, K, N1, N2)
    try:
        tickets = [rnl.rnl_pipeline_submit_mla(p, hx[i], Wa, gq, Wb, ho[i]) for i in range(CALLS)]
        for t in tickets:
            rnl.rnl_pipeline_wait(p, t)
    finally:
        rnl.rnl_pipeline_destroy(p)
    for i in range(CALLS):
        want = rnl.mla_q_chain(dev_bf16(xs[i]), Wa, gq, Wb)
        assert np.array_equal(_bits(ho[i]), host_bits(want)), i


def test_pipeline_rejects_pageable_host_memory_and_stays_usable():
    """A pageable host buffer is refused before anything is enqueued; the
    pipeline then serves a valid call normally."""
    T, K, N = 64, 256, 128
    d = si.make_projection(dict(seed=5, T=T, K=K, N=N, has_gamma=True))
    W, g = dev_bf16(d["W"]), dev_bf16(d["gamma"])
    p = rnl.rnl_pipeline_create(rnl.OP_BF16, T, K, N, 0)
    try:
        lib = rnl.load()
        x_pageable = np.ascontiguousarray(d["x"])
        out_pinned = pinned_empty((T, N), torch.bfloat16)
        tk = ctypes.c_int64(-1)
        st = lib.rnl_pipeline_submit_bf16(p.ptr, x_pageable.ctypes.data_as(ctypes.c_void_p),
                                          ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                          1e-6, 0, ctypes.c_void_p(out_pinned.data_ptr()), ctypes.byref(tk))
        assert st == 4  # RNL_ERR_ARG
        assert lib.rnl_pipeline_wait(p.ptr, 0, None) == 4  # no ticket issued yet
        hx = pinned_bf16(d["x"])  # held until the wait below
        t = rnl.rnl_pipeline_submit_bf16(p, hx, g, W, out_pinned)
        assert t == 0
        rnl.rnl_pipeline_wait(p, t)
    finally:
        rnl.rnl_pipeline_destroy(p)
    want = rnl.rmsnorm_linear_bf16(dev_bf16(d["x"]), g, W)
    assert np.array_equal(_bits(out_pinned), host_bits(want))
