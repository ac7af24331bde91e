"""The debug build (librnl_debug.so, compiled with RNL_DEBUG) on small ragged
shapes of every kernel family that carries device-side bounds checks (the
one-CTA and CTA-pair GEMMs incl. stream-K hand-offs and the integer and
batch-sum modes, the streamed norm pass and W8A8 quantiser, the W8A8 weight
preparation, the MXFP8 front end and block-scaled GEMM, the skinny stream and
its reduce, and both decode-step kernels).

Each case runs through the release library and then through the debug
library: no check may fire (rnl_check_device_error is clean), and the
outputs must be identical bit for bit (the checks only guard accesses).
The self-test shows the checks are live: a check on a deliberately smaller
limit fails and is reported as RNL_ERR_BOUNDS with its site.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

rnl = pytest.importorskip("rmsnorm_linear_projection_gb300")


@pytest.fixture(scope="module", autouse=True)
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rmsnorm_linear_projection_gb300 import build
    build.build()
    build.build(debug=True)
    torch.cuda.set_device(0)


def _bits(t):
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return host_bits(t)
    return t.cpu().numpy().view(np.uint8)


def _both(call):
    """Run `call` (returns a tensor or a tuple of tensors) on the release and
    on the debug library; compare bit for bit; no device error on either."""
    rel = call()
    rel = rel if isinstance(rel, tuple) else (rel,)
    rel = [_bits(t) for t in rel]
    rnl.rnl_check_device_error()
    with rnl.debug_library():
        assert rnl.rnl_debug_build()
        dbg = call()
        dbg = dbg if isinstance(dbg, tuple) else (dbg,)
        dbg = [_bits(t) for t in dbg]
        rnl.rnl_check_device_error()  # raises RnlError(RNL_ERR_BOUNDS) if a check fired
    for i, (a, b) in enumerate(zip(rel, dbg)):
        assert np.array_equal(a, b), f"output {i}: {(a != b).sum()} of {a.size} differ"


def test_selftest_check_fires():
    with rnl.debug_library():
        rnl.rnl_selftest_bounds_check()
        with pytest.raises(rnl.RnlError) as e:
            rnl.rnl_check_device_error()
        assert e.value.status == 10 and "site 98" in str(e.value)
        rnl.rnl_check_device_error()  # the word was cleared
    with pytest.raises(rnl.RnlError) as e:
        rnl.rnl_selftest_bounds_check()  # release build: not available
    assert e.value.status == 8


@pytest.mark.parametrize("T,K,N,pair", [
    (300, 520, 600, "0"),     # one CTA, ragged M, N, K tail
    (1000, 1024, 700, "1"),   # CTA pairs, data-parallel + stream-K
    (600, 3000, 1000, "1"),   # CTA pairs, every tile split
    (4, 4096, 2048, None),    # the decode-step kernel (CUDA cores)
    (3, 2056, 2000, "mma"),   # the decode-step kernel on the tensor cores, K split over 8 CTAs
])
def test_bf16(monkeypatch, T, K, N, pair):
    if pair == "mma":
        monkeypatch.setenv("RNL_DECODE_MMA", "1")
    elif pair is not None:
        monkeypatch.setenv("RNL_GEMM_PAIR", pair)
    d = si.make_projection(dict(seed=T + N, T=T, K=K, N=N))
    x, g, W = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"])
    _both(lambda: rnl.rmsnorm_linear_bf16(x, g, W))


@pytest.mark.parametrize("T,K,N", [(300, 20480, 24), (129, 16384, 64), (500, 1024, 200)])
def test_fp32_forms(T, K, N):
    d = si.make_projection(dict(seed=T + K, T=T, K=K, N=N, has_gamma=False))
    x, W = dev_bf16(d["x"]), dev_bf16(d["W"])
    _both(lambda: rnl.rmsnorm_linear_bf16(x, None, W, out_dtype=rnl.OUT_FP32))
    if N <= 64:
        _both(lambda: rnl.rmsnorm_linear_skinny_noalloc(x, W))


def test_ex_options():
    T, K, N = 260, 1032, 520
    d = si.make_projection(dict(seed=3, T=T, K=K, N=N))
    x, g, W = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"])
    res = dev_bf16(si.normal_bf16(3, "residual", (T, K), 1.0))
    beta = dev_bf16(si.normal_bf16(3, "beta", (K,), 0.1))
    bias = dev_bf16(si.normal_bf16(3, "bias", (N,), 0.5))

    def call():
        rstd = torch.empty(T, dtype=torch.float32, device="cuda")
        xs = torch.empty_like(x)
        out = rnl.rmsnorm_linear_bf16_ex(x, g, W, residual=res, x_sum_out=xs, beta=beta, bias=bias,
                                         rstd_out=rstd)
        return out, xs, rstd
    _both(call)


@pytest.mark.parametrize("pair", ["0", "1"])
def test_w8a8_and_s8(monkeypatch, pair):
    monkeypatch.setenv("RNL_GEMM_PAIR", pair)
    d = si.make_w8a8(dict(seed=9, T=300, K=2048, N=520))
    x, g, Wq, ws = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev(d["Wq"]), dev(d["w_scale"])

    def call():
        q = torch.empty((300, 2048), dtype=torch.int8, device="cuda")
        xs = torch.empty(300, dtype=torch.float32, device="cuda")
        return rnl.rmsnorm_linear_w8a8(x, g, Wq, ws, q_out=q, x_scale_out=xs), q, xs
    _both(call)

    def call_prepared():
        Wb = rnl.rnl_w8a8_prepare_weight(Wq)
        return Wb, rnl.rmsnorm_linear_w8a8_prepared(x, g, Wb, ws)
    _both(call_prepared)
    rng = np.random.default_rng(1)
    A = dev(rng.integers(-127, 128, (260, 2048)).astype(np.int8))
    B = dev(rng.integers(-127, 128, (300, 2048)).astype(np.int8))
    _both(lambda: rnl.rnl_gemm_s8s8s32(A, B))


def test_mla_and_head_norm():
    d = si.make_mla(dict(seed=4, T=200, K=1024, N1=512, N2=1024))
    args = (dev_bf16(d["x"]), dev_bf16(d["W_qa"]), dev_bf16(d["gamma_cq"]), dev_bf16(d["W_qb"]))
    _both(lambda: rnl.mla_q_chain(*args))
    _both(lambda: rnl.mla_q_chain_head_norm(*args, head_dim=128))


def test_qmrs():
    d = si.make_qmrs(dict(seed=5, B=3, M=130, K=272, N=208))
    args = (dev(d["x1"]), dev(d["x2"]), dev(d["x1_scale"]), dev_bf16(d["x2_scale"]))
    _both(lambda: rnl.quant_matmul_reduce_sum(*args))


def test_mxfp8():
    T, K, N = 200, 512, 384
    d = si.make_projection(dict(seed=6, T=T, K=K, N=N))
    rng = np.random.default_rng(6)
    wc = dev(rng.integers(0, 0x7E, (N, K)).astype(np.uint8))
    wsc = dev(rng.integers(118, 122, (N, K // 64)).astype(np.uint8))
    x, g = dev_bf16(d["x"]), dev_bf16(d["gamma"])

    def call():
        xc = torch.empty((T, K), dtype=torch.uint8, device="cuda")
        xsc = torch.empty((T, K // 64), dtype=torch.uint8, device="cuda")
        return rnl.rmsnorm_linear_mxfp8(x, g, wc, wsc, x_codes_out=xc, x_scale_out=xsc), xc, xsc
    _both(call)


@pytest.mark.parametrize("epilogue", ["1", "0"])
def test_qkv_rope(monkeypatch, epilogue):
    monkeypatch.setenv("RNL_QKV_ROPE_EPILOGUE", epilogue)
    monkeypatch.setenv("RNL_GEMM_PAIR", "1")
    T, K, Hq, Hkv, D = 300, 1024, 4, 2, 128
    N = (Hq + 2 * Hkv) * D
    d = si.make_projection(dict(seed=8, T=T, K=K, N=N))
    rng = np.random.default_rng(8)
    qg = dev_bf16(si.uniform_bf16(8, "qg", (D,), 0.5, 1.5))
    kg = dev_bf16(si.uniform_bf16(8, "kg", (D,), 0.5, 1.5))
    ang = rng.uniform(0, 6.3, (T, D // 2))
    cs = dev(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))
    pos = dev(np.arange(T, dtype=np.int32))
    x, g, W = dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"])
    _both(lambda: rnl.rmsnorm_linear_qkv_rope(x, g, W, Hq, Hkv, D, qg, kg, pos, cs))
