"""W8A8 (rmsnorm_linear_w8a8, rnl_w8a8_prepare_weight +
rmsnorm_linear_w8a8_prepared) against the oracle through the C ABI.

Codes and x_scale bit for bit: the front end's FP32 steps are the oracle's
(the FP32 sum of squares is the rounding of the exact sum, every later step
one correctly rounded operation).  The int32 accumulation is exact, so the
bf16 output differs from the oracle's only by the dequant's FP32 rounding
against binary64: within the acceptance bound.

Routes: the weight prepared once; the weight widened in every call; and the
three-read row kernels of the front end (RNL_W8A8_STREAM=0) in place of the
streamed quantiser.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import assert_bf16_close, dev, dev_bf16, host_bits, sample_rows
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


@pytest.fixture(params=["prepared", "per_call", "row_kernels"])
def route(request, monkeypatch):
    monkeypatch.setenv("RNL_W8A8_STREAM", "0" if request.param == "row_kernels" else "1")
    yield request.param
    rnl.rnl_check_device_error()


def _run(d, eps, mode, route):
    T, K = d["x"].shape
    q = torch.empty((T, K), dtype=torch.int8, device="cuda")
    xs = torch.empty((T,), dtype=torch.float32, device="cuda")
    g = dev_bf16(d["gamma"]) if d["gamma"] is not None else None
    if route == "prepared":
        Wb = rnl.rnl_w8a8_prepare_weight(dev(d["Wq"]))
        out = rnl.rmsnorm_linear_w8a8_prepared(dev_bf16(d["x"]), g, Wb, dev(d["w_scale"]), eps=eps,
                                               norm_mode=mode, q_out=q, x_scale_out=xs)
    else:
        out = rnl.rmsnorm_linear_w8a8(dev_bf16(d["x"]), g, dev(d["Wq"]), dev(d["w_scale"]), eps=eps,
                                      norm_mode=mode, q_out=q, x_scale_out=xs)
    return host_bits(out), q.cpu().numpy(), xs.cpu().numpy()


def _check(orc, d, eps, mode, got, rows=None):
    out, q, xs = got
    x = d["x"] if rows is None else d["x"][rows]
    r = orc.rmsnorm_linear_w8a8(x, d["gamma"], d["Wq"], d["w_scale"], eps, mode)
    if rows is not None:
        out, q, xs = out[rows], q[rows], xs[rows]
    assert np.array_equal(q, r["q"]), f"INT8 codes: {(q != r['q']).sum()} differ"
    assert np.array_equal(xs, r["x_scale"]), "x_scale differs"
    assert_bf16_close(out, r["out"], "w8a8 out")
    return r


@pytest.mark.parametrize("T,K,N,mode", [
    (200, 2048, 300, 0), (130, 4096, 520, 1), (5, 16, 7, 0),
    (40, 1024, 64, 0),
    (64, 6144, 136, 1),    # rows longer than 4096: the three-read row kernels on every route
    (33, 8704, 96, 0),     # a row length that is not a multiple of 1024 elements
    (700, 4096, 256, 0),   # several 8-row groups per CTA in the streamed quantiser
    (9, 4080, 48, 1),      # ragged last lane stride; 1/K not a power of two (sqrt+div form)
])
def test_w8a8_small(orc, route, T, K, N, mode):
    d = si.make_w8a8(dict(seed=3 + T + N, T=T, K=K, N=N))
    _check(orc, d, 1e-6, mode, _run(d, 1e-6, mode, route))


def test_w8a8_zero_and_no_gamma(orc, route):
    d = si.make_w8a8(dict(seed=5, T=12, K=64, N=16))
    d["x"][2] = 0
    got = _run(d, 1e-6, 0, route)
    assert not got[1][2].any() and got[2][2] == 0.0
    assert not bf16_bits_to_f64(got[0][2]).any()
    _check(orc, d, 1e-6, 0, got)
    d["gamma"] = None
    _check(orc, d, 1e-6, 1, _run(d, 1e-6, 1, route))


def _tie_rows(orc, K=256, want=6, seed=17):
    """Rows whose largest |x * gamma| is an exact tie between two elements with
    different factors (3s * 5 and 5s * 3), placed so that the later element
    (the one the quantiser's keyed maximum picks) rounds to the smaller |y|:
    the maximum must then come from the check pass, not from the guess."""
    rng = np.random.default_rng(seed)
    rows, gam = [], None
    g = np.ones(K, np.float32)
    g[10], g[20] = 5.0, 3.0
    gbits = (g.view(np.uint32) >> 16).astype(np.uint16)
    tries = 0
    while len(rows) < want and tries < 20000:
        tries += 1
        s = np.float32(2.0 ** rng.integers(-3, 3)) * np.float32(rng.choice([1.0, 1.25, 1.5, 1.75]))
        x = (rng.standard_normal(K) * 0.05).astype(np.float32)
        x[10], x[20] = 3 * s, 5 * s  # |x g| = 15 s for both
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)
        if not np.array_equal((xb.astype(np.uint32) << 16).view(np.float32)[[10, 20]], [3 * s, 5 * s]):
            continue
        _, _, rstd, _ = orc.quant_rows_f32(xb[None, :], gbits, 1e-6, 0)
        r = np.float32(rstd[0])
        y10 = np.float32(np.float32(np.float32(3 * s) * r) * np.float32(5))
        y20 = np.float32(np.float32(np.float32(5 * s) * r) * np.float32(3))
        if y20 < y10:  # the keyed maximum (higher position) holds the smaller y
            rows.append(xb)
    assert len(rows) == want, f"only {len(rows)} tie rows in {tries} tries"
    return np.stack(rows), gbits


def test_w8a8_amax_ties_take_the_check_pass(orc, route):
    x, g = _tie_rows(orc)
    T, K = x.shape
    d = {"x": x, "gamma": g, "Wq": si.uniform_int8(3, "Wq", (32, K), -127, 127),
         "w_scale": si.uniform_f32(3, "w_scale", (32,), 1e-3, 1e-2)}
    _check(orc, d, 1e-6, 0, _run(d, 1e-6, 0, route))


def test_w8a8_full_sampled(orc, route):
    c = si.CONFIGS["w8a8"]
    d = si.make_w8a8(c)
    rows = sample_rows(c["T"], 48)
    r = _check(orc, d, c["eps"], c["norm_mode"], _run(d, c["eps"], c["norm_mode"], route), rows)
    # the int32 accumulation of the full-size run is exact: recompute the
    # sampled rows' products from the oracle's own codes through the INT8 hook
    C = rnl.rnl_gemm_s8s8s32(dev(r["q"]), dev(d["Wq"])).cpu().numpy()
    assert np.array_equal(C, r["acc"])


def test_prepared_weight_is_the_exact_integers():
    rng = np.random.default_rng(4)
    Wq = rng.integers(-127, 128, (300, 272)).astype(np.int8)
    Wb = rnl.rnl_w8a8_prepare_weight(dev(Wq)).float().cpu().numpy()
    assert np.array_equal(Wb, Wq.astype(np.float32))
