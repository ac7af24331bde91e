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


# ---------------------------------------------------------------------------
# The integer GEMM on CTA pairs without chunks.  For RMSNorm-quantised rows
# sum |q| <= K max|gamma| / x_scale + K/2; a tile whose rows all keep that
# bound below 2^24 / 128 is accumulated in one FP32 accumulator (every
# partial sum an integer below 2^24: exact), any other tile in 1024-product
# chunks.  Both must give the exact integer sums, so the output is the
# dequant of the exact sums: the same bits as the one-CTA kernel (always
# chunked) and as an FP32 emulation of the dequant on the exact products.

def _bf16_rne_bits(f32: np.ndarray) -> np.ndarray:
    b = f32.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _dequant_emulated(q, Wq, xs, ws):
    """bf16(float(acc) * (x_scale * w_scale)) in binary32, acc exact."""
    acc = q.astype(np.int64) @ Wq.astype(np.int64).T
    scale = (xs.astype(np.float32)[:, None] * ws.astype(np.float32)[None, :]).astype(np.float32)
    return _bf16_rne_bits((acc.astype(np.float32) * scale).astype(np.float32))


def _run_route(x, Wb, ws, pair, monkeypatch, T, K, gamma=None):
    monkeypatch.setenv("RNL_GEMM_PAIR", "1" if pair else "0")
    q = torch.empty((T, K), dtype=torch.int8, device="cuda")
    xs = torch.empty((T,), dtype=torch.float32, device="cuda")
    out = rnl.rmsnorm_linear_w8a8_prepared(x, gamma, Wb, ws, eps=1e-6, norm_mode=0, q_out=q, x_scale_out=xs)
    torch.cuda.synchronize()
    rnl.rnl_check_device_error()
    return host_bits(out), q.cpu().numpy(), xs.cpu().numpy()


def _const_rows(n_nonzero, K, rows, value=1.0):
    """rows x K bf16 bits: `value` in the first n_nonzero columns, 0 after."""
    x = np.zeros((rows, K), np.float32)
    x[:, :n_nonzero] = value
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _both_routes_exact(orc, monkeypatch, x, W, ws, T, K):
    xd, Wb, wsd = dev_bf16(x), rnl.rnl_w8a8_prepare_weight(dev(W)), dev(ws)
    got_pair = _run_route(xd, Wb, wsd, True, monkeypatch, T, K)
    got_one = _run_route(xd, Wb, wsd, False, monkeypatch, T, K)
    r = orc.rmsnorm_linear_w8a8(x, None, W, ws, 1e-6, 0)
    for got in (got_pair, got_one):  # the same front end on both routes, as the oracle's
        assert np.array_equal(got[1], r["q"]) and np.array_equal(got[2], r["x_scale"])
    want = _dequant_emulated(r["q"], W, r["x_scale"], ws)
    assert np.array_equal(got_one[0], want), "one-CTA chunked route"
    assert np.array_equal(got_pair[0], want), "pair route"
    assert_bf16_close(got_pair[0], r["out"], "pair route vs oracle")
    return got_pair[0], r


def test_unchunked_pair_tiles_exact_near_the_bound(orc, monkeypatch):
    """K = 1008: rows of equal values give x_scale = 1/127, just above the
    bound's floor, so their tiles take one FP32 accumulator although
    sum |q| = 127 * 1008 = 128016: products summing to 16.26 M, to -16.39 M
    (int8 -128 weights) and to exactly 0 after partial sums of 8.1 M."""
    monkeypatch.setenv("RNL_W8A8_STREAM", "1")
    T, K, N = 512, 1008, 264
    d = si.make_w8a8(dict(seed=45, T=T, K=K, N=N))
    x = d["x"].copy()
    x[:256] = _const_rows(K, K, 256)
    W = d["Wq"].copy()
    W[0] = 127
    W[1, :504], W[1, 504:] = 127, -127
    W[2] = -128
    out, r = _both_routes_exact(orc, monkeypatch, x, W, d["w_scale"], T, K)
    assert np.abs(r["q"][:256].astype(np.int64)).sum(1).min() == 127 * K
    assert (r["acc"][:256, 0] == 127 * 127 * K).all() and (r["acc"][:256, 2] == -128 * 127 * K).all()
    assert not bf16_bits_to_f64(out[:256, 1]).any()


def test_chunked_pair_tiles_exact_past_the_bound(orc, monkeypatch):
    """K = 4096: random rows (their tiles unchunked) beside rows of 1000,
    1100 and 4096 codes of 127 (their tiles in chunks: sum |q| up to 520192),
    with weight rows whose products cancel to exactly 0 after partial sums of
    8 M and 33 M."""
    monkeypatch.setenv("RNL_W8A8_STREAM", "1")
    T, K, N = 768, 4096, 512
    d = si.make_w8a8(dict(seed=41, T=T, K=K, N=N))
    x = d["x"].copy()
    x[256:512:2] = _const_rows(1100, K, 128)
    x[257:512:2] = _const_rows(K, K, 128)
    x[512:768] = _const_rows(1000, K, 256)
    W = d["Wq"].copy()
    W[0] = 0
    W[0, :500], W[0, 500:1000] = 127, -127          # 0 after +8 M
    W[1] = 0
    W[1, :2048], W[1, 2048:] = 127, -127             # 4096-code rows: 0 after +33 M
    W[2] = 127
    W[3] = -128
    out, r = _both_routes_exact(orc, monkeypatch, x, W, d["w_scale"], T, K)
    assert np.abs(r["q"][257:512:2].astype(np.int64)).sum(1).min() == 127 * K
    assert not bf16_bits_to_f64(out[512:, 0]).any()
    assert not bf16_bits_to_f64(out[257:512:2, 1]).any()


@pytest.mark.parametrize("T,N", [(1000, 1000), (8192, 4096)])
def test_pair_and_one_cta_integer_routes_identical(orc, monkeypatch, T, N):
    """Random rows (every tile within the bound): the pair route's single
    FP32 accumulator and stream-K FP32 partials give the one-CTA route's
    bits, and the FP32 emulation of the dequant on sampled rows."""
    monkeypatch.setenv("RNL_W8A8_STREAM", "1")
    K = 4096
    c = dict(seed=43 + T, T=T, K=K, N=N)
    d = si.make_w8a8(c)
    xd, Wb, wsd = dev_bf16(d["x"]), rnl.rnl_w8a8_prepare_weight(dev(d["Wq"])), dev(d["w_scale"])
    got_pair = _run_route(xd, Wb, wsd, True, monkeypatch, T, K)
    got_one = _run_route(xd, Wb, wsd, False, monkeypatch, T, K)
    assert np.array_equal(got_pair[1], got_one[1]) and np.array_equal(got_pair[2], got_one[2])
    assert np.array_equal(got_pair[0], got_one[0]), \
        f"{(got_pair[0] != got_one[0]).sum()} outputs differ between the routes"
    rows = sample_rows(T, 32, seed=T)
    want = _dequant_emulated(got_one[1][rows], d["Wq"], got_one[2][rows], d["w_scale"])
    assert np.array_equal(got_pair[0][rows], want)


def test_pair_route_past_the_mark_table_chunks_every_tile(orc, monkeypatch):
    """More 256-row blocks than the pair kernel's mark table holds (1024):
    every tile in 1024-product chunks on CTA pairs, the same bits as the
    one-CTA route, and the oracle's on sampled rows."""
    monkeypatch.setenv("RNL_W8A8_STREAM", "1")
    T, K, N = 1025 * 256 + 37, 64, 48
    d = si.make_w8a8(dict(seed=47, T=T, K=K, N=N))
    d["gamma"] = None  # the routes run without gamma
    xd, Wb, wsd = dev_bf16(d["x"]), rnl.rnl_w8a8_prepare_weight(dev(d["Wq"])), dev(d["w_scale"])
    got_pair = _run_route(xd, Wb, wsd, True, monkeypatch, T, K)
    got_one = _run_route(xd, Wb, wsd, False, monkeypatch, T, K)
    assert np.array_equal(got_pair[0], got_one[0])
    rows = sample_rows(T, 64, seed=3)
    _check(orc, d, 1e-6, 0, got_pair, rows)
