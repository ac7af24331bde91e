"""QKV split + per-head RMSNorm + RoPE (rnl_qkv_rope, and the whole chain
rmsnorm_linear_qkv_rope) against the oracle.

Bound for q and k, derived from the arithmetic: the normed values z are
rounded to bf16 on both sides, and the GPU's FP32 head norm may put one on
the other side of a bf16 rounding boundary than the oracle's binary64 norm
(one ulp, at most 2^-7 relative); an output mixes two of them with the table's
cos and sin and is rounded once more, so
    |gpu - oracle| <= 2^-7 * (|z_i c_i| + |z_partner s_i| + |o_oracle|) + 2^-20.
The oracle's z comes from the same stage run at angle 0.  v heads: bit-exact.

For the whole chain (projection, then this stage) the expected values are the
oracle's chain from the same x, W: its projection output y may differ from the
GPU's by one bf16 ulp where |y| is not small, which moves z by at most one
more ulp, so the factor is 2^-6 there; where y is near zero after
cancellation the projection's error is absolute (its FP32 accumulation), and
such elements are held to the acceptance bound 1e-2 * max(1, |oracle|)
instead.  v is held to the bf16 output bound instead of bit equality.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import dev_bf16, host_bits, sample_rows
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


def assert_rope_close(orc, got, want, y_bits, Hq, Hkv, D, qg, kg, eps, pos, cs, what, chain=False):
    T = y_bits.shape[0]
    ident = np.concatenate([np.ones((1, D // 2), np.float32), np.zeros((1, D // 2), np.float32)], axis=1)
    zq, zk, _ = orc.qkv_rope(y_bits, Hq, Hkv, D, qg, kg, eps, np.zeros(T, np.int32), ident)
    h = D // 2
    c = cs[pos, :h].astype(np.float64)[:, None, :]
    s = cs[pos, h:].astype(np.float64)[:, None, :]
    for g_bits, w_bits, z_bits, name in ((got[0], want[0], zq, "q"), (got[1], want[1], zk, "k")):
        if w_bits.size == 0:
            continue
        g, w, z = bf16_bits_to_f64(g_bits), bf16_bits_to_f64(w_bits), bf16_bits_to_f64(z_bits)
        za, zb = np.abs(z[..., :h]), np.abs(z[..., h:])
        lo = za * np.abs(c) + zb * np.abs(s)
        hi = zb * np.abs(c) + za * np.abs(s)
        factor = 2.0**-6 if chain else 2.0**-7
        bound = factor * (np.concatenate([lo, hi], axis=-1) + np.abs(w)) + 2.0**-20
        if chain:
            bound = np.maximum(bound, 1e-2 * np.maximum(1.0, np.abs(w)))
        err = np.abs(g - w)
        bad = err > bound
        assert not bad.any(), f"{what} {name}: {bad.sum()} outside the bound, max err {err.max()}"
    if chain:
        from gpu_util import assert_bf16_close
        assert_bf16_close(got[2], want[2], f"{what} v")
    else:
        assert np.array_equal(got[2], want[2]), f"{what} v"


def _case(seed, T, Hq, Hkv, D, P):
    rng = np.random.default_rng(seed)
    y = si.normal_bf16(seed, "y", (T, (Hq + 2 * Hkv) * D), 1.0)
    qg = si.uniform_bf16(seed, "q_gamma", (D,), 0.5, 1.5)
    kg = si.uniform_bf16(seed, "k_gamma", (D,), 0.5, 1.5)
    pos = rng.integers(0, P, T).astype(np.int32)
    cs = si.rope_table(P, D)
    return y, qg, kg, pos, cs


def _run(y, Hq, Hkv, D, qg, kg, pos, cs, eps=1e-6):
    q, k, v = rnl.rnl_qkv_rope(dev_bf16(y), Hq, Hkv, D, dev_bf16(qg), dev_bf16(kg),
                               torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda(), eps=eps)
    return host_bits(q), host_bits(k), host_bits(v)


@pytest.mark.parametrize("T,Hq,Hkv,D,P", [
    (37, 4, 2, 128, 64),
    (50, 3, 1, 64, 100),
    (9, 2, 2, 256, 17),
    (20, 3, 0, 128, 20),    # query heads only
    (1, 1, 1, 64, 1),
])
def test_qkv_rope_stage(orc, T, Hq, Hkv, D, P):
    y, qg, kg, pos, cs = _case(T * 7 + D, T, Hq, Hkv, D, P)
    got = _run(y, Hq, Hkv, D, qg, kg, pos, cs)
    want = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    assert_rope_close(orc, got, want, y, Hq, Hkv, D, qg, kg, 1e-6, pos, cs, f"stage {T}x{Hq}/{Hkv}x{D}")


def test_qkv_rope_chain_small(orc):
    """rmsnorm_linear_qkv_rope = the oracle's AT-10 projection, then its V stage."""
    T, K, Hq, Hkv, D, P = 300, 520, 4, 2, 128, 512
    N = (Hq + 2 * Hkv) * D
    d = si.make_projection(dict(seed=41, T=T, K=K, N=N, has_gamma=True))
    _, qg, kg, pos, cs = _case(42, T, Hq, Hkv, D, P)
    q, k, v = rnl.rmsnorm_linear_qkv_rope(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                          Hq, Hkv, D, dev_bf16(qg), dev_bf16(kg),
                                          torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda())
    _, y_ref = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    want = orc.qkv_rope(y_ref, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    got = (host_bits(q), host_bits(k), host_bits(v))
    assert_rope_close(orc, got, want, y_ref, Hq, Hkv, D, qg, kg, 1e-6, pos, cs, "chain", chain=True)


def test_qkv_rope_full_size_sampled(orc):
    """The qkv_rope workload's size (32 + 8 + 8 heads of 128, positions
    0..4095): whole chain on the GPU, sampled tokens against the oracle's
    projection + V stage."""
    c = si.CONFIGS["qkv_rope"]
    T, K, N, Hq, Hkv, D = c["T"], c["K"], c["N"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"]
    d = si.make_projection(c)
    r = si.make_qkv_rope(c)
    q, k, v = rnl.rmsnorm_linear_qkv_rope(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                          Hq, Hkv, D, dev_bf16(r["q_gamma"]), dev_bf16(r["k_gamma"]),
                                          torch.from_numpy(r["positions"]).cuda(),
                                          torch.from_numpy(r["cos_sin"]).cuda())
    rows = sample_rows(T, 40, seed=3)
    _, y_ref = orc.rmsnorm_linear(d["x"][rows], d["gamma"], d["W"], 1e-6, 0, 0)
    pos = r["positions"][rows]
    want = orc.qkv_rope(y_ref, Hq, Hkv, D, r["q_gamma"], r["k_gamma"], 1e-6, pos, r["cos_sin"])
    got = (host_bits(q)[rows], host_bits(k)[rows], host_bits(v)[rows])
    assert_rope_close(orc, got, want, y_ref, Hq, Hkv, D, r["q_gamma"], r["k_gamma"], 1e-6, pos,
                      r["cos_sin"], "full size", chain=True)


def test_qkv_rope_bad_position_is_reported_and_context_survives(orc):
    """A position outside the table: that token's q / k rows are skipped (no
    table read), rnl_check_device_error reports RNL_ERR_ARG, the other tokens
    are right and the context keeps working."""
    T, Hq, Hkv, D, P = 8, 2, 1, 64, 8
    y, qg, kg, pos, cs = _case(7, T, Hq, Hkv, D, P)
    rnl.rnl_check_device_error()
    pos_bad = pos.copy()
    pos_bad[3] = P  # one past the end
    got = _run(y, Hq, Hkv, D, qg, kg, pos_bad, cs)
    with pytest.raises(rnl.RnlError) as e:
        rnl.rnl_check_device_error()
    assert e.value.status == 4  # RNL_ERR_ARG
    rnl.rnl_check_device_error()  # cleared
    want = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    keep = np.array([t for t in range(T) if t != 3])
    assert_rope_close(orc, tuple(g[keep] for g in got), tuple(w[keep] for w in want), y[keep], Hq, Hkv, D,
                      qg, kg, 1e-6, pos[keep], cs, "good tokens")
    got2 = _run(y, Hq, Hkv, D, qg, kg, pos, cs)
    assert_rope_close(orc, got2, want, y, Hq, Hkv, D, qg, kg, 1e-6, pos, cs, "after the error")


@pytest.fixture
def rope_route(monkeypatch):
    """Set the environment that picks the chain's route (CTA pairs forced, the
    stage in the GEMM epilogue or separate)."""
    def set_route(pair, epilogue):
        monkeypatch.setenv("RNL_GEMM_PAIR", "1" if pair else "0")
        monkeypatch.setenv("RNL_QKV_ROPE_EPILOGUE", "1" if epilogue else "0")
    return set_route


@pytest.mark.parametrize("T,K,Hq,Hkv", [(300, 520, 4, 2), (777, 1024, 6, 3), (64, 256, 2, 1)])
def test_qkv_rope_chain_in_pair_epilogue(orc, rope_route, T, K, Hq, Hkv):
    """The stage fused into the CTA-pair GEMM's epilogue (forced onto pairs at
    sizes where stream-K finishers add partner partial sums before it), and
    the separate route on the same inputs: both against the oracle chain."""
    D, P = 128, 1000
    N = (Hq + 2 * Hkv) * D
    d = si.make_projection(dict(seed=T + K, T=T, K=K, N=N, has_gamma=True))
    _, qg, kg, pos, cs = _case(T + 1, T, Hq, Hkv, D, P)
    _, y_ref = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    want = orc.qkv_rope(y_ref, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    for epilogue in (True, False):
        rope_route(True, epilogue)
        q, k, v = rnl.rmsnorm_linear_qkv_rope(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                              Hq, Hkv, D, dev_bf16(qg), dev_bf16(kg),
                                              torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda())
        got = (host_bits(q), host_bits(k), host_bits(v))
        assert_rope_close(orc, got, want, y_ref, Hq, Hkv, D, qg, kg, 1e-6, pos, cs,
                          f"epilogue={epilogue}", chain=True)


def test_qkv_rope_epilogue_bad_position(orc, rope_route):
    """A bad position on the fused route: RNL_ERR_ARG, the other tokens right."""
    T, K, Hq, Hkv, D, P = 260, 256, 2, 1, 128, 64
    N = (Hq + 2 * Hkv) * D
    d = si.make_projection(dict(seed=9, T=T, K=K, N=N, has_gamma=True))
    _, qg, kg, pos, cs = _case(10, T, Hq, Hkv, D, P)
    pos_bad = pos.copy()
    pos_bad[7] = -1
    rope_route(True, True)
    rnl.rnl_check_device_error()
    q, k, v = rnl.rmsnorm_linear_qkv_rope(dev_bf16(d["x"]), dev_bf16(d["gamma"]), dev_bf16(d["W"]),
                                          Hq, Hkv, D, dev_bf16(qg), dev_bf16(kg),
                                          torch.from_numpy(pos_bad).cuda(), torch.from_numpy(cs).cuda())
    with pytest.raises(rnl.RnlError) as e:
        rnl.rnl_check_device_error()
    assert e.value.status == 4  # RNL_ERR_ARG
    rnl.rnl_check_device_error()  # cleared
    _, y_ref = orc.rmsnorm_linear(d["x"], d["gamma"], d["W"], 1e-6, 0, 0)
    want = orc.qkv_rope(y_ref, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    keep = np.array([t for t in range(T) if t != 7])
    got = (host_bits(q)[keep], host_bits(k)[keep], host_bits(v)[keep])
    assert_rope_close(orc, got, tuple(w[keep] for w in want), y_ref[keep], Hq, Hkv, D, qg, kg, 1e-6, pos[keep],
                      cs, "good tokens", chain=True)
