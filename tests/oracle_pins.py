"""Pins for the CPU oracle: checks against facts fixed by the method's
definition and by mathematics, never by re-typing the oracle's own formula.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle is wrong.  ``test_oracle_pins.py`` runs them on the real oracle and
``test_oracle_mutants.py`` runs them on copies of the oracle with a planted
mistake, to show that each plausible mistake fails at least one pin.

Kinds of pin used (sources: the AT-10 pattern page, sec. 3 "RMSNorm
variants", sec. 4 "Linear modes", sec. 5 "MLAProlog"; the SK-03 skeleton
page, "quantised variant (AT-11)"; the SK-14 skeleton page,
"QuantMatMulReduceSum"):
  * closed forms: constant rows, one-hot rows, constructed exact ties;
  * invariants: scale invariance, identity / permutation weights, the
    composition of the two-stage chain, the skinny-form fold;
  * brute force: exact rationals (fractions + 60-digit decimal) on tiny
    inputs, Python integers for the int8 matmul, a table search for bf16;
  * library cross-checks: torch.nn.functional.rms_norm and matmul in float64.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

import exact
from oracle import bf16_bits_to_f64


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_bits_of_f32(v):
    """Standard float32 -> bf16 bit trick (independent of the oracle's codec)."""
    a = np.asarray(v, dtype=np.float32)
    b = np.ascontiguousarray(a.reshape(-1)).view(np.uint32)
    r = ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    return r.reshape(a.shape) if a.ndim else r[0]


def _rand_bf16(rng, shape, sigma=1.0):
    return _bf16_bits_of_f32((rng.standard_normal(shape) * sigma).astype(np.float32))


# ---------------------------------------------------------------------------
# bf16 codec
# ---------------------------------------------------------------------------

def pin_bf16_codec(orc):
    cases = {
        1.0: 0x3F80, -2.0: 0xC000, 0.0: 0x0000,
        1.0 + 2.0**-8: 0x3F80,            # tie -> even (down)
        1.0 + 3 * 2.0**-8: 0x3F82,        # tie -> even (up)
        1.0 + 2.0**-8 + 2.0**-30: 0x3F81,  # just above the tie
        2.0**-133: 0x0001,                # smallest subnormal
        2.0**-134: 0x0000,                # half of it: tie -> even (zero)
        3 * 2.0**-134: 0x0002,            # 1.5 quanta: tie -> even (2)
        (2 - 2.0**-7) * 2.0**127: 0x7F7F,  # largest finite
        (2 - 2.0**-8) * 2.0**127: 0x7F80,  # max + half ulp overflows (tie, odd max)
        float("inf"): 0x7F80, -float("inf"): 0xFF80,
    }
    for v, want in cases.items():
        got = int(orc.bf16_rne(v)[0])
        assert got == want, (v, hex(got), hex(want))
    assert int(orc.bf16_rne(-0.0)[0]) == 0x8000
    assert (int(orc.bf16_rne(float("nan"))[0]) & 0x7FFF) > 0x7F80
    # round trip of every finite pattern
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        vals = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    fin = np.isfinite(vals)
    back = orc.bf16_rne(vals[fin])
    assert np.array_equal(back, bits[fin].astype(np.uint16))
    # binary32 inputs: the well-known bit trick on the float's bits
    rng = _rng(1)
    f = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    assert np.array_equal(orc.bf16_rne(f.astype(np.float64)), _bf16_bits_of_f32(f))
    # binary64 inputs: brute force against the table of neighbours
    d = rng.standard_normal(400) * np.exp(rng.uniform(-80, 80, 400))
    got = orc.bf16_rne(d)
    for v, g in zip(d, got):
        want, _ = exact.bf16_round_exact(float(v))
        assert int(g) == want, (v, hex(int(g)), hex(want))


# ---------------------------------------------------------------------------
# AT-03 RMSNorm
# ---------------------------------------------------------------------------

def pin_rmsnorm_variants_agree(orc):
    rng = _rng(2)
    for K in (7, 256, 1000, 4096):
        x = _rand_bf16(rng, (6, K), 3.0)
        g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
        ya, ra = orc.rmsnorm_f64(x, g, 1e-6, 0)
        yb, rb = orc.rmsnorm_f64(x, g, 1e-6, 1)
        assert np.allclose(ra, rb, rtol=4e-16 * 8, atol=0), (K, np.max(np.abs(ra / rb - 1)))
        assert np.allclose(ya, yb, rtol=4e-15, atol=0)


def pin_rmsnorm_closed_forms(orc):
    K = 64
    g = _bf16_bits_of_f32(np.linspace(0.5, 1.5, K).astype(np.float32))
    gv = bf16_bits_to_f64(g)
    for variant in (0, 1):
        for c in (0.75, -3.0, 1e-3):
            x = np.full((1, K), _bf16_bits_of_f32(np.float32(c)), np.uint16)
            cv = bf16_bits_to_f64(x[0, 0])
            eps = 1e-6
            y, r = orc.rmsnorm_f64(x, g, eps, variant)
            want_r = exact.dec_sqrt_recip(Fraction(cv) ** 2 + Fraction(eps))
            assert exact.rel_close(r[0], want_r, 4e-16 * 4), (variant, c)
            want_y = np.array([float(Fraction(cv) * want_r * Fraction(gk)) for gk in gv])
            assert np.allclose(y[0], want_y, rtol=1e-15, atol=0)
            # eps = 0: a constant row normalises to +-gamma exactly up to rounding
            y0, _ = orc.rmsnorm_f64(x, g, 0.0, variant)
            assert np.allclose(y0[0], np.sign(cv) * gv, rtol=2e-16 * 4, atol=0)
        # one-hot row: y_j = sign(c) * sqrt(K) * gamma_j, zero elsewhere (eps = 0)
        for j, c in ((0, 2.0), (17, -0.5), (K - 1, 9.0)):
            x = np.zeros((1, K), np.uint16)
            x[0, j] = _bf16_bits_of_f32(np.float32(c))
            y, _ = orc.rmsnorm_f64(x, g, 0.0, variant)
            want = np.zeros(K)
            want[j] = np.sign(c) * np.sqrt(K) * gv[j]
            assert np.allclose(y[0], want, rtol=4e-16 * 4, atol=0), (variant, j)


def pin_rmsnorm_scale_invariance(orc):
    rng = _rng(3)
    x = _rand_bf16(rng, (4, 300))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, 300).astype(np.float32))
    xv = bf16_bits_to_f64(x)
    for variant in (0, 1):
        y1, _ = orc.rmsnorm_f64(x, g, 0.0, variant)
        for j in (-3, 1, 5):
            xs = orc.bf16_rne(xv * 2.0**j).reshape(x.shape)  # exact power-of-two scaling
            assert np.array_equal(bf16_bits_to_f64(xs), xv * 2.0**j)
            y2, _ = orc.rmsnorm_f64(xs, g, 0.0, variant)
            assert np.allclose(y1, y2, rtol=4e-16 * 4, atol=0), (variant, j)


def pin_rmsnorm_exact_small(orc):
    """Brute force: rstd and y from exact rationals (60-digit square root)."""
    rng = _rng(4)
    for variant in (0, 1):
        for K in (1, 3, 8):
            x = _rand_bf16(rng, (3, K))
            g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
            eps = 1e-6
            y, r = orc.rmsnorm_f64(x, g, eps, variant)
            for t in range(3):
                xs = [Fraction(exact.bf16_value(b)) for b in x[t]]
                ms = sum(v * v for v in xs) / K
                rr = exact.dec_sqrt_recip(ms + Fraction(eps))
                assert exact.rel_close(r[t], rr, 1e-15), (variant, K, t)
                for k in range(K):
                    want = xs[k] * rr * Fraction(exact.bf16_value(g[k]))
                    assert exact.rel_close(y[t, k], want, 1e-15) or abs(float(want)) < 1e-300


def pin_rmsnorm_torch(orc):
    import torch
    rng = _rng(5)
    x = _rand_bf16(rng, (16, 512), 2.0)
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    xt = torch.from_numpy(bf16_bits_to_f64(x))
    gt = torch.from_numpy(bf16_bits_to_f64(g))
    want = torch.nn.functional.rms_norm(xt, (512,), weight=gt, eps=1e-6).numpy()
    for variant in (0, 1):
        y, _ = orc.rmsnorm_f64(x, g, 1e-6, variant)
        assert np.allclose(y, want, rtol=1e-14, atol=1e-300)


# ---------------------------------------------------------------------------
# AT-10 RMSNorm + Linear (form 0) and the FP32 mhc_pre form (form 1)
# ---------------------------------------------------------------------------

def pin_linear_identity_and_permutation(orc):
    rng = _rng(6)
    K = 48
    x = _rand_bf16(rng, (5, K))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    one = _bf16_bits_of_f32(np.float32(1.0))
    y, _ = orc.rmsnorm_f64(x, g, 1e-6, 0)
    a_bits = orc.bf16_rne(y.ravel()).reshape(y.shape)
    # W = I: the projection returns the bf16-cast normed activations unchanged
    W = np.zeros((K, K), np.uint16)
    W[np.arange(K), np.arange(K)] = one
    _, out = orc.rmsnorm_linear(x, g, W, 1e-6, 0, 0)
    assert np.array_equal(out, a_bits)
    # W[n, k] = 1 iff k == perm[n]: out[:, n] = a[:, perm[n]] (catches a transposed W)
    perm = rng.permutation(K)
    Wp = np.zeros((K, K), np.uint16)
    Wp[np.arange(K), perm] = one
    _, outp = orc.rmsnorm_linear(x, g, Wp, 1e-6, 0, 0)
    assert np.array_equal(outp, a_bits[:, perm])
    # N != K, rectangular: rows of W pick single features, with a scale of 2
    two = _bf16_bits_of_f32(np.float32(2.0))
    Wr = np.zeros((7, K), np.uint16)
    cols = rng.choice(K, 7, replace=False)
    Wr[np.arange(7), cols] = two
    _, outr = orc.rmsnorm_linear(x, g, Wr, 1e-6, 0, 0)
    assert np.array_equal(bf16_bits_to_f64(outr), 2.0 * bf16_bits_to_f64(a_bits[:, cols]))


def pin_linear_exact_small(orc):
    """Brute force of the whole AT-10 row on tiny shapes in exact rationals."""
    rng = _rng(7)
    for (T, K, N) in ((2, 3, 2), (3, 8, 5), (1, 5, 8)):
        x = _rand_bf16(rng, (T, K))
        g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
        W = _rand_bf16(rng, (N, K), 0.5)
        eps = 1e-6
        ref, out = orc.rmsnorm_linear(x, g, W, eps, 0, 0)
        for t in range(T):
            xs = [Fraction(exact.bf16_value(b)) for b in x[t]]
            rr = exact.dec_sqrt_recip(sum(v * v for v in xs) / K + Fraction(eps))
            a = []
            for k in range(K):
                bits, near = exact.bf16_round_exact(xs[k] * rr * Fraction(exact.bf16_value(g[k])))
                assert not near  # the generator never hits a bf16 tie here
                a.append(Fraction(exact.bf16_value(bits)))
            for n in range(N):
                s = sum(a[k] * Fraction(exact.bf16_value(W[n, k])) for k in range(K))
                assert exact.rel_close(ref[t, n], s, 1e-15) or abs(float(s)) < 1e-300
                bits, near = exact.bf16_round_exact(s)
                assert near or int(out[t, n]) == bits, (T, K, N, t, n)


def pin_linear_torch(orc):
    import torch
    rng = _rng(8)
    T, K, N = 12, 320, 40
    x = _rand_bf16(rng, (T, K))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    W = _rand_bf16(rng, (N, K), 0.02)
    ref, out = orc.rmsnorm_linear(x, g, W, 1e-6, 0, 0)
    xt = torch.from_numpy(bf16_bits_to_f64(x))
    y = torch.nn.functional.rms_norm(xt, (K,), weight=torch.from_numpy(bf16_bits_to_f64(g)), eps=1e-6)
    a = y.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    want = a @ torch.from_numpy(bf16_bits_to_f64(W)).T
    scale = (a.abs() @ torch.from_numpy(np.abs(bf16_bits_to_f64(W))).T).numpy()
    # a may differ in rare elements by one bf16 step (double rounding in torch)
    assert np.all(np.abs(ref - want.numpy()) <= 2.0**-7 * scale * 0.05 + 1e-12 * scale)
    # form 1 without gamma equals rstd * (x @ W^T): the skinny-form fold
    ref1, out1 = orc.rmsnorm_linear(x, None, W, 1e-6, 0, 1)
    xv, wv = bf16_bits_to_f64(x), bf16_bits_to_f64(W)
    rstd = 1.0 / np.sqrt(np.mean(xv * xv, axis=1) + 1e-6)
    fold = rstd[:, None] * (xv @ wv.T)
    assert np.allclose(ref1, fold, rtol=1e-12, atol=1e-14)
    assert np.array_equal(out1, ref1.astype(np.float32))


def pin_linear_form1_gamma(orc):
    """Form 1 keeps the normed values unrounded: with W = I it returns them."""
    rng = _rng(9)
    K = 32
    x = _rand_bf16(rng, (3, K))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    W = np.zeros((K, K), np.uint16)
    W[np.arange(K), np.arange(K)] = _bf16_bits_of_f32(np.float32(1.0))
    y, _ = orc.rmsnorm_f64(x, g, 1e-6, 0)
    ref, out = orc.rmsnorm_linear(x, g, W, 1e-6, 0, 1)
    assert np.array_equal(ref, y)
    assert np.array_equal(out, y.astype(np.float32))


# ---------------------------------------------------------------------------
# MLA two-stage chain
# ---------------------------------------------------------------------------

def pin_mla_composition(orc):
    rng = _rng(10)
    T, K, N1, N2 = 4, 96, 40, 24
    x = _rand_bf16(rng, (T, K))
    Wa = _rand_bf16(rng, (N1, K), 0.1)
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, N1).astype(np.float32))
    Wb = _rand_bf16(rng, (N2, N1), 0.1)
    qa, ref, out = orc.mla_q_chain(x, Wa, g, Wb, 1e-6, 1)
    # stage 1 equals the bf16 rounding of an independent float64 matmul
    s1 = bf16_bits_to_f64(x) @ bf16_bits_to_f64(Wa).T
    for t in range(T):
        for j in range(N1):
            bits, near = exact.bf16_round_exact(float(s1[t, j]))
            assert near or int(qa[t, j]) == bits
    # stage 2 equals the single-stage AT-10 oracle applied to the stage-1 output
    ref2, out2 = orc.rmsnorm_linear(qa, g, Wb, 1e-6, 1, 0)
    assert np.array_equal(ref, ref2) and np.array_equal(out, out2)
    # and the gamma really is applied: gamma = 1 gives a different result
    ones = np.full(N1, _bf16_bits_of_f32(np.float32(1.0)), np.uint16)
    _, _, out_1 = orc.mla_q_chain(x, Wa, ones, Wb, 1e-6, 1)
    assert not np.array_equal(out, out_1)


# ---------------------------------------------------------------------------
# W8A8: per-token symmetric INT8 quant, exact INT32 matmul, dequant
# ---------------------------------------------------------------------------

def pin_quant_constructed_ties(orc):
    # x chosen so that sum x^2 / 8 + eps = 4096 exactly: rstd = 1/64, amax = 127/64,
    # qs = 64, and y * qs returns x exactly -> the codes are rint_half_even(x).
    x = np.array([[127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 0.0]], np.float32)
    ms = float(np.sum(x.astype(np.float64) ** 2)) / 8
    eps = 4096.0 - ms
    xb = _bf16_bits_of_f32(x)
    for variant in (0, 1):
        q, xs, rstd, v = orc.quant_rows_f32(xb, None, eps, variant)
        assert rstd[0] == np.float32(1 / 64)
        assert np.array_equal(v[0], x[0])
        assert q[0].tolist() == [127, 2, 4, -2, 0, 2, 0, 0]
        assert xs[0] == np.float32(127 / 64 / 127)


def pin_quant_properties(orc):
    rng = _rng(11)
    T, K = 24, 512
    x = _rand_bf16(rng, (T, K))
    x[3] = 0  # an all-zero row
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    for variant in (0, 1):
        q, xs, rstd, v = orc.quant_rows_f32(x, g, 1e-6, variant)
        assert q.min() >= -127 and q.max() <= 127
        y64, r64 = orc.rmsnorm_f64(x, g, 1e-6, variant)
        for t in range(T):
            if t == 3:
                assert not q[t].any() and xs[t] == 0.0
                continue
            assert np.abs(q[t]).max() == 127
            amax = np.abs(y64[t]).max()
            assert abs(float(xs[t]) - amax / 127) <= 1e-6 * amax / 127
            assert abs(float(rstd[t]) - r64[t]) <= 1e-6 * r64[t]
            # reconstruction error of the symmetric code: at most half a step
            err = np.abs(q[t].astype(np.float64) * float(xs[t]) - y64[t])
            assert np.all(err <= 0.5 * float(xs[t]) * (1 + 1e-4))
            # the code is the nearest integer to v (ties to even)
            assert np.all(np.abs(q[t] - v[t].astype(np.float64)) <= 0.5)
            assert np.array_equal(q[t], np.clip(np.rint(v[t]), -127, 127).astype(np.int8))


def _sum_of_squares_rows(rng, T, K):
    """bf16 rows whose binary32 sum of squares depends on the order of the
    additions.  Row kinds (cycled): one entry 2^12 first and the rest in
    (-1, 1) -- every small square is below half a unit in the last place of
    2^24, so a left-to-right binary32 sum returns 2^24 exactly while the
    exact sum is larger by about K/3; big entries 2^12 at the head of every
    64-element block with small ones between (a blocked or tree-shaped
    binary32 sum loses them too); one entry 1.5 * 2^12 and the rest ~N(0,1)
    (the running sum's last place is 4, so each addition rounds)."""
    rows = np.zeros((T, K), np.float32)
    for t in range(T):
        kind = t % 3
        if kind == 0:
            rows[t] = rng.uniform(-0.99, 0.99, K)
            rows[t, 0] = 4096.0
        elif kind == 1:
            rows[t] = rng.uniform(-0.99, 0.99, K)
            rows[t, ::64] = 4096.0
        else:
            rows[t] = rng.standard_normal(K)
            rows[t, 0] = 6144.0
    return _bf16_bits_of_f32(rows)


def _rstd_exact_sum_reading(xrow_bits, eps, variant):
    """rstd of the binary32 norm under the reading "the FP32 sum of squares is
    the binary32 rounding of the exact sum of the binary32 terms", every later
    step one correctly rounded binary32 operation, computed in exact rationals
    (AT-10 pattern page, sec. 3: the two RMSNorm variants in FP32).  K must be
    a power of two (1/K exact)."""
    K = xrow_bits.size
    assert K & (K - 1) == 0
    f32 = exact.f32_round_exact
    inv_d = Fraction(1, K)
    # each term: an exact binary64 product rounded once to binary32
    v = bf16_bits_to_f64(xrow_bits)
    terms = (v * v).astype(np.float32)
    if variant == 1:
        terms = (terms.astype(np.float64) * (1.0 / K)).astype(np.float32)
    # their exact sum: every binary32 value is an integer multiple of 2^-149
    total = sum(int(a) for a in np.ldexp(terms.astype(np.float64), 149).astype(object))
    s = f32(Fraction(total, 2**149))
    e = Fraction(float(np.float32(eps)))
    var = f32(f32(s * inv_d) + e) if variant == 0 else f32(s + e)
    return f32(1 / exact.f32_sqrt_exact(var))


def pin_quant_sum_of_squares_reading(orc):
    # The FP32 norm of the W8A8 and MXFP8 front ends decides integer codes, so
    # its sum of squares is fixed as one rounding of the exact sum.  Rows where
    # the order of binary32 additions changes the sum pin rstd (bit for bit)
    # against that reading in exact rationals, then the codes and scales that
    # follow from it (independent float32 steps; torch's E4M3 conversion).
    rng = _rng(13)
    T, K = 3, 4096
    x = _sum_of_squares_rows(rng, T, K)
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    eps = 1e-6
    xf = bf16_bits_to_f64(x).astype(np.float32)
    gf = bf16_bits_to_f64(g).astype(np.float32)
    for variant in (0, 1):
        q, xs, rstd, _ = orc.quant_rows_f32(x, g, eps, variant)
        want = np.array([float(_rstd_exact_sum_reading(x[t], eps, variant)) for t in range(T)], np.float32)
        assert np.array_equal(rstd, want), (variant, rstd, want)
        y = (xf * want[:, None]) * gf[None, :]  # binary32 products, as the method's FP32 norm
        amax = np.abs(y).max(axis=1)
        assert np.array_equal(xs, amax / np.float32(127))
        qs = np.float32(127) / amax
        assert np.array_equal(q, np.clip(np.rint(y * qs[:, None]), -127, 127).astype(np.int8))
        codes, scales = orc.mxfp8_quant_rows(x, g, eps, variant)
        want_c, want_s = _mx_expected(y.astype(np.float64))
        assert np.array_equal(scales, want_s) and np.array_equal(codes, want_c)


def pin_gemm_s8_bruteforce(orc):
    rng = _rng(12)
    for (M, N, K) in ((1, 1, 1), (3, 4, 5), (5, 7, 33)):
        A = rng.integers(-127, 128, (M, K)).astype(np.int8)
        B = rng.integers(-127, 128, (N, K)).astype(np.int8)
        C, ovf = orc.gemm_s8(A, B)
        assert not ovf
        for m in range(M):
            for n in range(N):
                assert int(C[m, n]) == sum(int(A[m, k]) * int(B[n, k]) for k in range(K))
    A = rng.integers(-127, 128, (17, 300)).astype(np.int8)
    B = rng.integers(-127, 128, (9, 300)).astype(np.int8)
    C, _ = orc.gemm_s8(A, B)
    assert np.array_equal(C, A.astype(np.int64) @ B.astype(np.int64).T)
    # worst case fits int32 up to K = 133144 (127*127*K <= 2^31 - 1)
    for K, want_ovf in ((1024, False), (133144, False), (133145, True)):
        A = np.full((1, K), 127, np.int8)
        B = np.full((2, K), 127, np.int8)
        B[1] = -127
        C, ovf = orc.gemm_s8(A, B)
        assert ovf == want_ovf
        if not want_ovf:
            assert int(C[0, 0]) == 127 * 127 * K and int(C[0, 1]) == -127 * 127 * K


def pin_dequant_exact(orc):
    rng = _rng(13)
    acc = rng.integers(-2**31, 2**31, (3, 5)).astype(np.int32)
    xs = rng.uniform(1e-3, 1.0, 3).astype(np.float32)
    ws = rng.uniform(1e-3, 1e-2, 5).astype(np.float32)
    ref, out = orc.dequant_bf16(acc, xs, ws)
    for m in range(3):
        for n in range(5):
            want = Fraction(int(acc[m, n])) * Fraction(float(xs[m])) * Fraction(float(ws[n]))
            assert exact.rel_close(ref[m, n], want, 2.3e-16)
            bits, near = exact.bf16_round_exact(want)
            assert near or int(out[m, n]) == bits


def pin_w8a8_composition(orc):
    rng = _rng(14)
    T, K, N = 6, 128, 20
    x = _rand_bf16(rng, (T, K))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    Wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    ws = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    r = orc.rmsnorm_linear_w8a8(x, g, Wq, ws, 1e-6, 0)
    q, xs, _, _ = orc.quant_rows_f32(x, g, 1e-6, 0)
    assert np.array_equal(r["q"], q) and np.array_equal(r["x_scale"], xs)
    assert np.array_equal(r["acc"], q.astype(np.int64) @ Wq.astype(np.int64).T)
    ref, out = orc.dequant_bf16(r["acc"], xs, ws)
    assert np.array_equal(r["out"], out)
    # and the quantised path approximates the unquantised FP32 form closely
    yv, _ = orc.rmsnorm_f64(x, g, 1e-6, 0)
    full = (yv @ Wq.astype(np.float64).T) * ws[None, :]
    assert np.allclose(r["ref"], full, rtol=0, atol=0.02 * np.abs(full).max())


# ---------------------------------------------------------------------------
# AT-10 with the residual add (x_add), the AT-03 norm bias and output_rstd,
# and the AT-09 projection bias
# ---------------------------------------------------------------------------

def pin_ex_reduces_to_base(orc):
    """With every option off the extended form is the AT-10 form itself."""
    rng = _rng(20)
    T, K, N = 9, 72, 30
    x = _rand_bf16(rng, (T, K))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    W = _rand_bf16(rng, (N, K), 0.05)
    for variant in (0, 1):
        ref, out = orc.rmsnorm_linear(x, g, W, 1e-6, variant, 0)
        ref2, out2, xs, r = orc.rmsnorm_linear_ex(x, None, g, None, W, None, 1e-6, variant)
        _, r_base = orc.rmsnorm_f64(x, g, 1e-6, variant)
        assert np.array_equal(out, out2) and np.array_equal(ref, ref2)
        assert np.array_equal(xs, x) and np.array_equal(r, r_base)


def pin_ex_residual_sum_exact(orc):
    """x_add = bf16(x + residual) with one rounding of the exact sum: random
    pairs against brute force, constructed ties (to even), a summand far
    below half an ulp, and cancellation to zero."""
    rng = _rng(21)
    K = 64
    x = _rand_bf16(rng, (4, K))
    res = _rand_bf16(rng, (4, K), 0.7)
    # constructed rows: 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7 -> 1 (even);
    # (1 + 2^-7) + 2^-8 is the midpoint of 1 + 2^-7 and 1 + 2^-6 -> 1 + 2^-6;
    # 1 + 2^-30 -> 1; x + (-x) -> 0
    one = _bf16_bits_of_f32(np.float32(1.0))
    x[0, :4] = [one, _bf16_bits_of_f32(np.float32(1 + 2**-7)), one, x[0, 3]]
    res[0, :4] = [_bf16_bits_of_f32(np.float32(2**-8)), _bf16_bits_of_f32(np.float32(2**-8)),
                  _bf16_bits_of_f32(np.float32(2**-30)), x[0, 3] ^ np.uint16(0x8000)]
    W = _rand_bf16(rng, (8, K), 0.05)
    _, _, xs, _ = orc.rmsnorm_linear_ex(x, res, None, None, W, None, 1e-6, 0)
    for t in range(4):
        for k in range(K):
            want, _ = exact.bf16_round_exact(Fraction(exact.bf16_value(x[t, k])) +
                                             Fraction(exact.bf16_value(res[t, k])))
            assert int(xs[t, k]) & 0x7FFF == want & 0x7FFF, (t, k)
            if want & 0x7FFF:
                assert int(xs[t, k]) == want, (t, k)
    assert bf16_bits_to_f64(xs[0, :4]).tolist() == [1.0, 1 + 2**-6, 1.0, 0.0]


def pin_ex_residual_composition(orc):
    """The norm and projection see x_add: the extended form on (x, residual)
    equals the AT-10 form on the x_sum it reports, rstd included; swapping x
    and residual changes nothing (the sum commutes)."""
    rng = _rng(22)
    T, K, N = 7, 96, 20
    x = _rand_bf16(rng, (T, K))
    res = _rand_bf16(rng, (T, K), 2.0)
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    W = _rand_bf16(rng, (N, K), 0.05)
    for variant in (0, 1):
        ref, out, xs, r = orc.rmsnorm_linear_ex(x, res, g, None, W, None, 1e-6, variant)
        ref_b, out_b = orc.rmsnorm_linear(xs, g, W, 1e-6, variant, 0)
        _, r_b = orc.rmsnorm_f64(xs, g, 1e-6, variant)
        assert np.array_equal(out, out_b) and np.array_equal(ref, ref_b) and np.array_equal(r, r_b)
        ref_s, out_s, xs_s, r_s = orc.rmsnorm_linear_ex(res, x, g, None, W, None, 1e-6, variant)
        assert np.array_equal(out, out_s) and np.array_equal(xs, xs_s) and np.array_equal(r, r_s)
    # rstd of a row whose x_add is constant c: 1/sqrt(c^2 + eps)
    xc = np.full((1, K), _bf16_bits_of_f32(np.float32(1.5)), np.uint16)
    rc = np.full((1, K), _bf16_bits_of_f32(np.float32(0.5)), np.uint16)
    _, _, _, r = orc.rmsnorm_linear_ex(xc, rc, None, None, W, None, 1e-6, 0)
    assert exact.rel_close(r[0], exact.dec_sqrt_recip(Fraction(4) + Fraction(1e-6)), 1e-15)


def pin_ex_norm_bias_closed_form(orc):
    """Constant row c with gamma g and norm bias b, W = I:
    out_k = bf16(bf16(c / sqrt(c^2 + eps) * g_k + b_k)) -- the bias comes after
    gamma and before the bf16 cast."""
    rng = _rng(23)
    K = 16
    one = _bf16_bits_of_f32(np.float32(1.0))
    W = np.zeros((K, K), np.uint16)
    W[np.arange(K), np.arange(K)] = one
    for c in (0.75, -3.0):
        x = np.full((1, K), _bf16_bits_of_f32(np.float32(c)), np.uint16)
        g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
        b = _bf16_bits_of_f32(rng.uniform(-2.0, 2.0, K).astype(np.float32))
        for variant in (0, 1):
            _, out, _, _ = orc.rmsnorm_linear_ex(x, None, g, b, W, None, 1e-6, variant)
            cf = Fraction(exact.bf16_value(x[0, 0]))
            rr = exact.dec_sqrt_recip(cf * cf + Fraction(1e-6))
            for k in range(K):
                y = cf * rr * Fraction(exact.bf16_value(g[k])) + Fraction(exact.bf16_value(b[k]))
                a_bits, near = exact.bf16_round_exact(y)
                assert near or int(out[0, k]) == a_bits, (c, variant, k)


def pin_ex_projection_bias(orc):
    """W = 0 gives out = bias exactly; with two unit weights per row,
    out = bf16(a_i + a_j + bias) rounded once (not bf16(bf16(a_i + a_j) + bias))."""
    rng = _rng(24)
    T, K, N = 5, 40, 12
    x = _rand_bf16(rng, (T, K))
    bias = _rand_bf16(rng, (N,), 3.0)
    W0 = np.zeros((N, K), np.uint16)
    _, out, _, _ = orc.rmsnorm_linear_ex(x, None, None, None, W0, bias, 1e-6, 0)
    assert np.array_equal(out, np.tile(bias, (T, 1)))
    one = _bf16_bits_of_f32(np.float32(1.0))
    W = np.zeros((N, K), np.uint16)
    pairs = [(rng.integers(0, K), rng.integers(0, K)) for _ in range(N)]
    for n, (i, j) in enumerate(pairs):
        W[n, i] = one
        W[n, j] = one if i != j else _bf16_bits_of_f32(np.float32(2.0))
    y, _ = orc.rmsnorm_f64(x, None, 1e-6, 0)
    a = [[Fraction(exact.bf16_value(exact.bf16_round_exact(Fraction(float(v)))[0])) for v in row] for row in y]
    _, out, _, _ = orc.rmsnorm_linear_ex(x, None, None, None, W, bias, 1e-6, 0)
    for t in range(T):
        for n, (i, j) in enumerate(pairs):
            s = a[t][i] + a[t][j] + Fraction(exact.bf16_value(bias[n]))
            want, near = exact.bf16_round_exact(s)
            assert near or int(out[t, n]) == want, (t, n)


def pin_ex_exact_small(orc):
    """Brute force of the whole extended row, every option on, in exact
    rationals (fractions + 60-digit square root)."""
    rng = _rng(25)
    for (T, K, N) in ((2, 3, 2), (3, 8, 5)):
        x = _rand_bf16(rng, (T, K))
        res = _rand_bf16(rng, (T, K), 0.5)
        g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
        b = _rand_bf16(rng, (K,), 0.3)
        W = _rand_bf16(rng, (N, K), 0.5)
        bias = _rand_bf16(rng, (N,), 0.3)
        for variant in (0, 1):
            ref, out, xs, r = orc.rmsnorm_linear_ex(x, res, g, b, W, bias, 1e-6, variant)
            for t in range(T):
                xa = []
                for k in range(K):
                    bits, _ = exact.bf16_round_exact(Fraction(exact.bf16_value(x[t, k])) +
                                                     Fraction(exact.bf16_value(res[t, k])))
                    assert int(xs[t, k]) == bits
                    xa.append(Fraction(exact.bf16_value(bits)))
                rr = exact.dec_sqrt_recip(sum(v * v for v in xa) / K + Fraction(1e-6))
                assert exact.rel_close(r[t], rr, 1e-15)
                a = []
                for k in range(K):
                    y = xa[k] * rr * Fraction(exact.bf16_value(g[k])) + Fraction(exact.bf16_value(b[k]))
                    bits, near = exact.bf16_round_exact(y)
                    assert not near
                    a.append(Fraction(exact.bf16_value(bits)))
                for n in range(N):
                    sacc = sum(a[k] * Fraction(exact.bf16_value(W[n, k])) for k in range(K))
                    sacc += Fraction(exact.bf16_value(bias[n]))
                    assert exact.rel_close(ref[t, n], sacc, 1e-15) or abs(float(sacc)) < 1e-300
                    bits, near = exact.bf16_round_exact(sacc)
                    assert near or int(out[t, n]) == bits, (T, K, N, variant, t, n)


def pin_ex_torch(orc):
    """Library cross-check: torch (float64) add, rms_norm, + beta, bf16 cast,
    matmul + bias."""
    import torch
    rng = _rng(26)
    T, K, N = 10, 256, 24
    x = _rand_bf16(rng, (T, K))
    res = _rand_bf16(rng, (T, K), 1.5)
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    b = _rand_bf16(rng, (K,), 0.1)
    W = _rand_bf16(rng, (N, K), 0.02)
    bias = _rand_bf16(rng, (N,), 0.5)
    ref, out, xs, r = orc.rmsnorm_linear_ex(x, res, g, b, W, bias, 1e-6, 0)
    xa = (torch.from_numpy(bf16_bits_to_f64(x)) + torch.from_numpy(bf16_bits_to_f64(res)))
    # the f64 sum is exact; so is its float32 copy while the two exponents are
    # within 16 of each other (true of these draws), so this rounds once
    xa_b = xa.to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(xa_b.view(torch.int16).numpy().view(np.uint16), xs)
    xa_d = xa_b.to(torch.float64)
    y = torch.nn.functional.rms_norm(xa_d, (K,), weight=torch.from_numpy(bf16_bits_to_f64(g)), eps=1e-6)
    y = y + torch.from_numpy(bf16_bits_to_f64(b))
    rstd = 1.0 / torch.sqrt((xa_d * xa_d).mean(dim=1) + 1e-6)
    assert np.allclose(r, rstd.numpy(), rtol=1e-14, atol=0)
    a = y.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    wt = torch.from_numpy(bf16_bits_to_f64(W))
    want = a @ wt.T + torch.from_numpy(bf16_bits_to_f64(bias))
    scale = (a.abs() @ wt.abs().T).numpy() + np.abs(bf16_bits_to_f64(bias))
    assert np.all(np.abs(ref - want.numpy()) <= 2.0**-7 * scale * 0.05 + 1e-12 * scale)


# ---------------------------------------------------------------------------
# QKV split + per-head RMSNorm + RoPE after the qkv projection (AT-10 page,
# sec. 6, Qwen3PreAttn)
# ---------------------------------------------------------------------------

def _qkv_case(rng, T=3, Hq=2, Hkv=1, D=8):
    y = _rand_bf16(rng, (T, (Hq + 2 * Hkv) * D))
    qg = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    kg = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    return y, qg, kg


def _table(cos, sin, D, P=1):
    """A one-row-per-position table with the same angle for every pair."""
    t = np.empty((P, D), np.float32)
    t[:, : D // 2] = cos
    t[:, D // 2:] = sin
    return t


def pin_rope_angle_zero_is_head_norm(orc):
    """At angle 0 (cos 1, sin 0) the rotation is the identity: q and k are the
    bf16 per-head RMSNorm of their column ranges (the pinned rmsnorm_f64 on the
    reshaped heads), v is y's last columns unchanged."""
    rng = _rng(30)
    T, Hq, Hkv, D = 5, 4, 2, 16
    y, qg, kg = _qkv_case(rng, T, Hq, Hkv, D)
    q, k, v = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, np.zeros(T, np.int32), _table(1.0, 0.0, D))
    yq = y[:, : Hq * D].reshape(T * Hq, D)
    yk = y[:, Hq * D:(Hq + Hkv) * D].reshape(T * Hkv, D)
    for got, heads, g in ((q, yq, qg), (k, yk, kg)):
        ref, _ = orc.rmsnorm_f64(heads, g, 1e-6, 0)
        want = orc.bf16_rne(ref.ravel()).reshape(got.shape)
        diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
        assert diff.max() <= 1 and (diff == 0).mean() > 0.99
    assert np.array_equal(v.reshape(T, -1), y[:, (Hq + Hkv) * D:])


def pin_rope_quarter_and_half_turn(orc):
    """cos 0, sin 1: o[i] = -z[i + D/2], o[i + D/2] = z[i] exactly (rotate-half
    pairing, sign); cos -1, sin 0: o = -z exactly."""
    rng = _rng(31)
    T, Hq, Hkv, D = 4, 2, 2, 16
    y, qg, kg = _qkv_case(rng, T, Hq, Hkv, D)
    pos = np.zeros(T, np.int32)
    z, zk, _ = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, _table(1.0, 0.0, D))
    q, k, _ = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, _table(0.0, 1.0, D))
    h = D // 2
    for got, base in ((q, z), (k, zk)):
        assert np.array_equal(got[..., :h], base[..., h:] ^ np.uint16(0x8000))
        assert np.array_equal(got[..., h:], base[..., :h])
    q2, _, _ = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, _table(-1.0, 0.0, D))
    assert np.array_equal(q2, z ^ np.uint16(0x8000))


def pin_rope_positions_index_the_table(orc):
    """Each token uses its own table row: a token at position p gives the same
    output as the same token alone with a one-row table holding row p."""
    rng = _rng(32)
    T, Hq, Hkv, D = 6, 2, 1, 8
    y, qg, kg = _qkv_case(rng, T, Hq, Hkv, D)
    P = 9
    ang = rng.uniform(-3, 3, (P, D // 2))
    cs = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    pos = rng.integers(0, P, T).astype(np.int32)
    q, k, v = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    for t in range(T):
        q1, k1, _ = orc.qkv_rope(y[t:t + 1], Hq, Hkv, D, qg, kg, 1e-6, np.zeros(1, np.int32),
                                 cs[pos[t]:pos[t] + 1])
        assert np.array_equal(q1[0], q[t]) and np.array_equal(k1[0], k[t])


def pin_rope_exact_small(orc):
    """Brute force in exact rationals: the head norm (60-digit square root),
    the bf16 cast of the normed values, the rotation with the fp32 table
    values, the final bf16 cast."""
    rng = _rng(33)
    T, Hq, Hkv, D = 2, 1, 1, 8
    y, qg, kg = _qkv_case(rng, T, Hq, Hkv, D)
    P = 3
    ang = rng.uniform(-3, 3, (P, D // 2))
    cs = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    pos = np.array([2, 1], np.int32)
    q, k, _ = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    h = D // 2
    for t in range(T):
        for got, col0, g in ((q[t, 0], 0, qg), (k[t, 0], Hq * D, kg)):
            row = [Fraction(exact.bf16_value(b)) for b in y[t, col0:col0 + D]]
            r = exact.dec_sqrt_recip(sum(a * a for a in row) / D + Fraction(1e-6))
            z = []
            for i in range(D):
                bits, near = exact.bf16_round_exact(row[i] * r * Fraction(exact.bf16_value(g[i])))
                assert not near
                z.append(Fraction(exact.bf16_value(bits)))
            c = [Fraction(float(x)) for x in cs[pos[t], :h]]
            sn = [Fraction(float(x)) for x in cs[pos[t], h:]]
            for i in range(h):
                for val, idx in ((z[i] * c[i] - z[i + h] * sn[i], i), (z[i + h] * c[i] + z[i] * sn[i], i + h)):
                    bits, near = exact.bf16_round_exact(val)
                    assert near or int(got[idx]) == bits, (t, idx)


def pin_rope_torch(orc):
    """Library cross-check: torch float64 rms_norm per head, bf16 cast, the
    rotate-half rotation (x * cos + rotate_half(x) * sin)."""
    import torch
    rng = _rng(34)
    T, Hq, Hkv, D = 8, 4, 2, 64
    y, qg, kg = _qkv_case(rng, T, Hq, Hkv, D)
    import synth_inputs as si
    cs = si.rope_table(16, D)
    pos = rng.integers(0, 16, T).astype(np.int32)
    q, k, _ = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, pos, cs)
    yt = torch.from_numpy(bf16_bits_to_f64(y))
    cos = torch.from_numpy(cs[pos, : D // 2].astype(np.float64))
    sin = torch.from_numpy(cs[pos, D // 2:].astype(np.float64))
    cos = torch.cat([cos, cos], dim=1)[:, None, :]
    sin = torch.cat([sin, sin], dim=1)[:, None, :]
    for got, lo, H, g in ((q, 0, Hq, qg), (k, Hq * D, Hkv, kg)):
        heads = yt[:, lo:lo + H * D].reshape(T, H, D)
        z = torch.nn.functional.rms_norm(heads, (D,), weight=torch.from_numpy(bf16_bits_to_f64(g)), eps=1e-6)
        z = z.to(torch.float32).to(torch.bfloat16).to(torch.float64)
        rot = torch.cat([-z[..., D // 2:], z[..., : D // 2]], dim=-1)
        want = z * cos + rot * sin
        err = np.abs(bf16_bits_to_f64(got) - want.numpy())
        assert np.all(err <= 2.0**-7 * np.abs(want.numpy()) + 1e-6), err.max()


def pin_rope_small_rows_closed_form(orc):
    """A constant head row c with c^2 of the order of eps: at angle 0 the
    output is bf16(c * gamma / sqrt(c^2 + eps)), far from +-gamma, so the eps
    of the per-head norm is visible."""
    D, Hq, Hkv = 8, 1, 1
    qg = _bf16_bits_of_f32(np.linspace(0.5, 1.5, D).astype(np.float32))
    kg = _bf16_bits_of_f32(np.linspace(1.5, 0.5, D).astype(np.float32))
    for c in (2.0**-10, -(2.0**-11)):
        cb = _bf16_bits_of_f32(np.float32(c))
        y = np.full((1, (Hq + 2 * Hkv) * D), cb, np.uint16)
        q, k, _ = orc.qkv_rope(y, Hq, Hkv, D, qg, kg, 1e-6, np.zeros(1, np.int32), _table(1.0, 0.0, D))
        cf = Fraction(c)
        r = exact.dec_sqrt_recip(cf * cf + Fraction(1e-6))
        for got, g in ((q[0, 0], qg), (k[0, 0], kg)):
            for i in range(D):
                bits, near = exact.bf16_round_exact(cf * r * Fraction(exact.bf16_value(g[i])))
                assert near or int(got[i]) == bits, (c, i)


def pin_rope_rejects_bad_position(orc):
    rng = _rng(35)
    y, qg, kg = _qkv_case(rng, 2, 1, 1, 8)
    for bad in (-1, 4):
        try:
            orc.qkv_rope(y, 1, 1, 8, qg, kg, 1e-6, np.array([0, bad], np.int32), _table(1.0, 0.0, 8, P=4))
        except RuntimeError:
            continue
        raise AssertionError(f"position {bad} accepted")


# ---------------------------------------------------------------------------
# QuantMatMulReduceSum (SK-14 skeleton page, variant A)
# ---------------------------------------------------------------------------

def _qmrs_case(rng, B, M, K, N, lo=-127, hi=127):
    x1 = rng.integers(lo, hi + 1, (B, M, K)).astype(np.int8)
    x2 = rng.integers(lo, hi + 1, (B, K, N)).astype(np.int8)
    return x1, x2


def pin_qmrs_unit_scales_exact(orc):
    """Unit scales: every step is exact while the sums stay below 2^24, so the
    output is the bf16 rounding of the exact integer sum over the batch
    (Python integers, x2 read as [K, N])."""
    rng = _rng(40)
    for (B, M, K, N) in ((1, 3, 5, 4), (3, 4, 16, 6)):
        x1, x2 = _qmrs_case(rng, B, M, K, N)
        xs = np.ones((B, M), np.float32)
        ws = np.full(N, _bf16_bits_of_f32(np.float32(1.0)), np.uint16)
        _, out = orc.quant_matmul_reduce_sum(x1, x2, xs, ws)
        for m in range(M):
            for n in range(N):
                tot = sum(int(x1[b, m, k]) * int(x2[b, k, n]) for b in range(B) for k in range(K))
                bits, near = exact.bf16_round_exact(tot)
                assert near or int(out[m, n]) == bits, (B, m, n)


def pin_qmrs_x2_is_k_by_n(orc):
    """x2[b] a permutation matrix of ones (K = N): out[m, n] sums x1[b, m, k]
    over the batch at the k with x2[b, k, n] = 1 (catches a transposed x2)."""
    rng = _rng(41)
    B, M, K = 2, 5, 12
    x1, _ = _qmrs_case(rng, B, M, K, K, -10, 10)
    x2 = np.zeros((B, K, K), np.int8)
    perms = [rng.permutation(K) for _ in range(B)]
    for b in range(B):
        x2[b, perms[b], np.arange(K)] = 1  # x2[b, perm[n], n] = 1
    xs = np.ones((B, M), np.float32)
    ws = np.full(K, _bf16_bits_of_f32(np.float32(1.0)), np.uint16)
    _, out = orc.quant_matmul_reduce_sum(x1, x2, xs, ws)
    want = sum(x1[b][:, perms[b]].astype(np.float64) for b in range(B))
    assert np.array_equal(bf16_bits_to_f64(out), want)


def pin_qmrs_power_of_two_scales(orc):
    """Multiplying x1_scale by 4 and x2_scale by 1/2 doubles every FP32 step
    exactly, so the output doubles bit for bit."""
    rng = _rng(42)
    B, M, K, N = 3, 6, 64, 10
    x1, x2 = _qmrs_case(rng, B, M, K, N)
    xs = rng.uniform(1e-3, 1e-2, (B, M)).astype(np.float32)
    ws = _bf16_bits_of_f32(rng.uniform(1e-3, 1e-2, N).astype(np.float32))
    ref, out = orc.quant_matmul_reduce_sum(x1, x2, xs, ws)
    ws_half = _bf16_bits_of_f32((bf16_bits_to_f64(ws) / 2).astype(np.float32))
    ref2, out2 = orc.quant_matmul_reduce_sum(x1, x2, xs * np.float32(4), ws_half)
    assert np.array_equal(ref2, ref * np.float32(2))
    assert np.array_equal(bf16_bits_to_f64(out2), 2 * bf16_bits_to_f64(out))


def pin_qmrs_batch_structure(orc):
    """Two batches in either order give the same sum (a + b = b + a in IEEE);
    a trailing batch of zeros changes nothing; batch b uses x1_scale[b]."""
    rng = _rng(43)
    B, M, K, N = 2, 4, 32, 8
    x1, x2 = _qmrs_case(rng, B, M, K, N)
    xs = rng.uniform(1e-3, 1e-2, (B, M)).astype(np.float32)
    ws = _bf16_bits_of_f32(rng.uniform(1e-3, 1e-2, N).astype(np.float32))
    ref, out = orc.quant_matmul_reduce_sum(x1, x2, xs, ws)
    ref_s, _ = orc.quant_matmul_reduce_sum(x1[::-1], x2[::-1], xs[::-1], ws)
    assert np.array_equal(ref, ref_s)
    z1 = np.concatenate([x1, np.zeros((1, M, K), np.int8)])
    z2 = np.concatenate([x2, x2[:1]])
    zs = np.concatenate([xs, xs[:1]])
    ref_z, _ = orc.quant_matmul_reduce_sum(z1, z2, zs, ws)
    assert np.array_equal(ref_z, ref)
    # the scale of batch 1 applies to batch 1 only: zeroing it leaves batch 0
    xs0 = xs.copy()
    xs0[1] = 0
    ref0, _ = orc.quant_matmul_reduce_sum(x1, x2, xs0, ws)
    ref_b0, _ = orc.quant_matmul_reduce_sum(x1[:1], x2[:1], xs[:1], ws)
    assert np.array_equal(ref0, ref_b0)


def pin_qmrs_numpy_float32(orc):
    """Library cross-check: numpy int64 matmul per batch, then the page's
    FP32 steps with numpy float32 scalars in the same order."""
    rng = _rng(44)
    B, M, K, N = 4, 5, 96, 7
    x1, x2 = _qmrs_case(rng, B, M, K, N)
    xs = rng.uniform(1e-3, 1e-2, (B, M)).astype(np.float32)
    ws = _bf16_bits_of_f32(rng.uniform(1e-3, 1e-2, N).astype(np.float32))
    wsf = bf16_bits_to_f64(ws).astype(np.float32)
    ref, _ = orc.quant_matmul_reduce_sum(x1, x2, xs, ws)
    acc = np.einsum("bmk,bkn->bmn", x1.astype(np.int64), x2.astype(np.int64))
    want = np.zeros((M, N), np.float32)
    for b in range(B):
        sc = xs[b][:, None] * wsf[None, :]
        want = want + acc[b].astype(np.float32) * sc
    assert np.array_equal(ref, want)


def pin_qmrs_overflow(orc):
    """|acc| > 2^31 - 1 is reported (the page's INT32 result cannot hold it)."""
    K = 133200  # 127 * 127 * K > 2^31 - 1
    x1 = np.full((1, 1, K), 127, np.int8)
    x2 = np.full((1, K, 1), 127, np.int8)
    try:
        orc.quant_matmul_reduce_sum(x1, x2, np.ones((1, 1), np.float32),
                                    np.full(1, _bf16_bits_of_f32(np.float32(1.0)), np.uint16))
    except OverflowError:
        return
    raise AssertionError("overflow not reported")


# ---------------------------------------------------------------------------
# MXFP8 (AT-09 quant_mode mxfp8; GMM-MXFP8 layout: E4M3FN data, E8M0FNU
# scale factors, one scale per 64 elements)
# ---------------------------------------------------------------------------

def _torch_e4m3_decode(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _torch_e4m3_encode(vals):
    """Round to nearest even through torch's float8_e4m3fn (valid for |v| < 464,
    where torch and a saturating conversion agree)."""
    import torch
    t = torch.from_numpy(np.asarray(vals, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def pin_e4m3_codec(orc):
    # facts of the format: bias 7, 3 mantissa bits, no infinity, S.1111.111 NaN
    known = {0x00: 0.0, 0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x08: 2.0**-6, 0x38: 1.0, 0x39: 1.125,
             0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in known.items():
        assert orc.e4m3_value(c) == v, hex(c)
    assert np.isnan(orc.e4m3_value(0x7F)) and np.isnan(orc.e4m3_value(0xFF))
    allc = np.arange(256, dtype=np.uint8)
    mine = np.array([orc.e4m3_value(int(c)) for c in allc])
    ref = _torch_e4m3_decode(allc)
    both_nan = np.isnan(mine) & np.isnan(ref)
    assert np.array_equal(mine[~both_nan], ref[~both_nan]) and both_nan.sum() == 2
    pos = mine[1:0x7F]
    assert np.all(np.diff(pos) > 0) and pos.size == 126  # monotone in the code
    # encoding: ties to even, the subnormal range, saturation to +-448
    enc = {1.0625: 0x38, 1.1875: 0x3A, 2.0**-10: 0x00, 3 * 2.0**-10: 0x02, 7.5 * 2.0**-9: 0x08,
           -1.0625: 0xB8, 448.0: 0x7E, 449.0: 0x7E, 464.0: 0x7E, 480.0: 0x7E, 1e30: 0x7E,
           -1e30: 0xFE, 0.1: 0x1D, 15.5 * 2.0**-10: 0x08}
    for v, c in enc.items():
        assert orc.e4m3_rne_sat(v) == c, (v, hex(orc.e4m3_rne_sat(v)), hex(c))
    assert orc.e4m3_rne_sat(0.0) == 0x00 and orc.e4m3_rne_sat(-0.0) == 0x80
    rng = _rng(60)
    v = np.concatenate([rng.standard_normal(3000) * 50, rng.standard_normal(3000) * 2.0**-7,
                        rng.uniform(-463, 463, 2000), np.ldexp(rng.uniform(-1, 1, 1000), -9)]).astype(np.float32)
    got = np.array([orc.e4m3_rne_sat(float(a)) for a in v], np.uint8)
    assert np.array_equal(got, _torch_e4m3_encode(v))
    # every finite code is a fixed point; midpoints go to the even neighbour
    for c in range(0x7F):
        assert orc.e4m3_rne_sat(orc.e4m3_value(c)) == c
        if c < 0x7E:
            mid = (orc.e4m3_value(c) + orc.e4m3_value(c + 1)) / 2
            assert orc.e4m3_rne_sat(mid) == (c if c % 2 == 0 else c + 1)


def pin_e8m0_scale(orc):
    assert orc.e8m0_value(127) == 1.0 and orc.e8m0_value(128) == 2.0 and orc.e8m0_value(119) == 2.0**-8
    assert orc.e8m0_value(0) == 2.0**-127 and orc.e8m0_value(254) == 2.0**127
    assert np.isnan(orc.e8m0_value(255))


def _mx_expected(y, block=64):
    """Codes and scale bytes of the MX rule for exact y (a closed form: shared
    exponent floor(log2 amax) - 8 via numpy's frexp, codes through torch's
    float8 conversion, saturation applied to the block maximum's range)."""
    T, K = y.shape
    codes = np.zeros((T, K), np.uint8)
    scales = np.zeros((T, K // block), np.uint8)
    for t in range(T):
        for b in range(K // block):
            blk = y[t, b * block:(b + 1) * block].astype(np.float64)
            amax = np.abs(blk).max()
            X = -127 if amax == 0 else max(-127, int(np.frexp(amax)[1]) - 1 - 8)
            scales[t, b] = X + 127
            v = np.ldexp(blk, -X)
            sat = np.abs(v) > 448
            c = _torch_e4m3_encode(np.where(sat, 0.0, v).astype(np.float32))
            c[sat] = np.where(v[sat] > 0, 0x7E, 0xFE)
            codes[t, b * block:(b + 1) * block] = c
    return codes, scales


def pin_mxfp8_constructed_ties(orc):
    # x and eps chosen so that the binary32 mean of squares plus eps rounds to
    # 4096 exactly (the tiny entries' squares are far below its last bit):
    # rstd = 1/64 and y = x / 64.
    # The block maximum y = 1.5 gives X = -8 (y * 256 = 384); the other
    # entries land on E4M3 ties, on the subnormal range and (row 1) on
    # saturation (y * 256 = 488 > 448).
    base = [96.0, 17 / 64, 19 / 64, -17 / 64, 2.0**-12, 3 * 2.0**-12, 7.5 * 2.0**-11, 0.0]
    rows = [base + [0.0] * 56, [122.0] + base[1:] + [0.0] * 56]
    want = [[0x7C, 0x38, 0x3A, 0xB8, 0x00, 0x02, 0x08, 0x00], [0x7E, 0x38, 0x3A, 0xB8, 0x00, 0x02, 0x08, 0x00]]
    for x, w in zip(rows, want):
        x = np.array([x], np.float32)
        xb = _bf16_bits_of_f32(x)
        assert np.array_equal(bf16_bits_to_f64(xb), x.astype(np.float64))
        ms = sum(Fraction(float(v)) ** 2 for v in x[0]) / 64
        eps = float(np.float32(float(Fraction(4096) - ms)))
        assert abs(Fraction(eps) + ms - 4096) <= Fraction(1, 2**13)  # within half an ulp below 4096
        for variant in (0, 1):
            assert orc.quant_rows_f32(xb, None, eps, variant)[2][0] == np.float32(1 / 64)
            codes, scales = orc.mxfp8_quant_rows(xb, None, eps, variant)
            assert scales.tolist() == [[119]]  # X = -8
            assert codes[0, :8].tolist() == w and not codes[0, 8:].any()


def pin_mxfp8_gamma_closed_form(orc):
    # x = 1 everywhere and eps = 0: rstd = 1 exactly in both variants, y = gamma
    rng = _rng(61)
    K = 256
    g = _bf16_bits_of_f32(rng.uniform(-3, 3, K).astype(np.float32))
    g[64:128] = _bf16_bits_of_f32((rng.uniform(-1, 1, 64) * 2.0**-20).astype(np.float32))
    g[128:192] = 0
    x = np.full((2, K), 0x3F80, np.uint16)
    x[1] = 0xC000  # -2: rstd = 1/2, y = -gamma
    y = np.stack([bf16_bits_to_f64(g), -bf16_bits_to_f64(g)])
    want_c, want_s = _mx_expected(y)
    assert want_s[0, 2] == 0  # a zero block: X = -127, zero codes
    for variant in (0, 1):
        codes, scales = orc.mxfp8_quant_rows(x, g, 0.0, variant)
        assert np.array_equal(scales, want_s) and np.array_equal(codes, want_c)


def pin_mxfp8_block_structure_and_bound(orc):
    rng = _rng(62)
    T, K = 12, 512
    x = _rand_bf16(rng, (T, K))
    x[:, 64:128] = _bf16_bits_of_f32((rng.standard_normal((T, 64)) * 1e-3).astype(np.float32))  # a quiet block
    x[2, :] = 0
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    for variant in (0, 1):
        codes, scales = orc.mxfp8_quant_rows(x, g, 1e-6, variant)
        assert scales.shape == (T, K // 64)
        assert not codes[2].any() and (scales[2] == 0).all()
        y64, _ = orc.rmsnorm_f64(x, g, 1e-6, variant)
        for t in range(T):
            if t == 2:
                continue
            for b in range(K // 64):
                blk = y64[t, b * 64:(b + 1) * 64]
                amax = np.abs(blk).max()
                X = int(scales[t, b]) - 127
                # the shared exponent puts the block maximum in [256, 512)
                assert 256 * (1 - 1e-6) <= amax * 2.0**-X < 512 * (1 + 1e-6), (t, b)
                dq = np.array([orc.e4m3_value(c) for c in codes[t, b * 64:(b + 1) * 64]]) * 2.0**X
                v = blk * 2.0**-X
                # half a step of the E4M3 grid at each magnitude (2^-10 in the
                # subnormal range), or the saturation of values above 448
                step = np.where(np.abs(v) < 2.0**-6, 2.0**-9,
                                2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 2.0**-6))) - 3))
                tol = np.where(np.abs(v) > 448, np.abs(v) - 448, step / 2) * (1 + 1e-5) + 1e-6 * np.abs(v)
                assert np.all(np.abs(dq * 2.0**-X - v) <= tol), (t, b)
        # the quiet block has its own, smaller scale
        assert (scales[[0, 1, 3], 1] < scales[[0, 1, 3], 0] - 5).all()
        # rows are independent
        assert np.array_equal(codes[1:], orc.mxfp8_quant_rows(x[1:], g, 1e-6, variant)[0])
    # block 32 (the OCP MX block) is the same rule on half blocks
    c64, s64 = orc.mxfp8_quant_rows(x, g, 1e-6, 0, block=64)
    c32, s32 = orc.mxfp8_quant_rows(x, g, 1e-6, 0, block=32)
    assert s32.shape == (T, K // 32) and (s32.reshape(T, -1, 2).max(axis=2) == s64).all()


def pin_mxfp8_power_of_two_invariance(orc):
    # eps = 0: x * 2^5 leaves y, so every code and scale, unchanged
    rng = _rng(63)
    x = _rand_bf16(rng, (6, 192))
    xs = _bf16_bits_of_f32((bf16_bits_to_f64(x) * 32).astype(np.float32))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, 192).astype(np.float32))
    for variant in (0, 1):
        a = orc.mxfp8_quant_rows(x, g, 0.0, variant)
        b = orc.mxfp8_quant_rows(xs, g, 0.0, variant)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        # and gamma * 2 moves every scale by exactly one, codes unchanged
        g2 = _bf16_bits_of_f32((bf16_bits_to_f64(g) * 2).astype(np.float32))
        c = orc.mxfp8_quant_rows(x, g2, 0.0, variant)
        assert np.array_equal(c[0], a[0]) and np.array_equal(c[1].astype(int), a[1].astype(int) + 1)


def _mx_random(rng, rows, K, sigma=1.0):
    codes = rng.integers(0, 256, (rows, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    scales = rng.integers(127 - 12, 127 + 4, (rows, K // 64)).astype(np.uint8)
    return codes, scales


def pin_mxfp8_scaled_mm_exact_small(orc):
    rng = _rng(64)
    T, K, N = 3, 128, 4
    xq, xs = _mx_random(rng, T, K)
    wq, ws = _mx_random(rng, N, K)
    ref, out = orc.mxfp8_scaled_mm(xq, xs, wq, ws, 0)
    _, out32 = orc.mxfp8_scaled_mm(xq, xs, wq, ws, 1)
    xv, wv = _torch_e4m3_decode(xq), _torch_e4m3_decode(wq)
    for t in range(T):
        for n in range(N):
            e = sum(Fraction(float(xv[t, k])) * Fraction(2) ** (int(xs[t, k // 64]) - 127) *
                    Fraction(float(wv[n, k])) * Fraction(2) ** (int(ws[n, k // 64]) - 127) for k in range(K))
            assert exact.rel_close(ref[t, n], e, 1e-13) or abs(float(e)) < 1e-300
            # the FP32 result: within half an FP32 ulp of the exact sum (plus
            # the binary64 accumulation's own error), and the bf16 output is
            # that FP32 value rounded once more
            assert abs(Fraction(float(out32[t, n])) - e) <= abs(e) * Fraction(1, 2**24) * (1 + Fraction(1, 10**9))
            bits, near = exact.bf16_round_exact(Fraction(float(out32[t, n])))
            assert near or int(out[t, n]) == bits


def pin_mxfp8_scaled_mm_torch(orc):
    import torch
    rng = _rng(65)
    T, K, N = 9, 256, 11
    xq, xs = _mx_random(rng, T, K)
    wq, ws = _mx_random(rng, N, K)
    ref, out32 = orc.mxfp8_scaled_mm(xq, xs, wq, ws, 1)
    xv = torch.from_numpy(_torch_e4m3_decode(xq)) * torch.pow(2.0, torch.from_numpy(xs.astype(np.float64) - 127)).repeat_interleave(64, 1)
    wv = torch.from_numpy(_torch_e4m3_decode(wq)) * torch.pow(2.0, torch.from_numpy(ws.astype(np.float64) - 127)).repeat_interleave(64, 1)
    want = (xv @ wv.T).numpy()
    mag = (xv.abs() @ wv.abs().T).numpy()
    assert np.all(np.abs(ref - want) <= 1e-14 * mag)
    assert np.array_equal(out32, ref.astype(np.float32))


def pin_mxfp8_scaled_mm_fp32_then_bf16(orc):
    # exact sum 1 + 2^-8 + 2^-30: its FP32 value 1 + 2^-8 is a bf16 tie, which
    # goes to 1.0 (even); rounding the binary64 sum straight to bf16 would give 1 + 2^-7.
    K = 128
    xq = np.zeros((1, K), np.uint8)
    wq = np.zeros((1, K), np.uint8)
    xq[0, 0] = xq[0, 1] = xq[0, 64] = 0x38  # 1.0
    wq[0, 0] = 0x78  # 256 * 2^-8 = 1
    wq[0, 1] = 0x38  # 1 * 2^-8
    wq[0, 64] = 0x38  # 1 * 2^-30
    xs = np.full((1, 2), 127, np.uint8)
    ws = np.array([[127 - 8, 127 - 30]], np.uint8)
    ref, out = orc.mxfp8_scaled_mm(xq, xs, wq, ws, 0)
    assert ref[0, 0] == 1 + 2.0**-8 + 2.0**-30
    assert int(out[0, 0]) == 0x3F80
    _, o32 = orc.mxfp8_scaled_mm(xq, xs, wq, ws, 1)
    assert o32[0, 0] == np.float32(1 + 2.0**-8)


def pin_mxfp8_composition(orc):
    # quantise the normed activations and a weight, then scaled_mm: close to
    # the unquantised FP32 projection (E4M3 keeps 4 significant bits)
    rng = _rng(66)
    T, K, N = 5, 256, 16
    x = _rand_bf16(rng, (T, K))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, K).astype(np.float32))
    W = rng.standard_normal((N, K)) * 0.02
    xq, xs = orc.mxfp8_quant_rows(x, g, 1e-6, 0)
    wq, ws = _mx_expected(W)
    ref, _ = orc.mxfp8_scaled_mm(xq, xs, wq, ws, 1)
    y64, _ = orc.rmsnorm_f64(x, g, 1e-6, 0)
    full = y64 @ W.T
    mag = np.abs(y64) @ np.abs(W).T
    assert np.all(np.abs(ref - full) <= 2 * 2.0**-4 * mag)
    assert np.abs(ref - full).max() < 0.1 * np.abs(full).max()


# ---------------------------------------------------------------------------
# Per-head RMSNorm after a projection (the MLA chain's norm after q_b_proj)
# ---------------------------------------------------------------------------

def pin_head_norm_constant_heads(orc):
    # every head constant (a different value per head), eps = 0: each head
    # normalises to sign(c) * gamma exactly, whatever the other heads hold
    rng = _rng(70)
    T, H, D = 3, 5, 64
    c = _bf16_bits_of_f32((rng.uniform(0.1, 50, (T, H)) * rng.choice([-1, 1], (T, H))).astype(np.float32))
    y = np.repeat(c[:, :, None], D, axis=2).reshape(T, H * D)
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    for variant in (0, 1):
        out = orc.head_rmsnorm(y, H, D, g, 0.0, variant).reshape(T, H, D)
        want = np.where(bf16_bits_to_f64(c)[:, :, None] < 0, g | np.uint16(0x8000), g)
        assert np.array_equal(out, np.broadcast_to(want, (T, H, D)))
        no_g = orc.head_rmsnorm(y, H, D, None, 0.0, variant).reshape(T, H, D)
        assert np.array_equal(no_g, np.where(bf16_bits_to_f64(c)[:, :, None] < 0, 0xBF80, 0x3F80).astype(np.uint16)
                              .repeat(D, axis=2))


def pin_head_norm_torch(orc):
    import torch
    rng = _rng(71)
    T, H, D = 6, 7, 96
    y = _rand_bf16(rng, (T, H * D), 2.0)
    y[2, 3 * D:4 * D] = _rand_bf16(rng, (D,), 1e-3)  # a quiet head beside loud ones
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    for eps in (1e-6, 0.5):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(bf16_bits_to_f64(y).reshape(T, H, D)), (D,),
                                           torch.from_numpy(bf16_bits_to_f64(g)), eps).numpy()
        for variant in (0, 1):
            out = orc.head_rmsnorm(y, H, D, g, eps, variant).reshape(T, H, D)
            for idx in np.ndindex(T, H, D):
                bits, near = exact.bf16_round_exact(Fraction(float(ref[idx])))
                assert near or int(out[idx]) == bits, (eps, variant, idx)


def pin_head_norm_scale_invariance(orc):
    # eps = 0: scaling each head by its own power of two changes nothing
    rng = _rng(72)
    T, H, D = 4, 6, 32
    y = _rand_bf16(rng, (T, H * D))
    s = np.ldexp(1.0, rng.integers(-6, 7, (T, H))).repeat(D, axis=1)
    ys = _bf16_bits_of_f32((bf16_bits_to_f64(y) * s).astype(np.float32))
    for variant in (0, 1):
        assert np.array_equal(orc.head_rmsnorm(y, H, D, None, 0.0, variant),
                              orc.head_rmsnorm(ys, H, D, None, 0.0, variant))


def pin_head_norm_exact_small(orc):
    rng = _rng(73)
    T, H, D = 2, 3, 4
    y = _rand_bf16(rng, (T, H * D))
    g = _bf16_bits_of_f32(rng.uniform(0.5, 1.5, D).astype(np.float32))
    eps = 0.25
    for variant in (0, 1):
        out = orc.head_rmsnorm(y, H, D, g, eps, variant)
        for t in range(T):
            for h in range(H):
                v = [Fraction(exact.bf16_value(int(b))) for b in y[t, h * D:(h + 1) * D]]
                r = exact.dec_sqrt_recip(sum(a * a for a in v) / D + Fraction(eps))
                for i in range(D):
                    bits, near = exact.bf16_round_exact(v[i] * r * Fraction(exact.bf16_value(int(g[i]))))
                    assert near or int(out[t, h * D + i]) == bits


ALL_PINS = [
    pin_head_norm_constant_heads,
    pin_head_norm_torch,
    pin_head_norm_scale_invariance,
    pin_head_norm_exact_small,
    pin_e4m3_codec,
    pin_e8m0_scale,
    pin_mxfp8_constructed_ties,
    pin_mxfp8_gamma_closed_form,
    pin_mxfp8_block_structure_and_bound,
    pin_mxfp8_power_of_two_invariance,
    pin_mxfp8_scaled_mm_exact_small,
    pin_mxfp8_scaled_mm_torch,
    pin_mxfp8_scaled_mm_fp32_then_bf16,
    pin_mxfp8_composition,
    pin_bf16_codec,
    pin_qmrs_unit_scales_exact,
    pin_qmrs_x2_is_k_by_n,
    pin_qmrs_power_of_two_scales,
    pin_qmrs_batch_structure,
    pin_qmrs_numpy_float32,
    pin_qmrs_overflow,
    pin_rope_angle_zero_is_head_norm,
    pin_rope_quarter_and_half_turn,
    pin_rope_positions_index_the_table,
    pin_rope_exact_small,
    pin_rope_torch,
    pin_rope_small_rows_closed_form,
    pin_rope_rejects_bad_position,
    pin_ex_reduces_to_base,
    pin_ex_residual_sum_exact,
    pin_ex_residual_composition,
    pin_ex_norm_bias_closed_form,
    pin_ex_projection_bias,
    pin_ex_exact_small,
    pin_ex_torch,
    pin_rmsnorm_variants_agree,
    pin_rmsnorm_closed_forms,
    pin_rmsnorm_scale_invariance,
    pin_rmsnorm_exact_small,
    pin_rmsnorm_torch,
    pin_linear_identity_and_permutation,
    pin_linear_exact_small,
    pin_linear_torch,
    pin_linear_form1_gamma,
    pin_mla_composition,
    pin_quant_constructed_ties,
    pin_quant_properties,
    pin_quant_sum_of_squares_reading,
    pin_gemm_s8_bruteforce,
    pin_dequant_exact,
    pin_w8a8_composition,
]
