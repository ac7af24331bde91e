"""The bound behind the integer GEMM's unchunked tiles, checked on the CPU.

For codes of RMSNorm-quantised rows (q = rint(y * 127 / amax), y = (x * rstd)
* gamma, x_scale = amax / 127) the kernels take

    sum_k |q_k| <= K * max|gamma| / x_scale + K / 2

(|q_k| <= |y_k| 127 / amax + 1/2, |y_k| <= |x_k| rstd max|gamma|, Cauchy-Schwarz
sum |x_k| <= sqrt(K sum x_k^2), and rstd^2 sum x_k^2 <= K), and run a row in
one FP32 accumulator when x_scale > K max|gamma| 1.005 / (2^24/128 - K/2 - 1):
then every partial sum of a row of codes times an int8 weight row stays below
128 sum |q| < 2^24, an exact binary32 integer.

The codes and x_scale come from the oracle's quantiser (the GPU's are the same
bits); the rows are chosen to press on each step of the bound: equal values
(where it is tight), one large value, sparse rows, outliers, gamma at its
maximum where x is large, both norm forms, tiny and huge magnitudes.
"""
import numpy as np
import pytest

L1_LIMIT = 131072.0  # 2^24 / 128


def floor_xs(K, gmax):
    """The kernels' threshold (exact_row_floor), in binary32 like them."""
    K32, g32 = np.float32(K), np.float32(gmax)
    return np.float32(np.float32(np.float32(K32 * g32) * np.float32(1.005)) /
                      np.float32(np.float32(L1_LIMIT) - np.float32(0.5) * K32 - np.float32(1.0)))


def to_bf16(a):
    a = np.asarray(a, np.float32)
    b = a.view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def rows_for(K, rng):
    out = []
    out.append(np.ones((3, K), np.float32) * np.float32([[1.0], [-3.5], [1e-3]]))      # equal values
    x = rng.standard_normal((4, K)).astype(np.float32)
    out.append(x)                                                                           # gaussian
    y = x.copy()
    y[:, rng.integers(0, K, (4,))] *= 40.0                                                 # outliers
    out.append(y)
    s = np.zeros((3, K), np.float32)
    s[0, 0] = 5.0
    s[1, : max(1, K // 7)] = -2.0
    s[2, ::3] = rng.uniform(-1, 1, s[2, ::3].shape)                                        # sparse
    out.append(s)
    out.append(rng.uniform(-1, 1, (3, K)).astype(np.float32) * np.float32([[1e-30], [1.0], [1e30]]))
    return np.concatenate(out)


@pytest.mark.parametrize("K", [16, 1008, 1024, 4096])
@pytest.mark.parametrize("gamma_kind", ["none", "uniform", "peaked"])
@pytest.mark.parametrize("variant", [0, 1])
def test_sum_abs_codes_bound_and_floor(orc, K, gamma_kind, variant):
    rng = np.random.default_rng(K * 7 + variant + len(gamma_kind))
    x = to_bf16(rows_for(K, rng))
    if gamma_kind == "none":
        gamma, gmax = None, 1.0
    elif gamma_kind == "uniform":
        g = rng.uniform(0.5, 1.5, K).astype(np.float32)
        gamma = to_bf16(g)
        gmax = float(np.abs((gamma.astype(np.uint32) << 16).view(np.float32)).max())
    else:  # gamma largest exactly where some rows are large
        g = np.full(K, 0.25, np.float32)
        g[: max(1, K // 7)] = 2.0
        gamma = to_bf16(g)
        gmax = 2.0
    q, xs, _, _ = orc.quant_rows_f32(x, gamma, 1e-6, variant)
    l1 = np.abs(q.astype(np.int64)).sum(1).astype(np.float64)
    fl = floor_xs(K, gmax)
    for t in range(x.shape[0]):
        if xs[t] == 0:
            assert l1[t] == 0
            continue
        bound = K * gmax / float(xs[t]) + K / 2
        # the bound itself, with room only for the roundings it was derived up to
        assert l1[t] <= bound * (1 + 1e-5) + 1, f"row {t}: sum |q| {l1[t]} above {bound}"
        if xs[t] > fl:  # the kernels' test: such a row may go unchunked
            assert 128 * l1[t] < 2 ** 24, f"row {t}: unchunked with sum |q| {l1[t]}"


def test_floor_separates_the_tight_case(orc):
    """Equal values are the bound's tight case: sum |q| = 127 K.  At K = 1008
    that is 128016 (inside the limit) and the floor lets the row through; at
    K = 1040 it is 132080 (outside) and the floor stops it."""
    for K, inside in ((1008, True), (1040, False)):
        x = to_bf16(np.ones((1, K), np.float32))
        q, xs, _, _ = orc.quant_rows_f32(x, None, 1e-6, 0)
        assert np.abs(q.astype(np.int64)).sum() == 127 * K
        assert bool(xs[0] > floor_xs(K, 1.0)) is inside
