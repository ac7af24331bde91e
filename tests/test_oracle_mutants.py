"""Planted mistakes: each test copies oracle.c, plants one plausible mistake
(a dropped term, a wrong sign, index or rounding rule, a transposed operand),
compiles the copy on the CPU into a temporary directory and runs every pin on
it in a child process.  At least one pin must fail (or the child must crash),
which shows that the pins would catch that mistake in the real oracle.
"""
import json
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, replacement).  Each text must occur exactly once.
MUTANTS = [
    ("drop_eps_rsqrt_form", "return 1.0 / sqrt(ms + eps);", "return 1.0 / sqrt(ms);"),
    ("drop_inv_d_sqrt_div_form", "s += (v * v) * inv_d;", "s += (v * v);"),
    ("mean_over_k_minus_1", "double inv_d = 1.0 / (double)K;", "double inv_d = 1.0 / (double)(K - 1);"),
    ("drop_gamma_at10", "                if (gamma)\n                    v = v * orc_bf16_value(gamma[k]);\n                a[k]",
     "                a[k]"),
    ("drop_bf16_cast_of_normed", "a[k] = (form == 0) ? orc_bf16_value(orc_bf16_rne(v)) : v;", "a[k] = v;"),
    ("transposed_weight", "const double *wr = wd + n * K;\n                double acc = 0.0;\n                for (int64_t k = 0; k < K; ++k)\n                    acc += a[k] * wr[k];\n                if (ref)",
     "const double *wr = wd + n;\n                double acc = 0.0;\n                for (int64_t k = 0; k < K; ++k)\n                    acc += a[k] * wr[(k % N) * K + (k / N) % K];\n                if (ref)"),
    ("wrong_sign_accumulate", "acc += a[k] * wr[k];\n                if (ref)", "acc -= a[k] * wr[k];\n                if (ref)"),
    ("mla_drop_gamma", "v = v * orc_bf16_value(gamma_cq[j]);", "v = v * 1.0;"),
    ("mla_stage2_unrounded_input", "z[j] = orc_bf16_value(orc_bf16_rne(v));", "z[j] = v;"),
    ("quant_round_half_away", "float r = rintf(v);", "float r = roundf(v);"),
    ("quant_scale_128", "float qs = 127.0f / amax;", "float qs = 128.0f / amax;"),
    ("quant_dequant_scale_inverted", "x_scale[t] = amax / 127.0f;", "x_scale[t] = 127.0f / amax;"),
    ("quant_drop_gamma", "            if (gamma)\n                y = y * bf16_as_float(gamma[k]);\n            float v = y * qs;",
     "            float v = y * qs;"),
    # the FP32 sum of squares taken as a left-to-right binary32 sum instead of
    # the rounding of the exact sum (both front ends, both norm variants)
    ("quant_sum_sequential_f32", "\n                s64 += (double)sq;",
     "\n                s64 = (double)((float)s64 + sq);"),
    ("quant_sum_sequential_f32_sqrt_div", "\n                s64 += (double)sc;",
     "\n                s64 = (double)((float)s64 + sc);"),
    ("mx_sum_sequential_f32", "\n                    s64 += (double)sq;",
     "\n                    s64 = (double)((float)s64 + sq);"),
    ("mx_sum_sequential_f32_sqrt_div", "\n                    s64 += (double)sc;",
     "\n                    s64 = (double)((float)s64 + sc);"),
    ("gemm_s8_off_by_one", "for (int64_t k = 0; k < K; ++k)\n                acc += (int64_t)A[m * K + k]",
     "for (int64_t k = 1; k < K; ++k)\n                acc += (int64_t)A[m * K + k]"),
    ("dequant_wrong_scale", "double scale = (double)x_scale[m] * (double)w_scale[n];",
     "double scale = (double)x_scale[m] * (double)w_scale[m % N];"),
    ("bf16_ties_away", "double r = nearbyint(m * 256.0);", "double r = round(m * 256.0);"),
    ("bf16_truncate", "double r = nearbyint(m * 256.0);", "double r = floor(m * 256.0);"),
    # AT-10 with residual add, norm bias, output_rstd and projection bias
    ("ex_drop_residual", "xa[k] = orc_bf16_rne(orc_bf16_value(xr[k]) +\n                                         orc_bf16_value(residual[t * K + k]));",
     "xa[k] = xr[k];"),
    ("ex_residual_subtracted", "orc_bf16_value(xr[k]) +\n                                         orc_bf16_value(residual",
     "orc_bf16_value(xr[k]) -\n                                         orc_bf16_value(residual"),
    ("ex_rstd_of_x_not_x_add", "double r = row_rstd_f64(xa, K, eps, variant);",
     "double r = row_rstd_f64(xr, K, eps, variant);"),
    ("ex_norm_bias_before_gamma",
     "                if (gamma)\n                    v = v * orc_bf16_value(gamma[k]);\n                if (beta)\n                    v = v + orc_bf16_value(beta[k]);",
     "                if (beta)\n                    v = v + orc_bf16_value(beta[k]);\n                if (gamma)\n                    v = v * orc_bf16_value(gamma[k]);"),
    ("ex_drop_norm_bias", "                if (beta)\n                    v = v + orc_bf16_value(beta[k]);", ""),
    ("ex_projection_bias_after_rounding", "acc = acc + orc_bf16_value(bias[n]);",
     "acc = orc_bf16_value(orc_bf16_rne(acc)) + orc_bf16_value(bias[n]);"),
    ("ex_drop_projection_bias", "acc = acc + orc_bf16_value(bias[n]);", "acc = acc;"),
    # QKV split + per-head RMSNorm + RoPE
    ("rope_sign_of_sine", "dst[i] = orc_bf16_rne(z0 * ci - z1 * si);", "dst[i] = orc_bf16_rne(z0 * ci + z1 * si);"),
    ("rope_cos_sin_swapped", "const float *c = cs + (int64_t)pos[t] * D;\n        const float *s = c + half;",
     "const float *s = cs + (int64_t)pos[t] * D;\n        const float *c = s + half;"),
    ("rope_k_heads_use_q_gamma", "                g = k_gamma;", "                g = q_gamma;"),
    ("rope_unrounded_norm", "double z0 = orc_bf16_value(orc_bf16_rne(orc_bf16_value(yh[i]) * r *\n                                                        orc_bf16_value(g[i])));",
     "double z0 = orc_bf16_value(yh[i]) * r * orc_bf16_value(g[i]);"),
    ("rope_adjacent_pairing", "double z1 = orc_bf16_value(orc_bf16_rne(orc_bf16_value(yh[i + half]) * r *",
     "double z1 = orc_bf16_value(orc_bf16_rne(orc_bf16_value(yh[(i + 1) % D]) * r *"),
    ("rope_head_norm_drops_eps", "double r = 1.0 / sqrt(ss / (double)D + eps);", "double r = 1.0 / sqrt(ss / (double)D);"),
    # QuantMatMulReduceSum
    ("qmrs_x2_transposed", "const int8_t *bc = x2 + b * K * N + n;\n                for (int64_t k = 0; k < K; ++k)\n                    acc += (int64_t)ar[k] * (int64_t)bc[k * N];",
     "const int8_t *bc = x2 + b * K * N + n * K;\n                for (int64_t k = 0; k < K; ++k)\n                    acc += (int64_t)ar[k] * (int64_t)bc[k % N];"),
    ("qmrs_scale_of_batch_0", "const float sc = x1_scale[b * M + m] * ws;", "const float sc = x1_scale[m] * ws;"),
    ("qmrs_scale_product_in_double", "const float scaled = mm * sc;", "const float scaled = (float)((double)mm * ((double)x1_scale[b * M + m] * (double)ws));"),
    ("qmrs_batch_sum_reversed", "            for (int64_t b = 0; b < B; ++b) {\n                int64_t acc = 0;",
     "            for (int64_t bb = 0; bb < B; ++bb) {\n                const int64_t b = B - 1 - bb;\n                int64_t acc = 0;"),
    ("qmrs_drop_x2_scale", "const float ws = bf16_as_float(x2_scale[n]);", "const float ws = 1.0f;"),
    # MXFP8: E4M3 codec, shared block exponent, scaled_mm
    ("e4m3_decode_wrong_bias", "ldexp(8.0 + m, e - 10)", "ldexp(8.0 + m, e - 11)"),
    ("e4m3_ties_away", "double r = nearbyint(ldexp(a, 3 - k));", "double r = round(ldexp(a, 3 - k));"),
    ("e4m3_overflow_to_nan", "return sign | 0x7E; /* 448 */", "return sign | 0x7F; /* 448 */"),
    ("e4m3_subnormal_threshold", "if (a < ldexp(1.0, -6)) { /* subnormal range", "if (a < ldexp(1.0, -7)) { /* subnormal range"),
    ("mx_exponent_off_by_one", "X = E - 1 - 8;", "X = E - 8;"),
    ("mx_amax_over_whole_row", "for (int64_t k = b0; k < b0 + block; ++k)\n                    if (fabsf(y[k]) > amax)",
     "for (int64_t k = 0; k < K; ++k)\n                    if (fabsf(y[k]) > amax)"),
    ("mx_drop_gamma", "                if (gamma)\n                    v = v * bf16_as_float(gamma[k]);\n                y[k] = v;",
     "                y[k] = v;"),
    ("mx_scaled_mm_first_weight_scale", "orc_e8m0_value(ws[n * nb + k / block])", "orc_e8m0_value(ws[n * nb])"),
    ("mx_scaled_mm_bf16_from_binary64", "((uint16_t *)out)[t * N + n] = orc_bf16_rne((double)f);",
     "((uint16_t *)out)[t * N + n] = orc_bf16_rne(acc);"),
    ("mx_scale_byte_bias", "scales[t * (K / block) + b0 / block] = (uint8_t)(X + 127);",
     "scales[t * (K / block) + b0 / block] = (uint8_t)(X + 128);"),
    # per-head RMSNorm
    ("head_norm_over_whole_row", "const double r = row_rstd_f64(yh, D, eps, variant);",
     "const double r = row_rstd_f64(y + t * H * D, H * D, eps, variant);"),
    ("head_norm_drops_eps", "const double r = row_rstd_f64(yh, D, eps, variant);",
     "const double r = row_rstd_f64(yh, D, 0.0, variant);"),
    ("head_norm_drops_gamma", "                if (gamma)\n                    v = v * orc_bf16_value(gamma[i]);\n                oh[i]",
     "                oh[i]"),
    ("head_norm_head_stride", "const uint16_t *yh = y + (t * H + h) * D;", "const uint16_t *yh = y + (t * H + h % 2) * D;"),
    ("rope_split_off_by_one_head", "            if (h < Hq) {\n                dst = q + (t * Hq + h) * D;",
     "            if (h <= Hq && h < Hq + Hkv) {\n                dst = q + (t * Hq + (h < Hq ? h : 0)) * D;"),
]

CHILD = textwrap.dedent("""
    import json, sys
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import oracle, oracle_pins
    o = oracle.Oracle(oracle.load({so!r}))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except Exception as e:  # AssertionError or a numpy error from garbage
            failed.append(pin.__name__)
    print(json.dumps(failed))
""")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    so = str(tmp_path / "liboracle_mutant.so")
    import oracle
    subprocess.run(["gcc", *oracle.CFLAGS, str(mutant), "-o", so, "-lm"], check=True)
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), so=so)
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, env=env)
    if r.returncode != 0:
        return  # the mutant crashed the child: caught
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"planted mistake {name} passed every pin"
