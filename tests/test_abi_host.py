"""The C-ABI library on the host, without a GPU: it builds, loads, exports
every function include/rnl.h declares, sizes workspaces and rejects bad
arguments with the documented status codes before touching a device.

The argument checks run in a child process with CUDA_VISIBLE_DEVICES="" so
that, whatever the machine, no call can reach a GPU."""
import json
import os
import re
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rnl.h")


@pytest.fixture(scope="module")
def lib_path():
    from rmsnorm_linear_projection_gb300 import build
    return build.build()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)
    keywords = {"typedef", "enum", "struct", "sizeof", "defined"}
    prefixes = ("rnl_", "rmsnorm_linear_", "mla_", "quant_", "mxfp8_")
    return sorted({n for n in names if n not in keywords and n.startswith(prefixes)})


def test_exports_every_declared_symbol(lib_path):
    import ctypes
    lib = ctypes.CDLL(lib_path)
    declared = header_functions()
    assert "rmsnorm_linear_bf16" in declared and "rnl_workspace_size" in declared
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, missing
    from rmsnorm_linear_projection_gb300 import EXPORTS
    assert sorted(EXPORTS) == declared


CHILD = textwrap.dedent("""
    import ctypes, json, sys
    sys.path.insert(0, {root!r})
    from rmsnorm_linear_projection_gb300 import _native as nat
    lib = nat.load({lib!r})
    P = ctypes.c_void_p
    A = P(0x10000)        # a 16-byte aligned fake address: never dereferenced,
    B = P(0x10008)        # every call below fails validation first
    ws = P(0x20000)
    r = {{}}
    r["version"] = lib.rnl_version()
    r["debug_build"] = lib.rnl_debug_build()
    r["bounds_selftest_release"] = lib.rnl_selftest_bounds_check(None)
    r["ws_bf16_qkv"] = lib.rnl_workspace_size(0, 4096, 4096, 6144, 0)
    r["ws_bf16_skinny"] = lib.rnl_workspace_size(0, 16384, 28672, 24, 1)
    r["ws_w8a8"] = lib.rnl_workspace_size(1, 8192, 4096, 4096, 0)
    r["ws_mla"] = lib.rnl_workspace_size(2, 2048, 7168, 1536, 24576)
    r["ws_bad_op"] = lib.rnl_workspace_size(9, 1, 8, 8, 0)
    r["ws_neg"] = lib.rnl_workspace_size(0, -1, 8, 8, 0)
    big = 1 << 40
    f = lib.rmsnorm_linear_bf16
    r["bf16_null_x"] = f(None, None, A, 4, 64, 8, 1e-6, 0, A, 0, ws, 1 << 20, None)
    r["bf16_null_out"] = f(A, None, A, 4, 64, 8, 1e-6, 0, None, 0, ws, 1 << 20, None)
    r["bf16_neg_T"] = f(A, None, A, -1, 64, 8, 1e-6, 0, A, 0, ws, 1 << 20, None)
    r["bf16_zero_K"] = f(A, None, A, 4, 0, 8, 1e-6, 0, A, 0, ws, 1 << 20, None)
    r["bf16_huge_N"] = f(A, None, A, 4, 64, big, 1e-6, 0, A, 0, ws, 1 << 20, None)
    r["bf16_K_not_mult8"] = f(A, None, A, 4, 60, 8, 1e-6, 0, A, 0, ws, 1 << 20, None)
    r["bf16_misaligned_x"] = f(B, None, A, 4, 64, 8, 1e-6, 0, A, 0, ws, 1 << 20, None)
    r["bf16_bad_mode"] = f(A, None, A, 4, 64, 8, 1e-6, 7, A, 0, ws, 1 << 20, None)
    r["bf16_bad_eps"] = f(A, None, A, 4, 64, 8, float("nan"), 0, A, 0, ws, 1 << 20, None)
    r["bf16_neg_eps"] = f(A, None, A, 4, 64, 8, -1.0, 0, A, 0, ws, 1 << 20, None)
    r["bf16_bad_dtype"] = f(A, None, A, 4, 64, 8, 1e-6, 0, A, 5, ws, 1 << 20, None)
    r["bf16_fp32_gamma"] = f(A, A, A, 4, 64, 8, 1e-6, 0, A, 1, ws, 1 << 20, None)
    r["bf16_small_ws"] = f(A, None, A, 4, 64, 8, 1e-6, 0, A, 0, ws, 16, None)
    r["bf16_null_ws"] = f(A, None, A, 4, 64, 8, 1e-6, 0, A, 0, None, 0, None)
    r["bf16_T0"] = f(None, None, None, 0, 64, 8, 1e-6, 0, None, 0, None, 0, None)
    r["bf16_no_device"] = f(A, None, A, 4, 64, 8, 1e-6, 0, A, 0, ws, 1 << 30, None)
    g = lib.rmsnorm_linear_w8a8
    r["w8a8_null_scale"] = g(A, None, A, None, 4, 64, 8, 1e-6, 0, A, None, None, ws, 1 << 20, None)
    r["w8a8_K_not_mult16"] = g(A, None, A, A, 4, 72, 8, 1e-6, 0, A, None, None, ws, 1 << 20, None)
    r["w8a8_small_ws"] = g(A, None, A, A, 4, 64, 8, 1e-6, 0, A, None, None, ws, 64, None)
    m = lib.mla_q_chain
    r["mla_null_gamma"] = m(A, A, None, A, 4, 64, 16, 8, 1e-6, 1, A, None, ws, 1 << 20, None)
    r["mla_N1_not_mult8"] = m(A, A, A, A, 4, 64, 12, 8, 1e-6, 1, A, None, ws, 1 << 20, None)
    s8 = lib.rnl_gemm_s8s8s32
    r["s8_K_not_mult16"] = s8(A, A, A, 4, 8, 24, ws, 1 << 20, None)
    r["s8_M0"] = s8(None, None, None, 0, 8, 32, None, 0, None)
    e = lib.rmsnorm_linear_bf16_ex
    C = P(0x30000)
    r["ex_sum_without_residual"] = e(A, None, C, None, None, A, None, 4, 64, 8, 1e-6, 0, A, None, ws, 1 << 20, None)
    r["ex_sum_partial_overlap"] = e(A, C, P(0x10010), None, None, A, None, 4, 64, 8, 1e-6, 0, A, None, ws, 1 << 20, None)
    r["ex_misaligned_bias"] = e(A, None, None, None, None, A, B, 4, 64, 8, 1e-6, 0, A, None, ws, 1 << 20, None)
    r["ex_misaligned_rstd"] = e(A, None, None, None, None, A, None, 4, 64, 8, 1e-6, 0, A, P(0x10002), ws, 1 << 20, None)
    r["ex_null_W"] = e(A, None, None, None, None, None, None, 4, 64, 8, 1e-6, 0, A, None, ws, 1 << 20, None)
    r["ex_bad_mode"] = e(A, None, None, None, None, A, None, 4, 64, 8, 1e-6, 3, A, None, ws, 1 << 20, None)
    r["ex_small_ws"] = e(A, None, None, None, None, A, None, 4, 64, 8, 1e-6, 0, A, None, ws, 16, None)
    r["ex_in_place_no_device"] = e(A, C, C, A, A, A, A, 4, 64, 8, 1e-6, 0, A, P(0x40000), ws, 1 << 30, None)
    qm = lib.quant_matmul_reduce_sum
    r["qmrs_N_not_mult16"] = qm(A, A, A, A, 2, 4, 32, 24, A, ws, 1 << 30, None)
    r["qmrs_B0"] = qm(A, A, A, A, 0, 4, 32, 32, A, ws, 1 << 30, None)
    r["qmrs_M0"] = qm(None, None, None, None, 2, 0, 32, 32, None, None, 0, None)
    r["qmrs_null_scale"] = qm(A, A, None, A, 2, 4, 32, 32, A, ws, 1 << 30, None)
    r["qmrs_small_ws"] = qm(A, A, A, A, 2, 4, 32, 32, A, ws, 64, None)
    r["qmrs_no_device"] = qm(A, A, A, A, 2, 4, 32, 32, A, ws, 1 << 30, None)
    r["ws_qmrs"] = lib.rnl_workspace_size(5, 2048, 4096, 4096, 4)
    r["ws_qmrs_b1"] = lib.rnl_workspace_size(5, 2048, 4096, 4096, 1)
    mx = lib.rmsnorm_linear_mxfp8
    #     x, gamma, w_codes, w_scale, T, K, N, eps, mode, block, out, out_dtype, codes, scales, ws, bytes, stream
    r["mx_bad_block"] = mx(A, None, A, A, 4, 128, 8, 1e-6, 0, 48, A, 0, None, None, ws, 1 << 30, None)
    r["mx_K_not_mult_block"] = mx(A, None, A, A, 4, 96, 8, 1e-6, 0, 64, A, 0, None, None, ws, 1 << 30, None)
    r["mx_bad_dtype"] = mx(A, None, A, A, 4, 128, 8, 1e-6, 0, 64, A, 2, None, None, ws, 1 << 30, None)
    r["mx_null_scale"] = mx(A, None, A, None, 4, 128, 8, 1e-6, 0, 64, A, 0, None, None, ws, 1 << 30, None)
    r["mx_misaligned_codes_out"] = mx(A, None, A, A, 4, 128, 8, 1e-6, 0, 64, A, 0, B, None, ws, 1 << 30, None)
    r["mx_small_ws"] = mx(A, None, A, A, 4, 128, 8, 1e-6, 0, 64, A, 0, None, None, ws, 64, None)
    r["mx_T0"] = mx(None, None, None, None, 0, 128, 8, 1e-6, 0, 64, None, 0, None, None, None, 0, None)
    r["mx_no_device"] = mx(A, A, A, A, 4, 128, 8, 1e-6, 0, 32, A, 1, A, A, ws, 1 << 30, None)
    r["mx_too_large"] = mx(A, None, A, A, 4, 1 << 20, 1 << 17, 1e-6, 0, 64, A, 0, None, None, ws, 1 << 30, None)
    hn = lib.rnl_head_rmsnorm
    r["hn_bad_dim"] = hn(A, 4, 8, 96, None, 1e-6, 1, A, None)
    r["hn_partial_overlap"] = hn(A, 4, 8, 128, None, 1e-6, 1, P(0x10010), None)
    r["hn_null_y"] = hn(None, 4, 8, 128, None, 1e-6, 1, A, None)
    r["hn_T0"] = hn(None, 0, 8, 128, None, 1e-6, 1, None, None)
    r["hn_in_place_no_device"] = hn(A, 4, 8, 192, None, 1e-6, 1, A, None)
    r["hn_bad_eps"] = hn(A, 4, 8, 128, None, -1.0, 1, A, None)
    mh = lib.mla_q_chain_head_norm
    r["mlahn_N2_not_mult"] = mh(A, A, A, A, 4, 64, 32, 1000, 1e-6, 1, 192, None, 1e-6, A, None, ws, 1 << 30, None)
    r["mlahn_bad_dim"] = mh(A, A, A, A, 4, 64, 32, 960, 1e-6, 1, 96, None, 1e-6, A, None, ws, 1 << 30, None)
    sm = lib.mxfp8_scaled_mm
    r["mxmm_null_x_scale"] = sm(A, None, A, A, 4, 128, 8, 64, A, 0, ws, 1 << 30, None)
    r["mxmm_bad_block"] = sm(A, A, A, A, 4, 128, 8, 16, A, 0, ws, 1 << 30, None)
    r["mxmm_no_device"] = sm(A, A, A, A, 4, 128, 8, 64, A, 1, ws, 1 << 30, None)
    r["ws_mxfp8"] = lib.rnl_workspace_size(6, 4096, 4096, 6144, 0)
    pp = ctypes.c_void_p(None)
    r["pipe_null_out"] = lib.rnl_pipeline_create(0, 4, 64, 8, 0, None)
    r["pipe_bad_op"] = lib.rnl_pipeline_create(3, 4, 64, 8, 0, ctypes.byref(pp))
    r["pipe_zero_K"] = lib.rnl_pipeline_create(0, 4, 0, 8, 0, ctypes.byref(pp))
    r["pipe_bad_dtype"] = lib.rnl_pipeline_create(0, 4, 64, 8, 7, ctypes.byref(pp))
    r["pipe_no_device"] = lib.rnl_pipeline_create(0, 4, 64, 8, 0, ctypes.byref(pp))
    r["pipe_handle_after_fail"] = pp.value
    tk = ctypes.c_int64(-1)
    r["pipe_submit_null"] = lib.rnl_pipeline_submit_bf16(None, A, None, A, 1e-6, 0, A, ctypes.byref(tk))
    r["pipe_submit_null_W"] = lib.rnl_pipeline_submit_bf16(None, A, None, None, 1e-6, 0, A, ctypes.byref(tk))
    r["pipe_submit_bad_eps"] = lib.rnl_pipeline_submit_w8a8(None, A, None, A, A, -1.0, 0, A, ctypes.byref(tk))
    r["pipe_submit_mla_bad_mode"] = lib.rnl_pipeline_submit_mla(None, A, A, A, A, 1e-6, 5, A, ctypes.byref(tk))
    r["pipe_wait_null"] = lib.rnl_pipeline_wait(None, 0, None)
    r["pipe_destroy_null"] = lib.rnl_pipeline_destroy(None)
    r["status_strings"] = [lib.rnl_status_string(i).decode() for i in range(11)]
    r["trace_enable"] = lib.rnl_trace_enable(1)
    r["trace_read_empty"] = lib.rnl_trace_read(None, (ctypes.c_float * 4)(), 4)
    lib.rnl_trace_enable(0)
    print(json.dumps(r))
""")


@pytest.fixture(scope="module")
def host_results(lib_path):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    code = CHILD.format(root=ROOT, lib=lib_path)
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=300)
    assert p.returncode == 0, p.stderr
    return json.loads(p.stdout.strip().splitlines()[-1])


OK, NULL, SHAPE, ALIGN, ARG, WORKSPACE, LAUNCH, TIMEOUT, UNSUP, DEVICE = range(10)


def test_workspace_sizes(host_results):
    r = host_results
    assert r["version"] >= 100
    part = 128 * 2 * 128 * 256 * 4  # GEMM K-split partial sums
    assert r["ws_bf16_qkv"] == 4096 * 4 + 4096 * 4096 * 2 + part  # rstd + A + partials
    # codes + widened weight + x_scale + max |gamma| (one 256-byte unit) + partials
    # + the pair GEMM's running int32 sums of chunked tiles (as large as the partials)
    assert r["ws_w8a8"] == 8192 * 4096 * 2 + 4096 * 4096 * 2 + 8192 * 4 + 256 + 2 * part
    assert r["ws_mla"] == 2 * 2048 * 1536 * 2 + 2048 * 4 + part
    # skinny partial records: (T/128 + 512) records of 128 rows x (32 + 1) floats
    assert r["ws_bf16_skinny"] == (16384 // 128 + 512) * 128 * 33 * 4
    # QuantMatMulReduceSum: widened x1 and x2, fp32 x2_scale, fp32 batch sum
    # + the flags of the one-launch batch sum: (2048/128) x (4096/128) tiles x 8 warps x 8 bytes
    assert r["ws_qmrs"] == (4 * 2048 * 4096 * 2 + 4 * 4096 * 4096 * 2 + 4096 * 4 + 2048 * 4096 * 4
                            + 16 * 32 * 64)
    assert r["ws_qmrs_b1"] == 2048 * 4096 * 2 + 4096 * 4096 * 2 + 4096 * 4  # no running sum
    # MXFP8: dequantised bf16 activations and weight, GEMM partials
    # codes + scale atoms of x (32 row blocks x 32 k-blocks) and W (32 tiles of 192 rows x 32 x 2)
    # for the block-scaled GEMM, then the dequantised operands of the emulation path
    assert r["ws_mxfp8"] == (4096 * 4096 + 32 * 32 * 512 + 32 * 32 * 2 * 512 + 4096 * 4096 * 2 +
                             6144 * 4096 * 2 + part)
    max_size = (1 << 64) - 1
    assert r["ws_bad_op"] == max_size and r["ws_neg"] == max_size


@pytest.mark.parametrize("key,want", [
    ("bf16_null_x", NULL), ("bf16_null_out", NULL), ("bf16_neg_T", SHAPE),
    ("bf16_zero_K", SHAPE), ("bf16_huge_N", SHAPE), ("bf16_K_not_mult8", ALIGN),
    ("bf16_misaligned_x", ALIGN), ("bf16_bad_mode", ARG), ("bf16_bad_eps", ARG),
    ("bf16_neg_eps", ARG), ("bf16_bad_dtype", ARG), ("bf16_fp32_gamma", UNSUP),
    ("bf16_small_ws", WORKSPACE), ("bf16_null_ws", WORKSPACE), ("bf16_T0", OK),
    ("bf16_no_device", DEVICE),
    ("w8a8_null_scale", NULL), ("w8a8_K_not_mult16", ALIGN), ("w8a8_small_ws", WORKSPACE),
    ("mla_null_gamma", NULL), ("mla_N1_not_mult8", ALIGN),
    ("s8_K_not_mult16", ALIGN), ("s8_M0", OK),
    ("trace_enable", OK), ("trace_read_empty", 0),
    ("debug_build", 0), ("bounds_selftest_release", UNSUP),
    ("ex_sum_without_residual", ARG), ("ex_sum_partial_overlap", ARG), ("ex_misaligned_bias", ALIGN),
    ("ex_misaligned_rstd", ALIGN), ("ex_null_W", NULL), ("ex_bad_mode", ARG), ("ex_small_ws", WORKSPACE),
    ("ex_in_place_no_device", DEVICE),
    ("qmrs_N_not_mult16", ALIGN), ("qmrs_B0", SHAPE), ("qmrs_M0", OK), ("qmrs_null_scale", NULL),
    ("qmrs_small_ws", WORKSPACE), ("qmrs_no_device", DEVICE),
    ("mx_bad_block", ARG), ("mx_K_not_mult_block", SHAPE), ("mx_bad_dtype", ARG), ("mx_null_scale", NULL),
    ("mx_misaligned_codes_out", ALIGN), ("mx_small_ws", WORKSPACE), ("mx_T0", OK), ("mx_too_large", SHAPE), ("mx_no_device", DEVICE),
    ("hn_bad_dim", UNSUP), ("hn_partial_overlap", ARG), ("hn_null_y", NULL), ("hn_T0", OK),
    ("hn_in_place_no_device", DEVICE), ("hn_bad_eps", ARG), ("mlahn_N2_not_mult", SHAPE), ("mlahn_bad_dim", UNSUP),
    ("mxmm_null_x_scale", NULL), ("mxmm_bad_block", ARG), ("mxmm_no_device", DEVICE),
    ("pipe_null_out", NULL), ("pipe_bad_op", ARG), ("pipe_zero_K", SHAPE),
    ("pipe_bad_dtype", ARG), ("pipe_no_device", DEVICE), ("pipe_handle_after_fail", None),
    ("pipe_submit_null", NULL), ("pipe_submit_null_W", NULL), ("pipe_submit_bad_eps", ARG),
    ("pipe_submit_mla_bad_mode", ARG), ("pipe_wait_null", NULL), ("pipe_destroy_null", OK),
])
def test_argument_checks(host_results, key, want):
    assert host_results[key] == want


def test_status_strings(host_results):
    s = host_results["status_strings"]
    assert s[0] == "ok" and len(set(s)) == 11


def test_binding_status_checks_are_well_formed():
    """Every status check in the binding names its call (static scan, no GPU)."""
    import ast
    src = open(os.path.join(ROOT, "rmsnorm_linear_projection_gb300", "_native.py")).read()
    calls = [n for n in ast.walk(ast.parse(src))
             if isinstance(n, ast.Call) and getattr(n.func, "id", None) == "_check"]
    assert len(calls) >= 15
    bad = [n.lineno for n in calls if len(n.args) != 2 or isinstance(n.args[1], ast.Tuple)]
    assert not bad, f"_check calls with the wrong arguments at lines {bad}"
