"""Fused RMSNorm -> Linear projection for one GB300 (sm_103a).

Python binding of the C library ``librnl.so`` (header ``include/rnl.h``).
The functions carry the names of the C entry points and only marshal
arguments; the computation runs in the library's CUDA kernels.

    rmsnorm_linear_bf16   AT-10 RMSNorm + Linear (bf16 out) / mhc_pre FP32 form
    rmsnorm_linear_bf16_ex  the same with residual add, norm bias, output_rstd and
                          projection bias
    rmsnorm_linear_w8a8   AT-11 RMSNorm + INT8 quant + exact INT8 matmul + dequant
    rnl_w8a8_prepare_weight / rmsnorm_linear_w8a8_prepared
                          the same with the weight widened once
    mla_q_chain           MLA q_a projection -> RMSNorm * gamma_cq -> q_b projection
    mla_q_chain_head_norm / rnl_head_rmsnorm
                          the same chain with the per-head RMSNorm after q_b, and that norm alone
    rnl_gemm_s8s8s32      the exact INT8 matmul on its own
    quant_matmul_reduce_sum  QuantMatMulReduceSum: batched exact INT8 matmul, FP32
                          dequant and sum over the batch
    rmsnorm_linear_mxfp8  AT-11 in MXFP8 mode: RMSNorm + MX quant + scaled_mm
    mxfp8_scaled_mm       scaled_mm on MXFP8 operands
    rnl_qkv_rope / rmsnorm_linear_qkv_rope
                          QKV split + per-head RMSNorm + RoPE after the qkv projection
    rnl_pipeline_*        host-buffer pipeline: calls fed from and answering into
                          pinned host memory, copies overlapped with the kernels
    debug_library()       route calls through librnl_debug.so, the build whose
                          kernels check their indices on the device
"""
from ._native import (  # noqa: F401
    EXPORTS,
    NORM_RSQRT,
    NORM_SQRT_DIV,
    OP_BF16,
    OP_GEMM_S8,
    OP_MLA,
    OP_MXFP8,
    OP_QKV_ROPE,
    OP_QMRS,
    OP_W8A8,
    OP_W8A8_PREPARED,
    OUT_BF16,
    OUT_FP32,
    PipelineHandle,
    RnlError,
    debug_library,
    load,
    mla_q_chain,
    mla_q_chain_head_norm,
    mxfp8_scaled_mm,
    quant_matmul_reduce_sum,
    rmsnorm_linear_bf16,
    rmsnorm_linear_bf16_ex,
    rmsnorm_linear_mxfp8,
    rmsnorm_linear_qkv_rope,
    rmsnorm_linear_skinny_noalloc,
    rmsnorm_linear_w8a8,
    rmsnorm_linear_w8a8_prepared,
    rnl_check_device_error,
    rnl_debug_build,
    rnl_gemm_s8s8s32,
    rnl_head_rmsnorm,
    rnl_pipeline_create,
    rnl_pipeline_destroy,
    rnl_pipeline_submit_bf16,
    rnl_pipeline_submit_mla,
    rnl_pipeline_submit_w8a8,
    rnl_pipeline_wait,
    rnl_qkv_rope,
    rnl_selftest_bounds_check,
    rnl_selftest_wait_timeout,
    rnl_trace_enable,
    rnl_trace_read,
    rnl_w8a8_prepare_weight,
    workspace_size,
)
