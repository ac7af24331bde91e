/*
 * rnl.h -- C ABI of librnl: the fused RMSNorm -> Linear projection on one
 * NVIDIA GB300 (sm_103a).
 *
 * What is computed (sources are the web pages this method is described on):
 *
 *   AT-03 RMSNorm, per token row x[t, 0..K):
 *       "PyPTO-Gym operator design pattern AT-10: RMSNorm + Linear fusion"
 *       page, sec. 3 "V stage: the two RMSNorm variants".  FP32 throughout:
 *       ms = mean of x^2; rsqrt form:  rstd = rsqrt(ms + eps);
 *                         sqrt+div form: rstd = 1 / sqrt(ms + eps)
 *       (the 1/K factor applied to each square before the sum);
 *       y = (x * rstd) * gamma   (gamma optional).
 *   AT-10 RMSNorm + Linear (same page, sec. 2 "standard compute flow" and
 *       sec. 4 "C stage", BF16 mode): a = bf16(y);
 *       out[t, n] = bf16(sum_k a[t, k] * W[n, k]), W stored [N, K]
 *       (b_trans = True), fp32 accumulation.
 *   mhc_pre skinny form (same page, sec. 8; "SK-03 Linear Projection
 *       (Norm->MatMul)" page, "shape variant: huge reduction x tiny output
 *       width"): no gamma, FP32 compute, FP32 output:
 *       out[t, n] = fp32(sum_k y[t, k] * W[n, k]).
 *   AT-11 RMSNorm + Linear + Quant (AT-10 page sec. 4, INT8 W8A8 mode; SK-03
 *       page, "quantised variant (AT-11)"): per-token symmetric INT8 codes
 *       q = sat(rint_half_even(y * 127 / amax)), amax = max_k |y[t, k]|,
 *       x_scale = amax / 127; exact int32 acc = sum_k q[t, k] * Wq[n, k];
 *       out = bf16(float(acc) * (x_scale[t] * w_scale[n])) (dequant order of
 *       the "SK-14 general multi-MatMul skeleton" page, QuantMatMulReduceSum).
 *   MLA q chain (AT-10 page, sec. 5 "MLAProlog" and sec. 9 golden chain):
 *       qa = bf16(x @ W_qa^T); z = bf16(RMSNorm(qa) * gamma_cq);
 *       out = bf16(z @ W_qb^T).
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer of the current CUDA device,
 *     contiguous and row-major, owned by the caller.  The library allocates
 *     no device memory: scratch space comes from the caller's `workspace`,
 *     sized by rnl_workspace_size().  (Exception: the host-buffer pipeline
 *     at the end, which takes host pointers for x and out and owns its
 *     device staging.)
 *   - bf16 data are passed as `const void*` (IEEE bfloat16 bit patterns).
 *   - Base pointers (tensors and workspace) must be 16-byte aligned; K must
 *     be a multiple of 8 (bf16 rows) -- the TMA copy engine moves rows whose
 *     pitch is a multiple of 16 bytes.  T and N are arbitrary (tails are
 *     handled).  T == 0 is a no-op.
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream).  Argument errors are returned before anything is enqueued.
 *     RNL_ERR_LAUNCH reports a CUDA launch error.  A kernel that gives up on
 *     a wait (a bug, never expected) records it in a device error word that
 *     rnl_check_device_error() reads.
 *   - The library keeps per-device set-up (kernel attributes, device
 *     properties, the address of the built-in scratch array) for the life of
 *     the process; after cudaDeviceReset() on a device, reload the library
 *     before using that device again.
 *   - Calls on the same stream are ordered; calls that share a workspace
 *     must not overlap on the GPU.
 *   - A call may be captured in a CUDA graph and replayed with new contents
 *     in the same buffers.  Make one uncaptured call of the same kind first
 *     (a first call per device and kernel does host-side set-up).  The
 *     cross-CTA flags some calls keep in the workspace (the CTA-pair GEMM's
 *     stream-K hand-off, QuantMatMulReduceSum's batch sum) are set back to 0
 *     by the launch that consumes them, so every replay waits for its own.
 *     After rnl_check_device_error() has reported RNL_ERR_TIMEOUT, set the
 *     failed call's workspace to zero before a graph that uses it replays.
 */
#ifndef RNL_H
#define RNL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream).  NULL = default stream. */
typedef struct CUstream_st *rnl_stream_t;

typedef enum rnl_status {
  RNL_OK = 0,
  RNL_ERR_NULL = 1,        /* a required pointer is NULL */
  RNL_ERR_SHAPE = 2,       /* a size is negative, zero where not allowed, or too large */
  RNL_ERR_ALIGN = 3,       /* a pointer or K violates the 16-byte rule */
  RNL_ERR_ARG = 4,         /* bad mode / dtype value, or eps not finite or negative */
  RNL_ERR_WORKSPACE = 5,   /* workspace smaller than rnl_workspace_size() */
  RNL_ERR_LAUNCH = 6,      /* CUDA returned an error when launching */
  RNL_ERR_TIMEOUT = 7,     /* a kernel gave up waiting (device error word set) */
  RNL_ERR_UNSUPPORTED = 8, /* argument combination the library does not provide */
  RNL_ERR_DEVICE = 9,      /* no sm_103 device current, or a driver entry point missing */
  RNL_ERR_BOUNDS = 10      /* a device-side bounds check failed (debug builds only) */
} rnl_status;

/* AT-03 rsqrt_mode */
enum { RNL_NORM_RSQRT = 0, RNL_NORM_SQRT_DIV = 1 };
/* AT-09 out_dtype */
enum { RNL_OUT_BF16 = 0, RNL_OUT_FP32 = 1 };
/* operation ids for rnl_workspace_size */
enum {
  RNL_OP_BF16 = 0,
  RNL_OP_W8A8 = 1,
  RNL_OP_MLA = 2,
  RNL_OP_GEMM_S8 = 3,
  RNL_OP_QKV_ROPE = 4,
  RNL_OP_QMRS = 5,
  RNL_OP_MXFP8 = 6,
  RNL_OP_W8A8_PREPARED = 7
};

/* Library version (major * 10000 + minor * 100 + patch). */
int rnl_version(void);

/*
 * 1 for a debug build (compiled with RNL_DEBUG), 0 otherwise.  A debug build
 * computes the same results and additionally checks, on the device, every
 * shared-memory stage offset, TMEM column range, workspace record or flag
 * index and output index of its GEMM, norm-pass and skinny kernels before
 * use; a failed check skips that access, and rnl_check_device_error() then
 * returns RNL_ERR_BOUNDS with the check's site.  No kernel traps.
 */
int rnl_debug_build(void);

/* Human-readable name of a status code (static string). */
const char *rnl_status_string(rnl_status s);

/*
 * Bytes of workspace an operation needs for the given sizes (0 is possible).
 *   RNL_OP_BF16:    T, K, N; N2 = out_dtype (RNL_OUT_BF16 / RNL_OUT_FP32)
 *   RNL_OP_W8A8:    T, K, N; N2 ignored
 *   RNL_OP_MLA:     T, K, N = N1, N2
 *   RNL_OP_GEMM_S8: T = M, K, N; N2 ignored
 *   RNL_OP_QKV_ROPE: T, K, N = (n_q_heads + 2 * n_kv_heads) * head_dim; N2 ignored
 *   RNL_OP_QMRS:    T = M, K, N, N2 = B (the batch)
 *   RNL_OP_MXFP8:   T, K, N; N2 ignored (rmsnorm_linear_mxfp8 and mxfp8_scaled_mm)
 *   RNL_OP_W8A8_PREPARED: T, K, N; N2 ignored (rmsnorm_linear_w8a8_prepared)
 * Returns (size_t)-1 for invalid sizes.  Host-only; needs no GPU.
 */
size_t rnl_workspace_size(int op, int64_t T, int64_t K, int64_t N, int64_t N2);

/*
 * AT-10 RMSNorm + Linear, or (out_dtype = RNL_OUT_FP32) the mhc_pre FP32 form.
 *   x      bf16 [T, K]          activations
 *   gamma  bf16 [K] or NULL     has_gamma = (gamma != NULL); must be NULL
 *                               with RNL_OUT_FP32 (the mhc_pre form has no
 *                               gamma), else RNL_ERR_UNSUPPORTED
 *   W      bf16 [N, K]          weight, K contiguous (b_trans = True)
 *   eps    >= 0, finite
 *   norm_mode  RNL_NORM_RSQRT or RNL_NORM_SQRT_DIV
 *   out    bf16 [T, N] (RNL_OUT_BF16) or fp32 [T, N] (RNL_OUT_FP32)
 * Kernels: bf16 out -> row-norm/cast pass then the tcgen05 GEMM;
 * bf16 out with T <= 4, K >= 2048, N >= 1024 and T * K * 2 <= 96 KB (a
 * decode step) -> one matrix-vector launch over every SM (the environment
 * variable RNL_DECODE=0 selects the GEMM path instead, RNL_DECODE_ROWS=1|2
 * fixes the weight rows per warp group; same result bound);
 * fp32 out with N <= 64 -> the split-K streaming kernel (one read of x);
 * fp32 out with N > 64 -> row rstd pass then the GEMM with a row-scale
 * epilogue.
 */
rnl_status rmsnorm_linear_bf16(const void *x, const void *gamma, const void *W, int64_t T,
                               int64_t K, int64_t N, float eps, int norm_mode, void *out,
                               int out_dtype, void *workspace, size_t workspace_bytes,
                               rnl_stream_t stream);

/*
 * AT-10 with the options of its two atoms and the residual add in front
 * (AT-10 pattern page: sec. 3, the AT-03 parameter table -- has_bias,
 * output_rstd; sec. 4, the AT-09 parameters -- has_bias; sec. 6,
 * Qwen3PreAttn -- the norm is applied to x_add, the input after the
 * residual add).  bf16 output.
 *   x         bf16 [T, K]
 *   residual  bf16 [T, K] or NULL: x_add = bf16(x + residual), rounded once
 *             (the correctly rounded bf16 of the exact sum); NULL: x_add = x
 *   x_sum_out bf16 [T, K] or NULL: receives x_add (needs residual, else
 *             RNL_ERR_ARG).  It may be x or residual itself (the in-place
 *             add of InplaceAddRmsNorm); any other overlap with them is
 *             RNL_ERR_ARG.
 *   gamma     bf16 [K] or NULL;  beta bf16 [K] or NULL (AT-03 has_bias)
 *   W         bf16 [N, K];  bias bf16 [N] or NULL (AT-09 has_bias)
 *   out       bf16 [T, N]:  out = bf16(sum_k a[t,k] * W[n,k] + bias[n]),
 *             a = bf16((x_add * rstd) * gamma + beta), FP32 arithmetic
 *   rstd_out  fp32 [T] or NULL (AT-03 output_rstd): rstd of x_add's row
 * Workspace: rnl_workspace_size(RNL_OP_BF16, T, K, N, RNL_OUT_BF16).
 * Alignment: 16 bytes for every tensor except rstd_out (4 bytes); K % 8.
 */
rnl_status rmsnorm_linear_bf16_ex(const void *x, const void *residual, void *x_sum_out,
                                  const void *gamma, const void *beta, const void *W,
                                  const void *bias, int64_t T, int64_t K, int64_t N, float eps,
                                  int norm_mode, void *out, float *rstd_out, void *workspace,
                                  size_t workspace_bytes, rnl_stream_t stream);

/*
 * The V stage after the qkv projection (AT-10 pattern page, sec. 6,
 * Qwen3PreAttn: the projection output is split into Q, K and V, then Q and K
 * get a per-head RMSNorm and the rotary embedding).
 *   y         bf16 [T, (n_q_heads + 2 * n_kv_heads) * head_dim]: the q heads,
 *             then the k heads, then the v heads (column ranges)
 *   head_dim  64, 128 or 256 (else RNL_ERR_UNSUPPORTED)
 *   q_gamma, k_gamma  bf16 [head_dim]: the per-head norms' weights
 *   eps       of the per-head norms (rsqrt form, FP32):
 *             z = bf16((h * rsqrt(mean(h^2) + eps)) * gamma)
 *   positions int32 [T]: each token's row of the angle table; a value outside
 *             [0, max_pos) leaves that token's q / k rows unwritten and makes
 *             the next rnl_check_device_error() return RNL_ERR_ARG
 *   cos_sin   fp32 [max_pos, head_dim]: row p = cos of the head_dim / 2
 *             angles, then their sin (a model's rotary cache); rotate-half
 *             pairing: o[i] = z[i] c_i - z[i + D/2] s_i,
 *             o[i + D/2] = z[i + D/2] c_i + z[i] s_i, bf16 out
 *   q_out bf16 [T, n_q_heads, head_dim];  k_out, v_out bf16 [T, n_kv_heads,
 *             head_dim] (v heads copied unchanged)
 * 16-byte aligned tensors (positions: 4 bytes).  No workspace.
 */
rnl_status rnl_qkv_rope(const void *y, int64_t T, int64_t n_q_heads, int64_t n_kv_heads,
                        int64_t head_dim, const void *q_gamma, const void *k_gamma, float eps,
                        const int32_t *positions, const float *cos_sin, int64_t max_pos,
                        void *q_out, void *k_out, void *v_out, rnl_stream_t stream);

/*
 * rmsnorm_linear_bf16 (AT-10, bf16 out, N = (n_q_heads + 2 * n_kv_heads) *
 * head_dim) followed by rnl_qkv_rope on its output.  With head_dim 128 and a
 * projection large enough for the CTA-pair GEMM, the stage runs in that
 * GEMM's epilogue on the bf16-rounded projection values and the projection
 * output is never written; otherwise it lives in the workspace and the
 * separate stage reads it.  Workspace: rnl_workspace_size(RNL_OP_QKV_ROPE,
 * T, K, N, 0) bytes either way.  head_eps is the per-head norms' eps.
 * Arguments of both stages are checked before anything is enqueued; a
 * position outside [0, max_pos) is reported by rnl_check_device_error as
 * RNL_ERR_ARG on both routes.
 */
rnl_status rmsnorm_linear_qkv_rope(const void *x, const void *gamma, const void *W, int64_t T,
                                   int64_t K, int64_t n_q_heads, int64_t n_kv_heads,
                                   int64_t head_dim, float eps, int norm_mode,
                                   const void *q_gamma, const void *k_gamma, float head_eps,
                                   const int32_t *positions, const float *cos_sin,
                                   int64_t max_pos, void *q_out, void *k_out, void *v_out,
                                   void *workspace, size_t workspace_bytes, rnl_stream_t stream);

/*
 * QuantMatMulReduceSum ("SK-14 general multi-MatMul skeleton" page, variant
 * A and its parameter table): a batch of exact INT8 matmuls, dequantised and
 * summed over the batch.
 *   x1        int8 [B, M, K];  x2 int8 [B, K, N] (N contiguous, as on the page)
 *   x1_scale  fp32 [B, M];     x2_scale bf16 [N]
 *   out       bf16 [M, N] = bf16(sum_b fp32(acc_b) * (x1_scale[b, m] *
 *             fp32(x2_scale[n]))), acc_b = x1[b] @ x2[b] exact in int32; every
 *             step after the matmul is one FP32 operation, the batch summed in
 *             increasing b (so the result does not depend on the kernel's
 *             tiling).  |acc_b| must fit int32 (K <= 133144 always does).
 * K % 16 == 0 and N % 16 == 0; 16-byte aligned x1, x2, out; 4-byte x1_scale.
 * Workspace: rnl_workspace_size(RNL_OP_QMRS, M, K, N, B) bytes.
 */
rnl_status quant_matmul_reduce_sum(const int8_t *x1, const int8_t *x2, const float *x1_scale,
                                   const void *x2_scale, int64_t B, int64_t M, int64_t K,
                                   int64_t N, void *out, void *workspace, size_t workspace_bytes,
                                   rnl_stream_t stream);

/*
 * AT-11 RMSNorm + per-token INT8 quant + exact INT8 x INT8 -> INT32 matmul +
 * FP32 dequant, BF16 out.
 *   x        bf16 [T, K];  gamma bf16 [K] or NULL
 *   Wq       int8 [N, K] with values in [-127, 127];  K % 16 == 0
 *   w_scale  fp32 [N]     per-output-channel weight scale
 *   out      bf16 [T, N]
 *   q_out        optional int8 [T, K]: the activation codes (NULL = not written)
 *   x_scale_out  optional fp32 [T]: amax / 127 per row (NULL = not written)
 * The integer accumulation is exact for every input (chunks of at most 1024
 * products are summed exactly on the tensor pipe, then added in int32);
 * a sum outside the int32 range wraps as two's complement (impossible for
 * K <= 133144).  Each call widens Wq to the tensor cores' bf16 operand in
 * the workspace; a weight used for many calls is better prepared once
 * (rnl_w8a8_prepare_weight, rmsnorm_linear_w8a8_prepared).
 */
rnl_status rmsnorm_linear_w8a8(const void *x, const void *gamma, const int8_t *Wq,
                               const float *w_scale, int64_t T, int64_t K, int64_t N, float eps,
                               int norm_mode, void *out, int8_t *q_out, float *x_scale_out,
                               void *workspace, size_t workspace_bytes, rnl_stream_t stream);

/*
 * The W8A8 weight prepared once, outside the per-call path, as the pages do
 * with weights (the SK-03 skeleton page, "shape variant: huge reduction x
 * tiny output width": the weight is transposed once on the host, not per
 * call).  Wq int8 [N, K] with values in [-127, 127] is widened exactly to
 * Wb bf16 [N, K], the operand the integer matmul reads (caller-owned,
 * 2 N K bytes).  K % 16 == 0; Wq and Wb 16-byte aligned.  Enqueued on
 * `stream`.
 */
rnl_status rnl_w8a8_prepare_weight(const int8_t *Wq, int64_t N, int64_t K, void *Wb,
                                   rnl_stream_t stream);

/*
 * rmsnorm_linear_w8a8 with a weight prepared by rnl_w8a8_prepare_weight:
 * Wb bf16 [N, K] (the exact integers of Wq; any other contents void the
 * exactness of the integer sums).  Other arguments, results and alignment
 * as rmsnorm_linear_w8a8; workspace rnl_workspace_size(RNL_OP_W8A8_PREPARED,
 * T, K, N, 0) bytes (no room for a widened weight).
 */
rnl_status rmsnorm_linear_w8a8_prepared(const void *x, const void *gamma, const void *Wb,
                                        const float *w_scale, int64_t T, int64_t K, int64_t N,
                                        float eps, int norm_mode, void *out, int8_t *q_out,
                                        float *x_scale_out, void *workspace, size_t workspace_bytes,
                                        rnl_stream_t stream);

/*
 * Per-head RMSNorm of a projection output (AT-10 pattern page, sec. 9: the
 * MLA prolog's golden chain reshapes q_b_proj to [num_heads, head_dim] and
 * normalises it again, each head row on its own).
 *   y      bf16 [T, n_heads * head_dim]
 *   gamma  bf16 [head_dim] or NULL (the page's helper for this norm has none)
 *   out    bf16 [T, n_heads * head_dim]; may be y itself (in place), must not
 *          overlap it otherwise (RNL_ERR_ARG)
 *   per head: rstd as norm_mode (FP32), out = bf16((y * rstd) * gamma)
 * head_dim a multiple of 64 in [64, 512] (else RNL_ERR_UNSUPPORTED); y, out,
 * gamma 16-byte aligned.  No workspace.
 */
rnl_status rnl_head_rmsnorm(const void *y, int64_t T, int64_t n_heads, int64_t head_dim,
                            const void *gamma, float eps, int norm_mode, void *out,
                            rnl_stream_t stream);

/*
 * mla_q_chain followed by rnl_head_rmsnorm on its output, in place: the MLA
 * q chain up to the per-head norm after q_b (the same page passage).  The
 * head norm uses the chain's norm_mode (the page's chain uses the sqrt+div
 * form for both norms), head_eps and head_gamma (bf16 [head_dim] or NULL);
 * N2 % head_dim == 0.  Arguments and workspace otherwise as mla_q_chain
 * (rnl_workspace_size(RNL_OP_MLA, ...)).
 */
rnl_status mla_q_chain_head_norm(const void *x, const void *W_qa, const void *gamma_cq,
                                 const void *W_qb, int64_t T, int64_t K, int64_t N1, int64_t N2,
                                 float eps, int norm_mode, int64_t head_dim, const void *head_gamma,
                                 float head_eps, void *out, void *qa_out, void *workspace,
                                 size_t workspace_bytes, rnl_stream_t stream);

/*
 * AT-11 in MXFP8 mode: RMSNorm, MX quantisation of the normed rows, and
 * scaled_mm(x_fp8, w_fp8, FP32, x_scale, w_scale) against an MXFP8 weight
 * (AT-10 pattern page, sec. 4, AT-09 quant_mode mxfp8; SK-14 skeleton page,
 * GMM-MXFP8: E4M3FN data, E8M0FNU scales, one scale per 64 elements).
 *   x        bf16 [T, K];  gamma bf16 [K] or NULL
 *   w_codes  E4M3FN bytes [N, K];  w_scale E8M0 bytes [N, K / block]
 *            (element k of row n is value(w_codes[n, k]) * 2^(w_scale[n, k / block] - 127))
 *   block    elements per scale along K: 64 (the page's) or 32 (OCP MX)
 *   out      bf16 [T, N] (RNL_OUT_BF16: the FP32 result cast once) or fp32 [T, N]
 *   x_codes_out  optional E4M3FN bytes [T, K]: the activation codes (NULL = not written)
 *   x_scale_out  optional E8M0 bytes [T, K / block]: their scales (NULL = not written)
 * Per block of the normed FP32 row y (the norm as in rmsnorm_linear_w8a8):
 * X = floor(log2 max|y|) - 8 (at least -127; an all-zero block gets -127),
 * scale byte X + 127, codes E4M3(y * 2^-X) rounded to nearest even and
 * saturated to +-448.  Codes and scales are exact functions of x, gamma and
 * eps (the FP32 sum of squares is the rounding of the exact sum).  The
 * product is accumulated in FP32 on the tensor cores from the exactly
 * dequantised operands.  K % block == 0, T * K and N * K below 2^36
 * (else RNL_ERR_SHAPE); x, gamma, w_codes, out 16-byte aligned.  Workspace: rnl_workspace_size(RNL_OP_MXFP8, T, K, N, 0) bytes.
 * Non-finite inputs and weights whose dequantised values exceed the bf16
 * range give unspecified (but memory-safe) results.
 */
rnl_status rmsnorm_linear_mxfp8(const void *x, const void *gamma, const uint8_t *w_codes,
                                const uint8_t *w_scale, int64_t T, int64_t K, int64_t N, float eps,
                                int norm_mode, int64_t block, void *out, int out_dtype,
                                uint8_t *x_codes_out, uint8_t *x_scale_out, void *workspace,
                                size_t workspace_bytes, rnl_stream_t stream);

/*
 * scaled_mm(x_fp8, w_fp8, FP32, x_scale, w_scale) on MXFP8 operands already
 * quantised (the same page passages): out[t, n] = sum_k value(x_codes[t, k])
 * 2^(x_scale[t, k/block] - 127) value(w_codes[n, k]) 2^(w_scale[n, k/block] - 127),
 * FP32 accumulation, bf16 or fp32 out as above.  Layouts, alignment and
 * workspace as rmsnorm_linear_mxfp8 (x_codes [T, K], x_scale [T, K / block]).
 */
rnl_status mxfp8_scaled_mm(const uint8_t *x_codes, const uint8_t *x_scale, const uint8_t *w_codes,
                           const uint8_t *w_scale, int64_t T, int64_t K, int64_t N, int64_t block,
                           void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                           rnl_stream_t stream);

/*
 * MLA two-stage q chain.
 *   x bf16 [T, K];  W_qa bf16 [N1, K];  gamma_cq bf16 [N1];  W_qb bf16 [N2, N1]
 *   out bf16 [T, N2];  qa_out optional bf16 [T, N1] (the stage-1 output)
 *   N1 % 8 == 0.  norm_mode as above (the pages' MLAProlog uses sqrt+div).
 */
rnl_status mla_q_chain(const void *x, const void *W_qa, const void *gamma_cq, const void *W_qb,
                       int64_t T, int64_t K, int64_t N1, int64_t N2, float eps, int norm_mode,
                       void *out, void *qa_out, void *workspace, size_t workspace_bytes,
                       rnl_stream_t stream);

/* Size of the scratch array built into the library for the call below. */
#define RNL_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * rmsnorm_linear_skinny_noalloc -- the mhc_pre FP32 form (the same result as
 * rmsnorm_linear_bf16 with gamma = NULL, out_dtype = RNL_OUT_FP32 and
 * N <= 64) without any workspace and without allocating device memory.
 * The source pages have no counterpart of this call; it exists for how the
 * library is embedded, not for the method.
 *
 * Who needs it: callers that cannot call cudaMalloc, such as code running
 * inside a host program that owns every device allocation (a serving
 * engine with a fixed memory pool, or a plugin that is handed only its
 * input and output buffers).  They have no scratch buffer to pass, and a
 * cudaMalloc of their own could synchronise the device and grow the
 * process's memory behind the owner's back.
 *
 * How: the split-K scratch lives in a RNL_NOALLOC_SCRATCH_BYTES (16 MiB)
 * array inside the library, which every GPU that loads the library holds
 * until the process exits.  The call makes no cudaMalloc, cudaFree or other
 * allocating call.  It needs (ceil(T/128) + G) * 128 * (NP + 1) * 4 bytes of
 * that array, G = min(SM count, work blocks), NP = 32 for N <= 32 and 64
 * for N <= 64: on a 152-SM GB300 up to T = 107,520 rows (N <= 32) or
 * T = 45,056 rows (N <= 64).  Larger T returns RNL_ERR_WORKSPACE with
 * nothing enqueued; N > 64 returns RNL_ERR_UNSUPPORTED.
 *
 * Sharing: all calls on a device use the same array.  Calls whose GPU work
 * can overlap (other streams, other host threads) race on it; serialise
 * them.  The array keeps the previous call's contents; every value the
 * kernels read is written earlier in the same call, so nothing is cleared.
 *
 * Set-up: the first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current) and caches it;
 * make that first call before any stream capture.
 *
 * Arguments as rmsnorm_linear_bf16: x bf16 [T, K], W bf16 [N, K],
 * out fp32 [T, N], 16-byte aligned, K % 8 == 0, eps >= 0, norm_mode.
 */
rnl_status rmsnorm_linear_skinny_noalloc(const void *x, const void *W, int64_t T, int64_t K,
                                         int64_t N, float eps, int norm_mode, float *out,
                                         rnl_stream_t stream);

/*
 * The exact integer matmul of the W8A8 path on its own (AT-09 INT8 mode):
 * C[m, n] = sum_k A[m, k] * B[n, k], int8 inputs in [-127, 127], int32 out
 * [M, N].  K % 16 == 0.  Used to check bit-exactness against a reference.
 */
rnl_status rnl_gemm_s8s8s32(const int8_t *A, const int8_t *B, int32_t *C, int64_t M, int64_t N,
                            int64_t K, void *workspace, size_t workspace_bytes,
                            rnl_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device error words of
 * every kernel module.  RNL_OK if no kernel gave up on a wait or met a bad
 * argument, RNL_ERR_TIMEOUT for a wait that gave up, RNL_ERR_ARG for a bad
 * argument seen on the device (a rotary position outside its table); *site,
 * if not NULL, receives the first recorded site.  RNL_ERR_LAUNCH if the
 * synchronisation itself failed.
 */
rnl_status rnl_check_device_error(rnl_stream_t stream, int *site);

/*
 * Failure-detection self-test (no counterpart on the pages).  Enqueues one
 * small kernel that waits, with a 1 ms limit, on a barrier nothing arrives
 * on -- the bounded wait every kernel of the library uses.  The wait gives
 * up and records wait site 99 in a device error word; the kernel then
 * returns normally.  A following rnl_check_device_error() reports
 * RNL_ERR_TIMEOUT with *site == 99 and clears the word; the CUDA context
 * stays usable.  Returns RNL_OK when the kernel was enqueued.
 */
rnl_status rnl_selftest_wait_timeout(rnl_stream_t stream);

/*
 * Bounds-check self-test of a debug build (no counterpart on the pages).
 * Enqueues one small kernel whose device-side check compares an index with
 * a deliberately smaller limit (the index still lies inside the kernel's own
 * array, so no access can leave it); the check fails, records site 98 and
 * skips the store.  A following rnl_check_device_error() reports
 * RNL_ERR_BOUNDS with *site == 98.  Release builds return
 * RNL_ERR_UNSUPPORTED and enqueue nothing.
 */
rnl_status rnl_selftest_bounds_check(rnl_stream_t stream);

/*
 * Host-buffer pipeline (no counterpart on the pages: how the projection is
 * fed when its activations live in host memory).  The calls above take
 * device pointers; a pipeline takes the activations x from, and returns the
 * output to, PAGE-LOCKED host memory (cudaHostAlloc / cudaHostRegister),
 * while the weights stay device pointers, resident across calls.
 *
 * A pipeline owns two slots of device staging (x and output buffers), one
 * workspace and three non-blocking streams: a host-to-device copy stream, a
 * kernel stream and a device-to-host copy stream.  Submitted call i uses
 * slot i % 2; its input copy overlaps the kernels of call i - 1 and the
 * output copy of call i - 2, so a stream of calls runs at the rate of the
 * slowest of the three (on GB300 usually the host link).  Submitting never
 * blocks the host.
 *
 * rnl_pipeline_create(op, T, K, N, N2, &pipe): sizes as rnl_workspace_size
 *   (RNL_OP_BF16: N2 = out_dtype; RNL_OP_W8A8: N2 ignored; RNL_OP_MLA:
 *   N = N1, N2).  Binds the pipeline to the current device and allocates
 *   2 * (T*K*2 + T*out_width*out_bytes) bytes of staging plus the workspace
 *   (cudaMalloc; RNL_ERR_WORKSPACE if that fails).  Every call is checked
 *   against these sizes only; the shape rules of the matching entry point
 *   apply (K % 8, K % 16 for W8A8, N1 % 8 for MLA).
 * rnl_pipeline_submit_*: the arguments of rmsnorm_linear_bf16 /
 *   rmsnorm_linear_w8a8 / mla_q_chain, with x_host and out_host host
 *   pointers (page-locked, else RNL_ERR_ARG) of T*K bf16 and of the output
 *   size; the weights, gamma and w_scale are device pointers that must stay
 *   valid and unchanged until the call completes.  x_host may be reused and
 *   out_host read only after rnl_pipeline_wait(ticket) returns.  *ticket
 *   receives the call's number (0, 1, 2, ...).  Argument errors return
 *   before anything is enqueued and leave the pipeline usable; a CUDA error
 *   while enqueuing makes every later submit return that status.  The
 *   W8A8 and MLA calls write no q_out / x_scale_out / qa_out.
 * rnl_pipeline_wait(pipe, ticket, &site): blocks until call `ticket` has
 *   written out_host (it may also wait for the next call of the same slot,
 *   if that one was already submitted), then reads the device error words
 *   as rnl_check_device_error does, without synchronising anything else.
 *   RNL_ERR_ARG for a ticket never issued.
 * rnl_pipeline_destroy(pipe): waits for everything submitted, frees the
 *   staging, workspace, streams and events.  NULL is a no-op.
 * A pipeline is not thread-safe; use one per host thread.
 */
typedef struct rnl_pipeline rnl_pipeline;
rnl_status rnl_pipeline_create(int op, int64_t T, int64_t K, int64_t N, int64_t N2,
                               rnl_pipeline **pipe);
rnl_status rnl_pipeline_submit_bf16(rnl_pipeline *pipe, const void *x_host, const void *gamma,
                                    const void *W, float eps, int norm_mode, void *out_host,
                                    int64_t *ticket);
rnl_status rnl_pipeline_submit_w8a8(rnl_pipeline *pipe, const void *x_host, const void *gamma,
                                    const int8_t *Wq, const float *w_scale, float eps,
                                    int norm_mode, void *out_host, int64_t *ticket);
rnl_status rnl_pipeline_submit_mla(rnl_pipeline *pipe, const void *x_host, const void *W_qa,
                                   const void *gamma_cq, const void *W_qb, float eps,
                                   int norm_mode, void *out_host, int64_t *ticket);
rnl_status rnl_pipeline_wait(rnl_pipeline *pipe, int64_t ticket, int *site);
rnl_status rnl_pipeline_destroy(rnl_pipeline *pipe);

/*
 * Kernel timing trace.  While enabled, every kernel launch made by the
 * library is bracketed by two CUDA events recorded on the launch stream
 * (up to 16384 launches between reads).  rnl_trace_read() waits for the recorded
 * events, copies up to `max` records (name, milliseconds) in launch order
 * and clears the ring; it returns the number copied.  names receives
 * 32-byte NUL-terminated strings.  Host bookkeeping only; not thread-safe.
 */
rnl_status rnl_trace_enable(int on);
int rnl_trace_read(char (*names)[32], float *ms, int max);

#ifdef __cplusplus
}
#endif

#endif /* RNL_H */
