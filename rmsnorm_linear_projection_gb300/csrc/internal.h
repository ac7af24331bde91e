// internal.h -- host-side interfaces between the C ABI (api.cu) and the
// kernel modules (rowwise.cu, gemm_tc.cu, skinny.cu).  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "rnl.h"

namespace rnl {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int major = 0, minor = 0;
  int max_smem_optin = 0;
};

// Current device's properties (cached per device).  RNL_ERR_DEVICE if the
// device is not a compute-capability 10.3 part.
rnl_status current_device(DeviceInfo* info);

// 2-D tensor map over a row-major matrix [outer, inner] of `elem_bytes`
// elements with row pitch `row_bytes`; box = box_inner x box_outer elements;
// 128-byte swizzle; out-of-range elements read as zero.
rnl_status make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                       uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                       uint32_t box_outer);
// The same without swizzle (boxes land in shared memory row after row).
rnl_status make_map_2d_plain(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                             uint64_t inner, uint64_t outer, uint64_t row_bytes,
                             uint32_t box_inner, uint32_t box_outer);

// Raises a kernel's dynamic shared-memory limit on `device` (the current one)
// to at least `bytes`: set on a (kernel, device)'s first call and again only
// when a call needs more than was set; thread-safe.  The cache outlives a
// cudaDeviceReset, which drops the attribute, so a reset device needs the
// library reloaded.
rnl_status ensure_smem_attr(const void* kernel, int device, size_t bytes);

// ---- kernel trace (api.cu) ----
void trace_before(cudaStream_t s);
void trace_after(cudaStream_t s, const char* name);

// ---- row-wise kernels (rowwise.cu) ----
// y = (x * rstd) * gamma cast to bf16 into A [T, K]; rstd_out optional.
rnl_status launch_norm_cast(const void* x, const void* gamma, int64_t T, int64_t K, float eps,
                            int mode, void* A, float* rstd_out, cudaStream_t s);
// The same as a persistent bulk-copy stream (normstream.cu), for K <= 4096;
// launched as a programmatic dependent.
bool norm_cast_stream_fits(int64_t K);
rnl_status launch_norm_cast_stream(const void* x, const void* gamma, int64_t T, int64_t K,
                                   float eps, int mode, void* A, cudaStream_t s);
// The same with the residual add in front and the AT-03 options (addnorm.cu,
// any K): x_add = bf16(x + residual) (residual may be null), written to
// x_sum_out when not null (may be x or residual); A = bf16((x_add * rstd) *
// gamma + beta) (gamma, beta may be null); rstd_out optional.
rnl_status launch_add_norm_cast(const void* x, const void* residual, void* x_sum_out,
                                const void* gamma, const void* beta, int64_t T, int64_t K,
                                float eps, int mode, void* A, float* rstd_out, cudaStream_t s);
// The same options on the streamed pass (normstream.cu), K <= 4096.
rnl_status launch_add_norm_cast_stream(const void* x, const void* residual, void* x_sum_out,
                                       const void* gamma, const void* beta, int64_t T, int64_t K,
                                       float eps, int mode, void* A, float* rstd_out,
                                       cudaStream_t s);
// rstd only.
rnl_status launch_row_rstd(const void* x, int64_t T, int64_t K, float eps, int mode, float* rstd,
                           cudaStream_t s);
// norm + per-token symmetric int8 codes: A gets the codes as bf16 values,
// q_out (optional) as int8, x_scale = amax / 127.
rnl_status launch_norm_quant(const void* x, const void* gamma, int64_t T, int64_t K, float eps,
                             int mode, void* A, int8_t* q_out, float* x_scale, cudaStream_t s);
// The same as a persistent stream (quantstream.cu) for K <= 4096: each row
// read once into registers; codes, int8 copy and x_scale as above.  With
// gamma and gmax_out (a device float, may be null): *gmax_out = max |gamma|.
bool quant_stream_fits(int64_t K);
rnl_status launch_quant_stream(const void* x, const void* gamma, int64_t T, int64_t K, float eps,
                               int mode, void* A, int8_t* q_out, float* x_scale, float* gmax_out,
                               cudaStream_t s);

// Exact integer products without chunks: a row of codes a (|a| <= 127) times
// an int8 weight row w (|w| <= 128) has every partial sum, in any order,
// bounded by 128 * sum_k |a_k|.  Below 2^24 every partial sum is an integer
// that binary32 holds exactly, so one FP32 accumulator over all of K gives
// the exact sum: sum_k |a_k| < 2^24 / 128.  For RMSNorm-quantised rows
// (q = rint(y * 127 / amax), y = (x * rstd) * gamma):
//   |q_k| <= |y_k| * 127 / amax + 1/2,  |y_k| <= |x_k| rstd max|gamma|,
//   sum |x_k| <= sqrt(K sum x_k^2)  (Cauchy-Schwarz),
//   rstd^2 sum x_k^2 = K ms / (ms + eps) <= K  (ms the mean square),
// each up to a few roundings, so sum |q| <= K max|gamma| / x_scale + K/2
// (x_scale = amax / 127): below the limit for every x_scale above
// exact_row_floor (the 1.005 covers the roundings many times over).
constexpr float kWideRowL1 = 131072.0f;
__host__ __device__ inline float exact_row_floor(float K, float gamma_max) {
  return K * gamma_max * 1.005f / (kWideRowL1 - 0.5f * K - 1.0f);
}
// the bound needs K/2 + 1 well below the limit
inline bool exact_rows_possible(int64_t K) { return K > 0 && K <= 65536; }
// Both of the above in one launch (norm-quantise rows of x and widening of
// the N x K weight run side by side); rows longer than 4096 fall back to the
// two launches.
rnl_status launch_w8a8_front(const void* x, const void* gamma, int64_t T, int64_t K, float eps,
                             int mode, void* A, int8_t* q_out, float* x_scale, const int8_t* Wq,
                             int64_t N, void* Wb, cudaStream_t s);
// QuantMatMulReduceSum operands in one launch (qmrs.cu): x1 int8 [B, M, K]
// -> bf16 [B * M, K]; x2 int8 [B, K, N] -> bf16 [B * N, K] (exact; the K-major
// operand of an ND int8 matrix); x2_scale bf16 [N] -> fp32.  K % 16 == 0 and
// N % 16 == 0; x2_dst 32-byte aligned.
rnl_status launch_qmrs_prep(const int8_t* x1, const int8_t* x2, const void* x2_scale, int64_t B,
                            int64_t M, int64_t K, int64_t N, void* x1_dst, void* x2_dst,
                            float* scale_dst, cudaStream_t s);
// int8 -> bf16 (exact), n elements, n % 16 == 0.
rnl_status launch_s8_to_bf16(const int8_t* src, int64_t n, void* dst, cudaStream_t s);

// ---- MXFP8 (mxfp8.cu) ----
// block must be 32 or 64 (elements per E8M0 scale along K).
bool mx_block_ok(int64_t block);
// norm + MX quantisation of x's rows, in one launch with the weight's part.
// Emulation path (sfa null): A = bf16 of the dequantised codes, codes
// [T, K] and scale bytes [T, K / block] optional, and the E4M3 weight
// [N, K] with its scales [N, K / block] dequantised into Wb.  Block-scaled
// path (sfa, sfb given): codes into q_out (required), scale bytes into s_out
// (optional), the scale atoms of the rows into sfa (128-row tiles, padded
// to a multiple of 256 rows) and of the weight into sfb (bn-row tiles), as
// mx_gemm_native reads them; A and Wb unused.  K % block == 0.
rnl_status launch_mx_front(const void* x, const void* gamma, int64_t T, int64_t K, float eps,
                           int mode, int64_t block, void* A, uint8_t* q_out, uint8_t* s_out,
                           const uint8_t* w_codes, const uint8_t* w_scale, int64_t N, void* Wb,
                           uint8_t* sfa, uint8_t* sfb, int bn, cudaStream_t s);
// Scale atoms of both operands from scale bytes [M, K / block] and [N, K / block].
rnl_status launch_mx_sf_prep(const uint8_t* a_scale, int64_t M, const uint8_t* b_scale, int64_t N,
                             int64_t K, int64_t block, uint8_t* sfa, uint8_t* sfb, int bn,
                             cudaStream_t s);
// Dequantisation of two MXFP8 operands [M, K] and [N, K] into bf16 A and B.
rnl_status launch_mx_dequant2(const uint8_t* a_codes, const uint8_t* a_scale, int64_t M,
                              const uint8_t* b_codes, const uint8_t* b_scale, int64_t N, int64_t K,
                              int64_t block, void* A, void* B, cudaStream_t s);

// ---- block-scaled MXFP8 GEMM (mxgemm.cu) ----
// Rows of B per output tile (the tiling of the weight's scale atoms).
int mx_native_bn();
// Bytes of the scale atoms of a [rows, K] operand cut into tiles of rows_per_tile rows.
size_t mx_sf_atoms_bytes(int64_t rows, int64_t K, int rows_per_tile);
// out [M, N] (bf16 or fp32) = scaled_mm of E4M3 codes a [M, K], b [N, K]
// (16-byte aligned, K % 32 == 0) with their scale atoms.
rnl_status launch_mx_gemm_native(const uint8_t* a_codes, const uint8_t* b_codes, const uint8_t* sfa,
                                 const uint8_t* sfb, int64_t M, int64_t N, int64_t K, void* out,
                                 int out_dtype, cudaStream_t s);

// ---- a few tokens against a wide weight (decode.cu) ----
// T <= 4 rows, K >= 2048, N >= 1024 outputs, the normalised rows within 96 KB.
bool decode_fits(int64_t T, int64_t K, int64_t N);
// AT-10 RMSNorm + Linear, bf16 out, the weight's rows spread over every SM.
rnl_status launch_decode(const void* x, const void* gamma, const void* W, int64_t T, int64_t K,
                         int64_t N, float eps, int mode, void* out, int sm_count, cudaStream_t s);
// The same on the tensor cores (decode_mma.cu): T <= 4, K % 8 == 0 and a K
// split whose ring and normalised rows fit in shared memory; the K split's
// partial sums and flags take decode_mma_workspace_bytes(N) of `ws`.
bool decode_mma_fits(int64_t T, int64_t K, int64_t N, int sm_count);
size_t decode_mma_workspace_bytes(int64_t N);
rnl_status launch_decode_mma(const void* x, const void* gamma, const void* W, int64_t T, int64_t K,
                             int64_t N, float eps, int mode, void* out, void* ws, size_t ws_bytes,
                             cudaStream_t s);

// ---- per-head RMSNorm (headnorm.cu) ----
// head_dim a multiple of 64 in [64, 512]
bool head_norm_dim_ok(int64_t D);
// out (may be y) = bf16((y * rstd) * gamma) per head row of D values of y
// [T, H * D]; gamma [D] may be null.
rnl_status launch_head_norm(const void* y, int64_t T, int64_t H, int64_t D, const void* gamma,
                            float eps, int mode, void* out, cudaStream_t s);

// ---- QKV split + per-head RMSNorm + RoPE (qkvrope.cu) ----
bool qkv_rope_head_dim_ok(int64_t D);
rnl_status launch_qkv_rope(const void* y, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                           const void* q_gamma, const void* k_gamma, float eps,
                           const int32_t* positions, const float* cos_sin, int64_t max_pos,
                           void* q, void* k, void* v, cudaStream_t s);

// ---- tcgen05 GEMM (gemm_tc.cu) ----
enum class Epi : int {
  kBf16 = 0,         // out bf16 = acc
  kRowScaleF32 = 1,  // out fp32 = acc * row_scale[m] (row_scale null: 1)
  kDequantBf16 = 2,  // out bf16 = float(exact int acc) * (row_scale[m] * col_scale[n])
  kInt32 = 3,        // out int32 = exact int acc
  // QuantMatMulReduceSum, one batch: v = fp32(exact int acc) * (row_scale[m] *
  // col_scale[n]) in FP32; acc_mode bit 0 adds the FP32 running sum in `out`
  // (earlier batches), bit 1 (last batch) writes bf16(v) to out_final instead
  // of v to `out`
  kDequantAccF32 = 4,
  // QuantMatMulReduceSum, all batches in one launch: work items (b, tile) in
  // b-major order; item (b, tile) adds v_b to the FP32 running sum that item
  // (b - 1, tile) left in `out` (waiting for its flag), and the last batch
  // writes bf16 to out_final.  A is [nbatch * M, K], B is [nbatch * N, K],
  // row_scale is [nbatch * M]
  kDequantBatchSum = 5,
  // bf16 projection y = bf16(acc) followed, in the CTA-pair kernel's
  // epilogue, by the QKV split + per-head RMSNorm + RoPE of head_dim 128
  // (each epilogue warp holds one 128-wide head of 32 rows); y itself is not
  // written
  kBf16QkvRope = 6,
};

// Arguments of the Epi::kBf16QkvRope epilogue (as rnl_qkv_rope's).
struct RopeEpiArgs {
  int Hq = 0, Hkv = 0;
  const void* q_gamma = nullptr;  // bf16 [128]
  const void* k_gamma = nullptr;  // bf16 [128]
  float eps = 0.f;
  const int32_t* pos = nullptr;   // [T]
  const float* cos_sin = nullptr; // [P, 128]
  int P = 0;
  void* q = nullptr;  // bf16 [T, Hq, 128]
  void* k = nullptr;  // bf16 [T, Hkv, 128]
  void* v = nullptr;  // bf16 [T, Hkv, 128]
};

struct GemmArgs {
  const void* A = nullptr;  // bf16 [M, K]
  const void* B = nullptr;  // bf16 [N, K]
  int64_t M = 0, N = 0, K = 0;
  void* out = nullptr;
  const float* row_scale = nullptr;
  const float* col_scale = nullptr;
  // Epi::kDequantBf16 on CTA pairs with A the codes of RMSNorm-quantised rows
  // (row_scale = x_scale = amax / 127, quantstream.cu): a tile whose rows all
  // pass the exactness bound on sum |q| (kWideRowL1) is accumulated in one
  // FP32 accumulator, the rest in 1024-product chunks; gamma_max (device
  // scalar, null: no gamma) is max |gamma|.  False: every tile in chunks.
  bool exact_rows = false;
  const float* gamma_max = nullptr;
  Epi epi = Epi::kBf16;
  // fused norm (bf16 epilogue only): A is raw x; the kernel feeds the MMA
  // bf16((x * a_rstd[m]) * a_gamma[k]) (a_gamma may be null)
  const float* a_rstd = nullptr;
  const void* a_gamma = nullptr;
  // AT-09 has_bias: bf16 [N] added to the accumulator before the output cast
  // (bf16 and dequant epilogues; may be null)
  const void* bias = nullptr;
  // partial sums and flags of the CTA-pair GEMM's stream-K tiles (see
  // gemm_pair.cu); without it every tile runs whole
  void* partial_ws = nullptr;
  size_t partial_ws_bytes = 0;
  // the CTA-pair GEMM's integer mode: one scratch slot per pair for the
  // running int32 sums of chunked tiles (kGemmPartialBytes suffice); the
  // integer mode runs on pairs only with it
  void* chunk_ws = nullptr;
  size_t chunk_ws_bytes = 0;
  // name of the launch in the kernel trace (default: the kernel's kind)
  const char* trace_name = nullptr;
  // Epi::kDequantAccF32 only
  int acc_mode = 0;
  void* out_final = nullptr;  // also Epi::kDequantBatchSum
  // Epi::kDequantBatchSum only: the batch count and one 64-bit flag per
  // (output tile, epilogue warp) of the 128 x 128 tiling (the finest), zeroed
  // or not: each launch uses its own tag
  int nbatch = 1;
  uint64_t* batch_flags = nullptr;
  // Epi::kBf16QkvRope only
  RopeEpiArgs rope;
};
// Bytes of the flags of Epi::kDequantBatchSum for M x N outputs.
inline size_t batch_flag_bytes(int64_t M, int64_t N) {
  return static_cast<size_t>((M + 127) / 128) * static_cast<size_t>((N + 127) / 128) * 8 * 8;
}

// Partial-sum slots of the CTA-pair GEMM's stream-K tiles (2 x 128 x 256
// 32-bit words each): one per pair, the last one holding the hand-off flags.
constexpr int kMaxPartialSlots = 128;
constexpr size_t kGemmPartialBytes = static_cast<size_t>(kMaxPartialSlots) * 2 * 128 * 256 * 4;
rnl_status launch_gemm(const GemmArgs& g, cudaStream_t s);
// The same GEMM on CTA pairs (tcgen05 cta_group::2, gemm_pair.cu); no fused norm.
rnl_status launch_gemm_pair(const GemmArgs& g, cudaStream_t s);
// A fresh tag for the cross-CTA flags of one launch (clock-seeded per-process
// counter, gemm_pair.cu): flags left in a reused workspace never match.
uint64_t next_flag_epoch();
// Whether launch_gemm runs a plain GEMM of this shape on CTA pairs.
bool gemm_uses_pair(int64_t M, int64_t N, int64_t K);
// Predicted pair-kernel time (microseconds) and resident CTA pairs (gemm_pair.cu).
double predict_pair_us(int64_t M, int64_t N, int64_t K, int sm_count, int pairs);
int resident_pairs_for(const DeviceInfo& dev);

// ---- skinny split-K streaming kernel (skinny.cu) ----
size_t skinny_workspace_bytes(int64_t T, int64_t K, int64_t N, int sm_count);
rnl_status launch_skinny(const void* x, const void* W, int64_t T, int64_t K, int64_t N, float eps,
                         int mode, float* out, void* workspace, size_t ws_bytes, int sm_count,
                         cudaStream_t s);

// ---- device error words (one per kernel module) ----
rnl_status read_clear_error_rowwise(unsigned int* word);
rnl_status read_clear_error_gemm(unsigned int* word);
rnl_status read_clear_error_skinny(unsigned int* word);
rnl_status read_clear_error_pair(unsigned int* word);
rnl_status read_clear_error_norm(unsigned int* word);
rnl_status read_clear_error_selftest(unsigned int* word);
rnl_status read_clear_error_rope(unsigned int* word);
rnl_status read_clear_error_mx(unsigned int* word);
rnl_status read_clear_error_quant(unsigned int* word);
rnl_status read_clear_error_decmma(unsigned int* word);
// Reads and clears all of them without synchronising (api.cu): RNL_OK, or
// RNL_ERR_TIMEOUT / RNL_ERR_ARG with the first recorded site in *site
// (optional).
rnl_status read_device_errors(int* site);

}  // namespace rnl
