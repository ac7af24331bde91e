// addnorm.cu -- the AT-10 V stage with the options of its RMSNorm atom and
// the residual add in front of it, for rows of any length (rows of up to 4096
// elements take the streamed pass of normstream.cu instead):
//
//   x_add = bf16(x + residual)                 (AT-10 pattern page, sec. 6:
//                                               Qwen3PreAttn normalises x_add,
//                                               the input after the residual add)
//   rstd  = rsqrt(mean(x_add^2) + eps)  |  1 / sqrt(...)   (sec. 3, variants A/B)
//   a     = bf16((x_add * rstd) * gamma + beta)            (sec. 3, AT-03 has_bias)
//
// with x_add written back on request (x_sum_out, as InplaceAddRmsNorm does)
// and rstd on request (AT-03 output_rstd).  Every option is a pointer that
// may be null.  The bf16 rounding of the FP32 sum x + residual is the
// correctly rounded bf16 of the exact sum for every pair of bf16 inputs: the
// FP32 sum is exact when the exponents differ by at most 16, and otherwise
// lies within 2^-16 of the larger input, far from any bf16 rounding midpoint.
//
// One warp per token row, 16-byte loads and stores, two passes over the row:
// the second reads x_add back from x_sum_out when it is written (this thread
// wrote those elements in the first pass), otherwise recomputes it.
// x_sum_out may be x or residual itself (in place): each element is read
// before the same thread writes it, and no load goes through the read-only
// path.
#include <cuda_bf16.h>

#include "internal.h"

namespace rnl {
namespace {

constexpr int kWarps = 8;  // rows per block

struct AddNormArgs {
  const uint4* x;
  const uint4* residual;  // may be null
  uint4* x_sum;           // may be null, x or residual
  const uint4* gamma;     // may be null
  const uint4* beta;      // may be null
  int64_t T;
  int nvec;  // K / 8
  float inv_d;
  float eps;
  uint4* A;
  float* rstd_out;  // may be null
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// bf16(a + b) element-wise on 8 bf16 pairs.
__device__ __forceinline__ uint4 add_bf16x8(const uint4& a, const uint4& b) {
  float fa[8], fb[8];
  unpack8(a, fa);
  unpack8(b, fb);
#pragma unroll
  for (int j = 0; j < 8; ++j) fa[j] = __fadd_rn(fa[j], fb[j]);
  return pack8(fa);
}

// Sum of squares of 8 elements into s, in the order of the variant.
template <int MODE>
__device__ __forceinline__ float add_squares(const uint4& u, float s, float inv_d) {
  float f[8];
  unpack8(u, f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (MODE == 0)
      s = fmaf(f[j], f[j], s);
    else
      s = fmaf(f[j] * f[j], inv_d, s);
  }
  return s;
}

// a = bf16((x_add * rstd) * gamma + beta) for one vector of 8.
__device__ __forceinline__ uint4 normed8(const uint4& u, float rstd, const uint4* gamma,
                                         const uint4* beta, int v) {
  float f[8];
  unpack8(u, f);
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], rstd);
  if (gamma != nullptr) {
    float g[8];
    unpack8(__ldg(gamma + v), g);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], g[j]);
  }
  if (beta != nullptr) {
    float b[8];
    unpack8(__ldg(beta + v), b);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = __fadd_rn(f[j], b[j]);
  }
  return pack8(f);
}

template <int MODE>
__global__ void __launch_bounds__(kWarps * 32) add_norm_cast_kernel(AddNormArgs p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= p.T) return;
  const int64_t off = row * p.nvec;
  const uint4* xr = p.x + off;
  const uint4* rr = p.residual != nullptr ? p.residual + off : nullptr;
  uint4* sr = p.x_sum != nullptr ? p.x_sum + off : nullptr;
  uint4* ar = p.A + off;
  float s = 0.f;
  for (int v = lane; v < p.nvec; v += 32) {
    uint4 u = xr[v];
    if (rr != nullptr) u = add_bf16x8(u, rr[v]);
    if (sr != nullptr) sr[v] = u;
    s = add_squares<MODE>(u, s, p.inv_d);
  }
  s = warp_sum(s);
  const float rstd = (MODE == 0) ? rsqrtf(s * p.inv_d + p.eps) : 1.0f / sqrtf(s + p.eps);
  if (p.rstd_out != nullptr && lane == 0) p.rstd_out[row] = rstd;
  for (int v = lane; v < p.nvec; v += 32) {
    uint4 u;
    if (sr != nullptr) {
      u = sr[v];  // written by this thread in the first pass
    } else {
      u = xr[v];
      if (rr != nullptr) u = add_bf16x8(u, rr[v]);
    }
    ar[v] = normed8(u, rstd, p.gamma, p.beta, v);
  }
}

}  // namespace

rnl_status launch_add_norm_cast(const void* x, const void* residual, void* x_sum_out,
                                const void* gamma, const void* beta, int64_t T, int64_t K,
                                float eps, int mode, void* A, float* rstd_out, cudaStream_t s) {
  if (T == 0) return RNL_OK;
  AddNormArgs a;
  a.x = static_cast<const uint4*>(x);
  a.residual = static_cast<const uint4*>(residual);
  a.x_sum = static_cast<uint4*>(x_sum_out);
  a.gamma = static_cast<const uint4*>(gamma);
  a.beta = static_cast<const uint4*>(beta);
  a.T = T;
  a.nvec = static_cast<int>(K / 8);
  a.inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  a.eps = eps;
  a.A = static_cast<uint4*>(A);
  a.rstd_out = rstd_out;
  const unsigned blocks = static_cast<unsigned>((T + kWarps - 1) / kWarps);
  trace_before(s);
  if (mode == RNL_NORM_RSQRT)
    add_norm_cast_kernel<0><<<blocks, kWarps * 32, 0, s>>>(a);
  else
    add_norm_cast_kernel<1><<<blocks, kWarps * 32, 0, s>>>(a);
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "add_norm_cast");
  return st;
}

}  // namespace rnl
