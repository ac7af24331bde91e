// decode.cu -- the AT-10 RMSNorm + Linear (bf16 out) for a handful of tokens
// (T <= 8, a decode step) against a wide weight.  With so few rows the
// projection is a matrix-vector product bound by reading W once: the
// tensor-core GEMM would use one 128-row tile per weight block and occupy a
// fraction of the SMs (about 1.7 TB/s measured at T = 1 against the qkv
// weight), so this kernel spreads W's rows over every SM instead:
//
//   every CTA normalises the T rows into shared memory, all its threads
//   sharing each row (AT-10 pattern page, sec. 3: rstd = rsqrt(mean(x^2) +
//   eps) | 1 / sqrt(...), a = bf16((x rstd) gamma));
//   each warp then takes weight rows n in turn (grid-stride, every warp the
//   same number of rows, the grid resident at once), streams the row with
//   16-byte loads (four in flight per lane; the first row's issued before
//   the norm), accumulates the T dot products in FP32 and reduces them across
//   the warp: out[t, n] = bf16(sum).
//
// bf16 products are exact in FP32; the summation order differs from the
// tensor-core path, inside the same bf16 output bound.
#include <cuda_bf16.h>

#include "internal.h"

namespace rnl {
namespace {

constexpr int kMaxTokens = 8;
constexpr int kWarps = 8;
constexpr int kSmemMax = 96 * 1024;  // the normalised rows: T * K * 2 bytes
constexpr int kInFlight = 4;         // 16-byte weight loads in flight per lane

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int MODE>
__global__ void __launch_bounds__(kWarps * 32)
    decode_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gamma,
                  const uint4* __restrict__ W, int T, int nvec, int N, float inv_d, float eps,
                  __nv_bfloat16* __restrict__ out) {
  extern __shared__ uint4 a_s[];  // [T][nvec]
  __shared__ float red[kWarps][kMaxTokens];
  __shared__ float rstd_s[kMaxTokens];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the first weight row's first loads go out before the norm, which does
  // not need them: their round trip overlaps it
  const int stride = gridDim.x * kWarps;
  const int n_first = blockIdx.x * kWarps + warp;
  uint4 w_first[kInFlight];
#pragma unroll
  for (int i = 0; i < kInFlight; ++i) {
    const int v = lane + 32 * i;
    w_first[i] = (n_first < N && v < nvec) ? __ldcs(W + static_cast<int64_t>(n_first) * nvec + v)
                                           : make_uint4(0u, 0u, 0u, 0u);
  }
  // 1. the normalised rows: all 256 threads share every row (thread i takes
  //    vectors i, i + 256, ...), the rows' loads issued together
  {
    float ss[kMaxTokens];
#pragma unroll
    for (int t = 0; t < kMaxTokens; ++t) ss[t] = 0.f;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      uint4 u[kMaxTokens];
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t < T) u[t] = __ldg(x + static_cast<int64_t>(t) * nvec + v);
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t) {
        if (t >= T) break;
        float f[8];
        unpack8(u[t], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss[t] = MODE == 0 ? fmaf(f[j], f[j], ss[t]) : fmaf(f[j] * f[j], inv_d, ss[t]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t < T) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t) red[warp][t] = ss[t];
    }
    __syncthreads();
    if (threadIdx.x < T) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red[w][threadIdx.x];
      rstd_s[threadIdx.x] = MODE == 0 ? rsqrtf(s * inv_d + eps) : 1.0f / sqrtf(s + eps);
    }
    __syncthreads();
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float g[8];
      if (gamma != nullptr) unpack8(__ldg(gamma + v), g);
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t) {
        if (t >= T) break;
        float f[8];
        unpack8(__ldg(x + static_cast<int64_t>(t) * nvec + v), f);
        const float r = rstd_s[t];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], r);
        if (gamma != nullptr) {
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], g[j]);
        }
        a_s[t * nvec + v] = make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
      }
    }
  }
  __syncthreads();
  // 2. weight rows, one warp each
  bool first = true;
  for (int n = n_first; n < N; n += stride) {
    const uint4* wr = W + static_cast<int64_t>(n) * nvec;
    float acc[kMaxTokens];
#pragma unroll
    for (int t = 0; t < kMaxTokens; ++t) acc[t] = 0.f;
    int v = lane;
    for (; v + 32 * (kInFlight - 1) < nvec; v += 32 * kInFlight) {  // kInFlight loads in flight per lane
      uint4 w4[kInFlight];
      if (first) {
#pragma unroll
        for (int i = 0; i < kInFlight; ++i) w4[i] = w_first[i];
        first = false;
      } else {
#pragma unroll
        for (int i = 0; i < kInFlight; ++i) w4[i] = __ldcs(wr + v + 32 * i);  // read once: do not keep in L2
      }
#pragma unroll
      for (int i = 0; i < kInFlight; ++i) {
        float w[8];
        unpack8(w4[i], w);
#pragma unroll
        for (int t = 0; t < kMaxTokens; ++t) {
          if (t >= T) break;
          float a[8];
          unpack8(a_s[t * nvec + v + 32 * i], a);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[t] = fmaf(a[j], w[j], acc[t]);
        }
      }
    }
    first = false;  // a row shorter than kInFlight vectors a lane: the tail loop reloads
    for (; v < nvec; v += 32) {
      float w[8];
      unpack8(__ldcs(wr + v), w);
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t) {
        if (t >= T) break;
        float a[8];
        unpack8(a_s[t * nvec + v], a);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[t] = fmaf(a[j], w[j], acc[t]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t < T) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
#pragma unroll
    for (int t = 0; t < kMaxTokens; ++t)
      if (t < T && lane == t) out[static_cast<int64_t>(t) * N + n] = __float2bfloat16_rn(acc[t]);
  }
}

}  // namespace

// Up to 4 tokens: at 8 the FP32 dot products on the CUDA cores measured
// slower than the tensor-core path (40 against 25 us through the qkv weight),
// and rows of at least 2048 elements (at 1536 many short rows measured
// slightly slower: 26.3 against 25.0 us for 1 x 1536 -> 24576).
bool decode_fits(int64_t T, int64_t K, int64_t N) {
  return T >= 1 && T <= 4 && K >= 2048 && N >= 1024 && T * K * 2 <= kSmemMax;
}

rnl_status launch_decode(const void* x, const void* gamma, const void* W, int64_t T, int64_t K,
                         int64_t N, float eps, int mode, void* out, int sm_count, cudaStream_t s) {
  static bool attr_set[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RNL_ERR_DEVICE;
  const int nvec = static_cast<int>(K / 8);
  const size_t smem = static_cast<size_t>(T) * K * 2;
  auto kern = mode == RNL_NORM_RSQRT ? decode_kernel<0> : decode_kernel<1>;
  const int mi = mode == RNL_NORM_RSQRT ? 0 : 1;
  if (smem > 48 * 1024 && !attr_set[dev][mi]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax) != cudaSuccess)
      return RNL_ERR_LAUNCH;
    attr_set[dev][mi] = true;
  }
  // every warp the same number of weight rows, all CTAs resident at once
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int64_t warps = static_cast<int64_t>(per_sm) * sm_count * kWarps;
  const int64_t rows_per_warp = (N + warps - 1) / warps;
  const int64_t grid = (N + kWarps * rows_per_warp - 1) / (kWarps * rows_per_warp);
  trace_before(s);
  kern<<<static_cast<unsigned>(grid), kWarps * 32, smem, s>>>(
      static_cast<const uint4*>(x), static_cast<const uint4*>(gamma), static_cast<const uint4*>(W),
      static_cast<int>(T), nvec, static_cast<int>(N), static_cast<float>(1.0 / static_cast<double>(K)), eps,
      static_cast<__nv_bfloat16*>(out));
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "decode_gemv");
  return st;
}

}  // namespace rnl
