// headnorm.cu -- per-head RMSNorm of a projection output: the MLA chain's
// second norm (AT-10 pattern page, sec. 9, the golden chain of the MLA
// prolog test: q_b_proj reshaped to [num_heads, head_dim], then RMSNorm
// again), each head row of D values normalised on its own:
//
//   y [T, H * D] bf16;  per head row h of a token:
//   rstd = rsqrt(mean(h^2) + eps)  |  1 / sqrt(mean(h^2) + eps)   (FP32, the two forms)
//   z    = bf16((h * rstd) * gamma)                              (gamma [D] optional)
//
// One warp per (token, group of heads).  A head row is D / 2 32-bit words;
// lane l holds words l, l + 32, l + 64, ..., so every load and store
// instruction of the warp covers 128 contiguous bytes.  All heads of the
// group are loaded before any is processed.  The output may be the input
// itself (each lane reads its words before it writes them), so no load goes
// through the read-only path.
#include <cuda_bf16.h>

#include "internal.h"

namespace rnl {
namespace {

constexpr int kWarps = 8;  // warps per block

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// W = D / 64 words per lane, HPW heads per warp.
template <int MODE, int W, int HPW>
__global__ void __launch_bounds__(kWarps * 32)
    head_norm_kernel(const uint32_t* y, int64_t T, int H, int groups, const uint32_t* gamma,
                     float inv_d, float eps, uint32_t* out) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (wid >= T * groups) return;
  const int64_t t = wid / groups;
  const int h0 = static_cast<int>(wid - t * groups) * HPW;
  const int nh = H - h0 < HPW ? H - h0 : HPW;
  constexpr int kWordsPerHead = 32 * W;
  const int64_t row0 = (t * H + h0) * static_cast<int64_t>(kWordsPerHead);
  uint32_t u[HPW][W];
#pragma unroll
  for (int j = 0; j < HPW; ++j)
    if (j < nh) {
#pragma unroll
      for (int w = 0; w < W; ++w) u[j][w] = y[row0 + j * kWordsPerHead + lane + 32 * w];
    }
  float g[2 * W];
  if (gamma != nullptr) {
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const uint32_t gw = __ldg(gamma + lane + 32 * w);
      g[2 * w] = __uint_as_float(gw << 16);
      g[2 * w + 1] = __uint_as_float(gw & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int j = 0; j < HPW; ++j) {
    if (j >= nh) break;
    float f[2 * W];
#pragma unroll
    for (int w = 0; w < W; ++w) {
      f[2 * w] = __uint_as_float(u[j][w] << 16);
      f[2 * w + 1] = __uint_as_float(u[j][w] & 0xFFFF0000u);
    }
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 2 * W; ++e) s = MODE == 0 ? fmaf(f[e], f[e], s) : fmaf(f[e] * f[e], inv_d, s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float r = MODE == 0 ? rsqrtf(s * inv_d + eps) : __fdiv_rn(1.0f, __fsqrt_rn(s + eps));
#pragma unroll
    for (int e = 0; e < 2 * W; ++e) {
      f[e] = __fmul_rn(f[e], r);
      if (gamma != nullptr) f[e] = __fmul_rn(f[e], g[e]);
    }
#pragma unroll
    for (int w = 0; w < W; ++w) out[row0 + j * kWordsPerHead + lane + 32 * w] = pack2(f[2 * w], f[2 * w + 1]);
  }
}

template <int MODE, int W>
void launch_w(unsigned blocks, const uint32_t* y, int64_t T, int H, const uint32_t* g, float inv_d,
              float eps, uint32_t* out, cudaStream_t s) {
  constexpr int kHpw = W <= 4 ? 8 : 4;
  const int groups = (H + kHpw - 1) / kHpw;
  head_norm_kernel<MODE, W, kHpw><<<blocks, kWarps * 32, 0, s>>>(y, T, H, groups, g, inv_d, eps, out);
}

template <int MODE>
void launch_mode(int W, unsigned blocks, const uint32_t* y, int64_t T, int H, const uint32_t* g,
                 float inv_d, float eps, uint32_t* out, cudaStream_t s) {
  switch (W) {
    case 1: launch_w<MODE, 1>(blocks, y, T, H, g, inv_d, eps, out, s); break;
    case 2: launch_w<MODE, 2>(blocks, y, T, H, g, inv_d, eps, out, s); break;
    case 3: launch_w<MODE, 3>(blocks, y, T, H, g, inv_d, eps, out, s); break;
    case 4: launch_w<MODE, 4>(blocks, y, T, H, g, inv_d, eps, out, s); break;
    case 5: launch_w<MODE, 5>(blocks, y, T, H, g, inv_d, eps, out, s); break;
    case 6: launch_w<MODE, 6>(blocks, y, T, H, g, inv_d, eps, out, s); break;
    case 7: launch_w<MODE, 7>(blocks, y, T, H, g, inv_d, eps, out, s); break;
    default: launch_w<MODE, 8>(blocks, y, T, H, g, inv_d, eps, out, s); break;
  }
}

}  // namespace

bool head_norm_dim_ok(int64_t D) { return D >= 64 && D <= 512 && D % 64 == 0; }

rnl_status launch_head_norm(const void* y, int64_t T, int64_t H, int64_t D, const void* gamma,
                            float eps, int mode, void* out, cudaStream_t s) {
  if (T * H == 0) return RNL_OK;
  const int W = static_cast<int>(D / 64);
  const int hpw = W <= 4 ? 8 : 4;
  const int64_t warps = T * ((H + hpw - 1) / hpw);
  const unsigned blocks = static_cast<unsigned>((warps + kWarps - 1) / kWarps);
  const auto* yp = static_cast<const uint32_t*>(y);
  const auto* gp = static_cast<const uint32_t*>(gamma);
  auto* op = static_cast<uint32_t*>(out);
  const float inv_d = static_cast<float>(1.0 / static_cast<double>(D));
  trace_before(s);
  if (mode == RNL_NORM_RSQRT)
    launch_mode<0>(W, blocks, yp, T, static_cast<int>(H), gp, inv_d, eps, op, s);
  else
    launch_mode<1>(W, blocks, yp, T, static_cast<int>(H), gp, inv_d, eps, op, s);
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "head_norm");
  return st;
}

}  // namespace rnl
