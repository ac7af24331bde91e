// widen.cuh -- int8 -> bf16 widening of operands for the exact integer GEMM
// (every int8 value is exact in bf16, which has 8 significant bits).
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace rnl {

// 16 int8 values -> 16 bf16 values (two 16-byte vectors).
__device__ __forceinline__ void widen16(const uint4& u, uint4* dst) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float a = static_cast<float>(static_cast<int8_t>(w[k] & 0xFF));
    const float b = static_cast<float>(static_cast<int8_t>((w[k] >> 8) & 0xFF));
    const float c = static_cast<float>(static_cast<int8_t>((w[k] >> 16) & 0xFF));
    const float d = static_cast<float>(static_cast<int8_t>((w[k] >> 24) & 0xFF));
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    o[2 * k] = *reinterpret_cast<uint32_t*>(&lo);
    o[2 * k + 1] = *reinterpret_cast<uint32_t*>(&hi);
  }
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Each thread of a block widens kS8Vec x 16 elements (16-byte vectors v =
// block * blockDim * kS8Vec + threadIdx + i * blockDim), issuing all its loads
// before converting.
constexpr int kS8Vec = 4;

__device__ __forceinline__ void widen_block(unsigned block, const uint4* __restrict__ src,
                                            int64_t nvec16, uint4* __restrict__ dst) {
  const int64_t base = (static_cast<int64_t>(block) * blockDim.x) * kS8Vec + threadIdx.x;
  uint4 u[kS8Vec];
#pragma unroll
  for (int i = 0; i < kS8Vec; ++i) {
    const int64_t v = base + static_cast<int64_t>(i) * blockDim.x;
    u[i] = v < nvec16 ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < kS8Vec; ++i) {
    const int64_t v = base + static_cast<int64_t>(i) * blockDim.x;
    if (v < nvec16) widen16(u[i], dst + 2 * v);
  }
}

}  // namespace rnl
