// qmrs.cu -- operand preparation for QuantMatMulReduceSum (SK-14 skeleton
// page, variant A): the page's x2 is an int8 [B, K, N] matrix with N
// contiguous (ND), while the tcgen05 GEMM reads its B operand K-major, so x2
// is transposed while it is widened to bf16 (exact for integers of up to 8
// bits); the bf16 x2_scale is widened to fp32 once for the epilogue.
#include <cuda_bf16.h>

#include "internal.h"

namespace rnl {
namespace {

constexpr int kTile = 64;  // 64 x 64 int8 tile per block

// Block (nb, kb, b): reads x2[b, k0 .. k0+63, n0 .. n0+63] with 16-byte loads
// along N into shared memory, writes dst[b, n0 .. n0+63, k0 .. k0+63] as bf16
// with 16-byte stores along K.  K % 16 == 0 and N % 16 == 0, so every 16-byte
// segment is either wholly inside the matrix or wholly outside.
__global__ void __launch_bounds__(256)
    s8_transpose_widen_kernel(const int8_t* __restrict__ src, int64_t K, int64_t N,
                              uint4* __restrict__ dst) {
  __shared__ uint32_t tile[kTile][kTile / 4 + 1];  // [k][n / 4], one word of padding per row
  const int64_t b = blockIdx.z;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * kTile;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int8_t* s = src + b * K * N;
  {
    const int r = threadIdx.x >> 2;           // k within the tile
    const int seg = (threadIdx.x & 3) * 16;   // n within the tile
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + r < K && n0 + seg < N) u = __ldg(reinterpret_cast<const uint4*>(s + (k0 + r) * N + n0 + seg));
    tile[r][seg / 4 + 0] = u.x;
    tile[r][seg / 4 + 1] = u.y;
    tile[r][seg / 4 + 2] = u.z;
    tile[r][seg / 4 + 3] = u.w;
  }
  __syncthreads();
  const int nn = threadIdx.x >> 2;            // n within the tile (output row)
  const int kseg = (threadIdx.x & 3) * 16;    // k within the tile
  if (n0 + nn >= N || k0 + kseg >= K) return;
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const uint32_t w0 = tile[kseg + j][nn / 4];
    const uint32_t w1 = tile[kseg + j + 1][nn / 4];
    const int sh = (nn & 3) * 8;
    const float a = static_cast<float>(static_cast<int8_t>((w0 >> sh) & 0xFFu));
    const float c = static_cast<float>(static_cast<int8_t>((w1 >> sh) & 0xFFu));
    __nv_bfloat162 h = __floats2bfloat162_rn(a, c);
    o[j / 2] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint4* d = dst + ((b * N + n0 + nn) * K + k0 + kseg) / 8;
  d[0] = make_uint4(o[0], o[1], o[2], o[3]);
  d[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void __launch_bounds__(256)
    bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ src, int64_t n, float* __restrict__ dst) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = __bfloat162float(src[i]);
}

}  // namespace

rnl_status launch_s8_transpose_widen(const int8_t* src, int64_t B, int64_t K, int64_t N, void* dst,
                                     cudaStream_t s) {
  if (B == 0 || K == 0 || N == 0) return RNL_OK;
  const dim3 grid(static_cast<unsigned>((N + kTile - 1) / kTile),
                  static_cast<unsigned>((K + kTile - 1) / kTile), static_cast<unsigned>(B));
  trace_before(s);
  s8_transpose_widen_kernel<<<grid, 256, 0, s>>>(src, K, N, static_cast<uint4*>(dst));
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "s8_transpose_widen");
  return st;
}

rnl_status launch_bf16_to_f32(const void* src, int64_t n, float* dst, cudaStream_t s) {
  if (n == 0) return RNL_OK;
  trace_before(s);
  bf16_to_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(src), n, dst);
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "bf16_to_f32");
  return st;
}

}  // namespace rnl
