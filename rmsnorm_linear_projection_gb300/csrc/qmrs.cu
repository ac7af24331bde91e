// qmrs.cu -- operand preparation for QuantMatMulReduceSum (SK-14 skeleton
// page, variant A): the page's x2 is an int8 [B, K, N] matrix with N
// contiguous (ND), while the tcgen05 GEMM reads its B operand K-major, so x2
// is transposed while it is widened to bf16 (exact for integers of up to 8
// bits); x1 [B, M, K] is widened in place order; the bf16 x2_scale is widened
// to fp32 once for the epilogue.  All three in one launch (their blocks share
// no data), every part HBM bound.
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "internal.h"
#include "widen.cuh"

namespace rnl {
namespace {

constexpr int kTK = 128;  // k rows of a transpose tile
constexpr int kTN = 64;   // n columns of a transpose tile

// Transpose tile `t` (b, k tile, n tile; n fastest): reads x2[b, k0 .. k0+127,
// n0 .. n0+63] with two 16-byte loads per thread along N, writes
// dst[b, n0 .. n0+63, k0 .. k0+127] as bf16 with two 32-byte stores per
// thread along K (full sectors).  The 32 lanes of a warp read 32 consecutive
// columns of one k range from shared memory (8 distinct words: no bank
// conflicts).  K % 16 == 0 and N % 16 == 0, so every 16-byte load and every
// 32-byte store segment is either wholly inside the matrix or wholly outside.
__device__ __forceinline__ void transpose_tile(int64_t t, const int8_t* __restrict__ src, int64_t K,
                                               int64_t N, uint32_t* __restrict__ dst,
                                               uint32_t (*tile)[kTN / 4 + 1]) {
  const int64_t tiles_n = (N + kTN - 1) / kTN, tiles_k = (K + kTK - 1) / kTK;
  const int64_t b = t / (tiles_n * tiles_k);
  const int64_t r = t - b * tiles_n * tiles_k;
  const int64_t k0 = (r / tiles_n) * kTK, n0 = (r % tiles_n) * kTN;
  const int8_t* s = src + b * K * N;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = (threadIdx.x >> 2) + 64 * h;  // k within the tile
    const int seg = (threadIdx.x & 3) * 16;       // n within the tile
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + row < K && n0 + seg < N) u = __ldg(reinterpret_cast<const uint4*>(s + (k0 + row) * N + n0 + seg));
    tile[row][seg / 4 + 0] = u.x;
    tile[row][seg / 4 + 1] = u.y;
    tile[row][seg / 4 + 2] = u.z;
    tile[row][seg / 4 + 3] = u.w;
  }
  __syncthreads();
  const int nn = threadIdx.x & 63;           // output row (n) within the tile
  const int kseg = (threadIdx.x >> 6) * 32;  // 32 k values
  if (n0 + nn < N && k0 + kseg < K) {
    const int sh = (nn & 3) * 8;
    uint32_t o[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float a = static_cast<float>(static_cast<int8_t>((tile[kseg + j][nn / 4] >> sh) & 0xFFu));
      const float c = static_cast<float>(static_cast<int8_t>((tile[kseg + j + 1][nn / 4] >> sh) & 0xFFu));
      __nv_bfloat162 p = __floats2bfloat162_rn(a, c);
      o[j / 2] = *reinterpret_cast<uint32_t*>(&p);
    }
    uint32_t* d = dst + ((b * N + n0 + nn) * K + k0 + kseg) / 2;
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lo[i] = o[i];
      hi[i] = o[8 + i];
    }
    gemm::st_global_v8(d, lo);
    if (k0 + kseg + 16 < K) gemm::st_global_v8(d + 8, hi);
  }
}

struct PrepArgs {
  const int8_t* x2;
  int64_t K, N;
  uint32_t* x2_dst;
  unsigned transpose_blocks;
  const uint4* x1;
  int64_t x1_nvec16;
  uint4* x1_dst;
  unsigned widen_blocks;
  const __nv_bfloat16* scale;
  int64_t scale_n;
  float* scale_dst;
};

__global__ void __launch_bounds__(256) qmrs_prep_kernel(PrepArgs p) {
  __shared__ uint32_t tile[kTK][kTN / 4 + 1];  // [k][n / 4], one word of padding per row
  const unsigned b = blockIdx.x;
  if (b < p.transpose_blocks) {
    transpose_tile(b, p.x2, p.K, p.N, p.x2_dst, tile);
  } else if (b < p.transpose_blocks + p.widen_blocks) {
    widen_block(b - p.transpose_blocks, p.x1, p.x1_nvec16, p.x1_dst);
  } else {
    const int64_t i = static_cast<int64_t>(b - p.transpose_blocks - p.widen_blocks) * blockDim.x + threadIdx.x;
    if (i < p.scale_n) p.scale_dst[i] = __bfloat162float(p.scale[i]);
  }
}

}  // namespace

rnl_status launch_qmrs_prep(const int8_t* x1, const int8_t* x2, const void* x2_scale, int64_t B,
                            int64_t M, int64_t K, int64_t N, void* x1_dst, void* x2_dst,
                            float* scale_dst, cudaStream_t s) {
  PrepArgs p;
  p.x2 = x2;
  p.K = K;
  p.N = N;
  p.x2_dst = static_cast<uint32_t*>(x2_dst);
  p.transpose_blocks = static_cast<unsigned>(B * ((K + kTK - 1) / kTK) * ((N + kTN - 1) / kTN));
  p.x1 = reinterpret_cast<const uint4*>(x1);
  p.x1_nvec16 = B * M * K / 16;
  p.x1_dst = static_cast<uint4*>(x1_dst);
  p.widen_blocks = static_cast<unsigned>((p.x1_nvec16 + 256 * kS8Vec - 1) / (256 * kS8Vec));
  p.scale = static_cast<const __nv_bfloat16*>(x2_scale);
  p.scale_n = N;
  p.scale_dst = scale_dst;
  const unsigned scale_blocks = static_cast<unsigned>((N + 255) / 256);
  const unsigned grid = p.transpose_blocks + p.widen_blocks + scale_blocks;
  if (grid == 0) return RNL_OK;
  trace_before(s);
  qmrs_prep_kernel<<<grid, 256, 0, s>>>(p);
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "qmrs_prep");
  return st;
}

}  // namespace rnl
