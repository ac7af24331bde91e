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
// n columns of a transpose tile: whole 128-byte lines of each k row (at
// B = 4, M = 2048, K = N = 4096 the operand kernel measured 57.3 us against
// 59.7 us with 64 columns, and 57.7 us with 256)
constexpr int kTN = 128;
constexpr int kThreadsT = 256;
constexpr int kVecPerRow = kTN / 16;                 // 16-byte loads per k row
constexpr int kRowsPerPass = kThreadsT / kVecPerRow;  // k rows loaded per pass
constexpr int kThreadsPerN = kThreadsT / kTN;        // threads per output row
constexpr int kKPerThread = kTK / kThreadsPerN;      // k values each thread writes

// Transpose tile `t` (b, k tile, n tile; n fastest): reads x2[b, k0 .. k0+127,
// n0 .. n0+kTN-1] with 16-byte loads along N, writes dst[b, n0 .., k0 .. k0+127]
// as bf16 with 32-byte stores along K (full sectors).  The tile's rows are
// padded by one word, so the lanes' stores into it fall on distinct banks, and
// the 32 lanes reading one k row back read 8 distinct words.  K % 16 == 0 and
// N % 16 == 0, so every 16-byte load and every 32-byte store segment is either
// wholly inside the matrix or wholly outside.
__device__ __forceinline__ void transpose_tile(int64_t t, const int8_t* __restrict__ src, int64_t K,
                                               int64_t N, uint32_t* __restrict__ dst,
                                               uint32_t (*tile)[kTN / 4 + 1]) {
  const int64_t tiles_n = (N + kTN - 1) / kTN, tiles_k = (K + kTK - 1) / kTK;
  const int64_t b = t / (tiles_n * tiles_k);
  const int64_t r = t - b * tiles_n * tiles_k;
  const int64_t k0 = (r / tiles_n) * kTK, n0 = (r % tiles_n) * kTN;
  const int8_t* s = src + b * K * N;
  uint4 u[kTK / kRowsPerPass];
#pragma unroll
  for (int h = 0; h < kTK / kRowsPerPass; ++h) {
    const int row = threadIdx.x / kVecPerRow + kRowsPerPass * h;  // k within the tile
    const int seg = (threadIdx.x % kVecPerRow) * 16;               // n within the tile
    u[h] = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + row < K && n0 + seg < N) u[h] = __ldg(reinterpret_cast<const uint4*>(s + (k0 + row) * N + n0 + seg));
  }
#pragma unroll
  for (int h = 0; h < kTK / kRowsPerPass; ++h) {
    const int row = threadIdx.x / kVecPerRow + kRowsPerPass * h;
    const int seg = (threadIdx.x % kVecPerRow) * 16;
    tile[row][seg / 4 + 0] = u[h].x;
    tile[row][seg / 4 + 1] = u[h].y;
    tile[row][seg / 4 + 2] = u[h].z;
    tile[row][seg / 4 + 3] = u[h].w;
  }
  __syncthreads();
  const int nn = threadIdx.x % kTN;                  // output row (n) within the tile
  const int kseg = (threadIdx.x / kTN) * kKPerThread;  // kKPerThread k values
  if (n0 + nn < N && k0 + kseg < K) {
    const int sh = (nn & 3) * 8;
    uint32_t* d = dst + ((b * N + n0 + nn) * K + k0 + kseg) / 2;
#pragma unroll
    for (int q = 0; q < kKPerThread / 16; ++q) {
      if (k0 + kseg + 16 * q >= K) break;
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const int kk = kseg + 16 * q + j;
        const float a = static_cast<float>(static_cast<int8_t>((tile[kk][nn / 4] >> sh) & 0xFFu));
        const float c = static_cast<float>(static_cast<int8_t>((tile[kk + 1][nn / 4] >> sh) & 0xFFu));
        __nv_bfloat162 p = __floats2bfloat162_rn(a, c);
        o[j / 2] = *reinterpret_cast<uint32_t*>(&p);
      }
      gemm::st_global_v8(d + 8 * q, o);
    }
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
