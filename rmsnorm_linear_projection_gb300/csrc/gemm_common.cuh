// gemm_common.cuh -- pieces shared by the one-CTA (gemm_tc.cu) and CTA-pair
// (gemm_pair.cu) tcgen05 GEMM kernels: tile geometry, tile order and the
// epilogue stores of one thread's 32 consecutive output columns.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace rnl {
namespace gemm {

constexpr int BM = 128;     // rows of A per CTA (and TMEM lanes)
constexpr int BK = 64;      // 64 bf16 = one 128-byte swizzle row
constexpr uint32_t kABytes = BM * BK * 2;
constexpr int kChunkKBlocks = 16;       // 1024 products per exact integer chunk
constexpr int kMaxStages = 8;
constexpr size_t kSmemLimit = 232448;   // 227 KB opt-in shared memory per block
constexpr uint32_t kAccStride = 256;    // TMEM column offset between the two accumulators
constexpr int kThreads = 320;           // producer + MMA + 8 epilogue warps (or 4 + 4 transform)

// Tile order: groups of G row blocks, row block fastest within a group column,
// so the CTAs running at the same time share A panels and B panels in L2.  G
// is chosen on the host: all row blocks when A fits comfortably in L2 (then
// every B panel is fetched from HBM once), else 8.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int G, int& mb,
                                            int& nb) {
  const int group_tiles = G * num_n;
  const int group = tile / group_tiles;
  const int first_m = group * G;
  const int gm = min(num_m - first_m, G);
  const int r = tile - group * group_tiles;
  mb = first_m + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 256-bit global store / load (one full 32-byte sector per thread); p must
// be 32-byte aligned.  The load is a plain (coherent) load.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void ld_global_v8(const void* p, uint32_t (&v)[8]) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "l"(p)
               : "memory");
}

// Whether a thread's 32 consecutive outputs of row m starting at column n0
// (a multiple of 32) can go out as 32-byte stores: the row pitch and the base
// are multiples of 32 bytes.
__device__ __forceinline__ bool rows_32b_aligned(const void* out, int N, int elem_bytes) {
  return ((static_cast<int64_t>(N) * elem_bytes) & 31) == 0 &&
         (reinterpret_cast<uintptr_t>(out) & 31) == 0;
}

// out[m, n0 .. n0+31] = bf16(v), v given as fp32 bit patterns (TMEM words).
// Each thread writes its own row, so full 32-byte sectors (256-bit stores)
// halve the number of memory transactions against 16-byte stores.
__device__ __forceinline__ void store_bf16_32(void* out, int64_t m, int n0, int N,
                                              const uint32_t (&r)[32]) {
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(out) + m * N;
  if (n0 + 32 <= N && rows_32b_aligned(out, N, 2)) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        o[i] = bf16x2_bits(__uint_as_float(r[16 * h + 2 * i]), __uint_as_float(r[16 * h + 2 * i + 1]));
      st_global_v8(orow + n0 + 16 * h, o);
    }
  } else if (n0 + 32 <= N && (N & 7) == 0) {
    uint4* dst = reinterpret_cast<uint4*>(orow + n0);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dst[j] = make_uint4(bf16x2_bits(__uint_as_float(r[8 * j]), __uint_as_float(r[8 * j + 1])),
                          bf16x2_bits(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                          bf16x2_bits(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                          bf16x2_bits(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n0 + j < N) orow[n0 + j] = __float2bfloat16_rn(__uint_as_float(r[j]));
  }
}

// out[m, n0 .. n0+31] = bf16(v + bias[n]) (AT-09 has_bias; bias bf16 [N],
// 16-byte aligned; n0 is a multiple of 32).  Each 16-byte chunk of the bias
// is loaded next to the 8 outputs it feeds, so few registers stay live.
__device__ __forceinline__ void store_bf16_bias_32(void* out, int64_t m, int n0, int N,
                                                   const uint32_t (&r)[32],
                                                   const __nv_bfloat16* __restrict__ bias) {
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(out) + m * N;
  if (n0 + 32 <= N && rows_32b_aligned(out, N, 2)) {
    const uint4* b = reinterpret_cast<const uint4*>(bias + n0);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t o[8];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 u = __ldg(b + 2 * h + q);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = 16 * h + 8 * q + 2 * i;
          o[4 * q + i] = bf16x2_bits(__fadd_rn(__uint_as_float(r[k]), __uint_as_float(w[i] << 16)),
                                     __fadd_rn(__uint_as_float(r[k + 1]), __uint_as_float(w[i] & 0xFFFF0000u)));
        }
      }
      st_global_v8(orow + n0 + 16 * h, o);
    }
  } else if (n0 + 32 <= N && (N & 7) == 0) {
    uint4* dst = reinterpret_cast<uint4*>(orow + n0);
    const uint4* b = reinterpret_cast<const uint4*>(bias + n0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 u = __ldg(b + j);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = bf16x2_bits(__fadd_rn(__uint_as_float(r[8 * j + 2 * i]), __uint_as_float(w[i] << 16)),
                           __fadd_rn(__uint_as_float(r[8 * j + 2 * i + 1]), __uint_as_float(w[i] & 0xFFFF0000u)));
      dst[j] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n0 + j < N)
        orow[n0 + j] = __float2bfloat16_rn(__fadd_rn(__uint_as_float(r[j]), __bfloat162float(bias[n0 + j])));
  }
}

// out[m, n0 .. n0+31] = fp32(v) * rs.
__device__ __forceinline__ void store_f32_scaled_32(void* out, int64_t m, int n0, int N,
                                                    const uint32_t (&r)[32], float rs) {
  float* orow = static_cast<float*>(out) + m * N;
  if (n0 + 32 <= N && rows_32b_aligned(out, N, 4)) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__uint_as_float(r[8 * h + i]) * rs);
      st_global_v8(orow + n0 + 8 * h, o);
    }
  } else if (n0 + 32 <= N && (N & 3) == 0) {
    float4* dst = reinterpret_cast<float4*>(orow + n0);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      dst[j] = make_float4(__uint_as_float(r[4 * j]) * rs, __uint_as_float(r[4 * j + 1]) * rs,
                           __uint_as_float(r[4 * j + 2]) * rs, __uint_as_float(r[4 * j + 3]) * rs);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n0 + j < N) orow[n0 + j] = __uint_as_float(r[j]) * rs;
  }
}

// out[m, n0 .. n0+31] = the exact int32 sums.
__device__ __forceinline__ void store_i32_32(void* out, int64_t m, int n0, int N,
                                             const int (&a)[32]) {
  int* orow = static_cast<int*>(out) + m * N;
  if (n0 + 32 <= N && (N & 3) == 0) {
    int4* dst = reinterpret_cast<int4*>(orow + n0);
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = make_int4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n0 + j < N) orow[n0 + j] = a[j];
  }
}

// AT-06 dequant in the order of the SK-14 skeleton page (QuantMatMulReduceSum):
// float(acc) * (x_scale[m] * w_scale[n]) (+ bias[n] when given), then bf16.
__device__ __forceinline__ void store_dequant_32(void* out, int64_t m, int n0, int N,
                                                 const int (&a)[32], float xs,
                                                 const float* __restrict__ w_scale,
                                                 const __nv_bfloat16* __restrict__ bias) {
  uint32_t v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int n = n0 + j;
    const float ws = n < N ? __ldg(w_scale + n) : 0.f;
    v[j] = __float_as_uint(static_cast<float>(a[j]) * (xs * ws));
  }
  if (bias != nullptr)
    store_bf16_bias_32(out, m, n0, N, v, bias);
  else
    store_bf16_32(out, m, n0, N, v);
}

// The same dequant of an accumulator that holds the exact integer sum as a
// binary32 value (|sum| < 2^24): float(acc) is then acc itself, so the
// output is the one store_dequant_32 writes for that integer.
__device__ __forceinline__ void store_dequant_f32_32(void* out, int64_t m, int n0, int N,
                                                     const uint32_t (&r)[32], float xs,
                                                     const float* __restrict__ w_scale,
                                                     const __nv_bfloat16* __restrict__ bias) {
  uint32_t v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int n = n0 + j;
    const float ws = n < N ? __ldg(w_scale + n) : 0.f;
    v[j] = __float_as_uint(__uint_as_float(r[j]) * (xs * ws));
  }
  if (bias != nullptr)
    store_bf16_bias_32(out, m, n0, N, v, bias);
  else
    store_bf16_32(out, m, n0, N, v);
}

// QuantMatMulReduceSum epilogue of one batch (SK-14 skeleton page, variant A)
// for outputs [m, n0 .. n0+31]: v = fp32(acc) * (x1_scale * x2_scale), each a
// correctly rounded FP32 operation; mode bit 0: v = acc_buf[m, n] + v (the
// earlier batches' FP32 sum); bit 1: write bf16(v) to out_final (last batch),
// else v to acc_buf.  The first batch adds nothing (0 + v, so -0 becomes +0 as
// in a sum that starts at zero).
__device__ __forceinline__ void store_dequant_acc_32(float* acc_buf, __nv_bfloat16* out_final,
                                                     int64_t m, int n0, int N, const int (&a)[32],
                                                     float xs, const float* __restrict__ w_scale,
                                                     int mode) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int n = n0 + j;
    const float ws = n < N ? __ldg(w_scale + n) : 0.f;
    v[j] = __fmul_rn(__int2float_rn(a[j]), __fmul_rn(xs, ws));
  }
  float* arow = acc_buf + m * N;
  const bool full = n0 + 32 <= N;
  if (mode & 1) {
    if (full && rows_32b_aligned(acc_buf, N, 4)) {
      uint32_t p[4][8];  // all four loads in flight before the first use
#pragma unroll
      for (int h = 0; h < 4; ++h) ld_global_v8(arow + n0 + 8 * h, p[h]);
#pragma unroll
      for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[8 * h + i] = __fadd_rn(__uint_as_float(p[h][i]), v[8 * h + i]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < N) v[j] = __fadd_rn(arow[n0 + j], v[j]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __fadd_rn(0.0f, v[j]);
  }
  if (mode & 2) {
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
    store_bf16_32(out_final, m, n0, N, r);
  } else if (full && rows_32b_aligned(acc_buf, N, 4)) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t p[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = __float_as_uint(v[8 * h + i]);
      st_global_v8(arow + n0 + 8 * h, p);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n0 + j < N) arow[n0 + j] = v[j];
  }
}

}  // namespace gemm
}  // namespace rnl
