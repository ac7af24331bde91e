// decode.cu -- the AT-10 RMSNorm + Linear (bf16 out) for a handful of tokens
// (T <= 4, a decode step) against a wide weight.  With so few rows the
// projection is a matrix-vector product bound by reading W once: the
// tensor-core GEMM would use one 128-row tile per weight block and occupy a
// fraction of the SMs (about 1.7 TB/s measured at T = 1 against the qkv
// weight), so this kernel spreads W's rows over every SM instead:
//
//   every CTA normalises the T rows into shared memory (AT-10 pattern page,
//   sec. 3: rstd = rsqrt(mean(x^2) + eps) | 1 / sqrt(...),
//   a = bf16((x rstd) gamma)): one read of x from global memory, the raw rows
//   parked in shared memory and normalised in place, gamma read in the same
//   pass and parked beside them when it fits;
//   each warp then takes units of weight rows, u = w, w + W, ... (W = the
//   warps of the whole grid, which is resident at once; warp w is warp
//   w / grid of CTA w % grid): with R = 2 the first P units are pairs of
//   adjacent rows and the rest single rows, where the host sets P to whole
//   rounds of pairs when single rows for the remainder shorten the longest
//   warp's sequence (at 6144 rows over 2432 warps: one round of pairs and
//   1280 single rows, 6 chunks at most a warp instead of 8), else to all
//   pairs; with R = 1 every unit is a row.  Each warp streams its units as
//   one sequence of chunks (8 16-byte loads per lane: 4 of each row of a
//   pair, 8 of a single row; 4 KB per warp) with the next chunk's loads
//   issued before the current one is used, so that two chunks are in flight
//   per warp across unit boundaries; the first chunk's loads go out once
//   the token norm's first pass has its x and gamma (issued before those
//   loads, or right behind them, the weight's loads held x back and the
//   call measured 13.4-13.7 or 13.0-13.1 us against 12.5-12.7);
//   each normalised 16-byte vector read from shared memory serves the rows
//   of the unit; the dot products accumulate in FP32 with the mixed-precision FMA
//   (bf16 x bf16 + f32, one rounding; the bf16 product is exact) and reduce
//   across the warp: out[t, n] = bf16(sum).
//
// The kernel is launched as a programmatic dependent of the kernel before it
// in the stream, so that its launch overlaps that kernel's last CTAs, and
// waits for it (griddepcontrol.wait) before its first load: x, gamma and W
// may all come from it.  It does not let the next kernel launch early: a
// chain of decode calls measured 1.8 us a call slower when it did.
//
// The summation order differs from the tensor-core path, inside the same
// bf16 output bound.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

constexpr int kMaxTokens = 4;
constexpr int kWarps = 8;
constexpr int kSmemMax = 96 * 1024;  // the normalised rows: T * K * 2 bytes (+ K * 2 for gamma)
constexpr int kChunk = 8;            // 16-byte weight loads per lane per chunk

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

// acc_lo += a.lo * w.lo, acc_hi += a.hi * w.hi on the two bf16 halves of a
// word, each product and sum rounded once to FP32 (the mixed-precision FMA:
// the bf16 product is exact, so this equals widening both operands and an
// FP32 fma).
__device__ __forceinline__ void fma2_bf16(uint32_t a, uint32_t w, float& acc_lo, float& acc_hi) {
  asm("{\n\t.reg .b16 al, ah, wl, wh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {wl, wh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, wl, %0;\n\t"
      "fma.rn.f32.bf16 %1, ah, wh, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(a), "r"(w));
}

// chunk q of the R weight rows from n0: vectors lane + 32 * (q * C + i),
// i < C = kChunk / R, of each row (rows at or past N read as zero)
template <int R>
__device__ __forceinline__ void load_chunk(const uint4* __restrict__ W, int n0, int N, int q, int nvec,
                                           int lane, uint4 (&buf)[kChunk]) {
  constexpr int C = kChunk / R;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint4* wr = W + static_cast<int64_t>(n0 + r) * nvec;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int v = lane + 32 * (q * C + i);
      buf[r * C + i] = (n0 + r < N && v < nvec) ? __ldcs(wr + v)  // read once: do not keep in L2
                                                : make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// the T x R dot products of one chunk (C = kChunk / R vectors per lane of each row)
template <int T, int R>
__device__ __forceinline__ void dot_chunk(const uint4* __restrict__ a_s, const uint4 (&cur)[kChunk], int q,
                                          int nvec, int lane, float (&acc)[2][T], float (&acc2)[2][T]) {
  constexpr int C = kChunk / R;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int v = lane + 32 * (q * C + i);
    if (v < nvec) {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const uint4 a = a_s[t * nvec + v];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint4 w = cur[r * C + i];
          fma2_bf16(a.x, w.x, acc[r][t], acc2[r][t]);
          fma2_bf16(a.y, w.y, acc[r][t], acc2[r][t]);
          fma2_bf16(a.z, w.z, acc[r][t], acc2[r][t]);
          fma2_bf16(a.w, w.w, acc[r][t], acc2[r][t]);
        }
      }
    }
  }
}

// a unit of R rows from n0 is complete: reduce across the warp and store
template <int T, int R>
__device__ __forceinline__ void reduce_store(float (&acc)[2][T], float (&acc2)[2][T], int n0, int N, int lane,
                                             __nv_bfloat16* __restrict__ out) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < T; ++t) {
      acc[r][t] += acc2[r][t];
      acc2[r][t] = 0.f;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < T; ++t) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], o);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int n = n0 + r;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      if (lane == r * T + t && n < N) out[static_cast<int64_t>(t) * N + n] = __float2bfloat16_rn(acc[r][t]);
      acc[r][t] = 0.f;
    }
  }
}

template <int MODE, int T, int R>
__global__ void __launch_bounds__(kWarps * 32, 2)
    decode_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gamma,
                  const uint4* __restrict__ W, int nvec, int N, float inv_d, float eps,
                  int gamma_smem, int P, __nv_bfloat16* __restrict__ out) {
  extern __shared__ uint4 a_s[];  // [T][nvec] rows, then [nvec] gamma when gamma_smem
  uint4* g_s = a_s + T * nvec;
  __shared__ float red[kWarps][kMaxTokens];
  __shared__ float rstd_s[kMaxTokens];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int stride = gridDim.x * kWarps;  // in units
  // units: with R = 2 the first P are pairs of rows (2p, 2p + 1), the rest
  // single rows 2P + s; with R = 1 every unit is a single row
  const int Pp = R == 2 ? P : 0;
  const int S = N - 2 * Pp;
  const int cpr2 = (nvec + 127) / 128, cpr1 = (nvec + 255) / 256;  // chunks per pair / single row
  const int w0 = warp * gridDim.x + blockIdx.x;
  const int kp = w0 < Pp ? (Pp - 1 - w0) / stride + 1 : 0;
  const int ks = w0 < S ? (S - 1 - w0) / stride + 1 : 0;
  const int units = kp + ks;
  auto load = [&](int u, int qq, uint4 (&buf)[kChunk]) {
    if (R == 2 && u < kp)
      load_chunk<2>(W, 2 * (w0 + u * stride), N, qq, nvec, lane, buf);
    else
      load_chunk<1>(W, 2 * Pp + w0 + (u - kp) * stride, N, qq, nvec, lane, buf);
  };
  int u = 0, q = 0;
  grid_dependency_wait();  // x, gamma and W may come from the previous kernel
  uint4 cur[kChunk];

  // 1. the normalised rows: thread i takes vectors i, i + 256, ... of every
  //    row; the raw vectors stay in shared memory for the second pass, which
  //    touches only the thread's own vectors
  {
    float ss[T];
#pragma unroll
    for (int t = 0; t < T; ++t) ss[t] = 0.f;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      uint4 u[T];
#pragma unroll
      for (int t = 0; t < T; ++t) u[t] = __ldg(x + static_cast<int64_t>(t) * nvec + v);
      if (gamma_smem) g_s[v] = __ldg(gamma + v);
#pragma unroll
      for (int t = 0; t < T; ++t) {
        a_s[t * nvec + v] = u[t];
        float f[8];
        unpack8(u[t], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss[t] = MODE == 0 ? fmaf(f[j], f[j], ss[t]) : fmaf(f[j] * f[j], inv_d, ss[t]);
      }
    }
    if (units > 0) load(0, 0, cur);  // the first chunk, behind x and gamma
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int t = 0; t < T; ++t) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < T; ++t) red[warp][t] = ss[t];
    }
    __syncthreads();
    if (threadIdx.x < T) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red[w][threadIdx.x];
      rstd_s[threadIdx.x] = MODE == 0 ? rsqrtf(s * inv_d + eps) : 1.0f / sqrtf(s + eps);
    }
    __syncthreads();
    float r[T];
#pragma unroll
    for (int t = 0; t < T; ++t) r[t] = rstd_s[t];
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float gm[8];
      if (gamma != nullptr) unpack8(gamma_smem ? g_s[v] : __ldg(gamma + v), gm);
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float f[8];
        unpack8(a_s[t * nvec + v], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], r[t]);
        if (gamma != nullptr) {
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], gm[j]);
        }
        a_s[t * nvec + v] = make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
      }
    }
  }
  __syncthreads();

  // 2. the units as one stream of chunks, the next chunk in flight
  float acc[2][T], acc2[2][T];  // even and odd elements
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int t = 0; t < T; ++t) acc[r][t] = acc2[r][t] = 0.f;
  while (u < units) {
    const bool pair = R == 2 && u < kp;
    const int cpr = pair ? cpr2 : cpr1;
    int u2 = u, q2 = q + 1;
    if (q2 == cpr) {
      q2 = 0;
      u2 = u + 1;
    }
    uint4 nxt[kChunk];
    if (u2 < units) load(u2, q2, nxt);
    if (pair) {
      dot_chunk<T, 2>(a_s, cur, q, nvec, lane, acc, acc2);
      if (q == cpr - 1) reduce_store<T, 2>(acc, acc2, 2 * (w0 + u * stride), N, lane, out);
    } else {
      dot_chunk<T, 1>(a_s, cur, q, nvec, lane, acc, acc2);
      if (q == cpr - 1) reduce_store<T, 1>(acc, acc2, 2 * Pp + w0 + (u - kp) * stride, N, lane, out);
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) cur[i] = nxt[i];
    u = u2;
    q = q2;
  }
}

template <int MODE, int R>
void* decode_entry(int64_t T) {
  switch (T) {
    case 1: return reinterpret_cast<void*>(decode_kernel<MODE, 1, R>);
    case 2: return reinterpret_cast<void*>(decode_kernel<MODE, 2, R>);
    case 3: return reinterpret_cast<void*>(decode_kernel<MODE, 3, R>);
    default: return reinterpret_cast<void*>(decode_kernel<MODE, 4, R>);
  }
}

// Units of two rows (pairs, with single rows for a remainder) for 3 or 4
// tokens when the pairs of rows still give every resident warp (two CTAs of
// 8 warps per SM) at least one pair, else single rows throughout.  Measured (GPU time, flushed CUDA graph): 4 x 4096 -> 6144
// 15.4 us with pairs against 16.1 us; 1 and 2 tokens 13.3 and 14.0 us with
// single rows against 13.5 and 14.5 us; 4 x 12288 -> 2048 (1024 pairs for
// 2432 warps) 20.6 us single against 21.1 us.  RNL_DECODE_ROWS=1 or 2
// overrides.
int decode_rows(int64_t T, int64_t N, int sm_count) {
  if (const char* e = std::getenv("RNL_DECODE_ROWS"))
    if (e[0] == '1' || e[0] == '2') return e[0] - '0';
  return T >= 3 && N / 2 >= static_cast<int64_t>(sm_count) * 2 * kWarps ? 2 : 1;
}

}  // namespace

// Up to 4 tokens: at 8 the FP32 dot products on the CUDA cores measured
// slower than the tensor-core path (40 against 25 us through the qkv weight),
// and rows of at least 2048 elements (at 1536 many short rows measured
// slightly slower: 26.3 against 25.0 us for 1 x 1536 -> 24576).
bool decode_fits(int64_t T, int64_t K, int64_t N) {
  return T >= 1 && T <= kMaxTokens && K >= 2048 && N >= 1024 && T * K * 2 <= kSmemMax;
}

rnl_status launch_decode(const void* x, const void* gamma, const void* W, int64_t T, int64_t K,
                         int64_t N, float eps, int mode, void* out, int sm_count, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RNL_ERR_DEVICE;
  if (T < 1 || T > kMaxTokens) return RNL_ERR_SHAPE;
  const int nvec = static_cast<int>(K / 8);
  // gamma beside the rows when it fits the same limit
  const int gamma_smem = gamma != nullptr && (T + 1) * K * 2 <= kSmemMax ? 1 : 0;
  const size_t smem = static_cast<size_t>(T + gamma_smem) * K * 2;
  const int mi = mode == RNL_NORM_RSQRT ? 0 : 1;
  const int R = decode_rows(T, N, sm_count);
  void* kern = R == 1 ? (mi == 0 ? decode_entry<0, 1>(T) : decode_entry<1, 1>(T))
                      : (mi == 0 ? decode_entry<0, 2>(T) : decode_entry<1, 2>(T));
  if (smem > 48 * 1024 && ensure_smem_attr(kern, dev, kSmemMax) != RNL_OK) return RNL_ERR_LAUNCH;
  // the whole grid resident at once, each warp at least one row group
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int64_t groups = (N + R - 1) / R;
  const int64_t grid = std::min<int64_t>(static_cast<int64_t>(per_sm) * sm_count, (groups + kWarps - 1) / kWarps);
  // with pairs of rows: whole rounds of pairs for every warp and the rest as
  // single rows (half the chunks of a pair) when that shortens the longest
  // warp's sequence, else pairs throughout
  const int64_t wt = grid * kWarps;
  int P = 0;
  if (R == 2) {
    const int64_t k = N / (2 * wt), rest = N - 2 * k * wt;
    const int64_t cpr2 = (nvec + 127) / 128, cpr1 = (nvec + 255) / 256;
    const int64_t pairs_max = (groups + wt - 1) / wt * cpr2;
    const int64_t mixed_max = k * cpr2 + (rest + wt - 1) / wt * cpr1;
    P = static_cast<int>(mixed_max < pairs_max ? k * wt : groups);
  }
  const uint4* xp = static_cast<const uint4*>(x);
  const uint4* gp = static_cast<const uint4*>(gamma);
  const uint4* wp = static_cast<const uint4*>(W);
  int nv = nvec, nn = static_cast<int>(N), gs = gamma_smem;
  float inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  __nv_bfloat16* op = static_cast<__nv_bfloat16*>(out);
  void* args[] = {&xp, &gp, &wp, &nv, &nn, &inv_d, &eps, &gs, &P, &op};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_before(s);
  const cudaError_t e = cudaLaunchKernelExC(&cfg, kern, args);
  if (e != cudaSuccess) cudaGetLastError();
  const rnl_status st = e == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "decode_gemv");
  return st;
}

}  // namespace rnl
