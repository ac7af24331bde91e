// quantstream.cu -- the AT-11 quantising front end as a persistent stream:
// RMSNorm of every token row, then per-token symmetric INT8 codes (SK-03
// skeleton page, "quantised variant (AT-11)"; AT-10 pattern page, sec. 4,
// INT8 W8A8 mode):
//   y = (x * rstd) * gamma        FP32, one correctly rounded product each
//   amax = max |y|;  qs = 127 / amax;  q = rint_half_even(y * qs);
//   x_scale = amax / 127          (amax == 0: q = 0, x_scale = 0)
// with the FP32 sum of squares taken as the binary32 rounding of the exact
// sum (float-float accumulation, exactsum.cuh), so the codes are a function
// of the row alone.  The codes go to A [T, K] as exact bf16 integers (the
// integer GEMM's operand), optionally to q_out [T, K] as int8.
//
// Like the streamed norm pass (normstream.cu): one CTA per SM walks its own
// contiguous range of rows in groups of 8; a producer thread bulk-copies each
// row into a shared-memory ring, and 16 consumer warps take the rows into
// registers, two warps per row, half a row each (rows of up to 4096
// elements; 16 warps hide the latency of the reductions and divisions that 8
// register-heavy warps, one per row, did not: 45 us at 8192 x 4096).  The
// pair combines its halves' float-float sums, maxima and checks through
// shared memory in a fixed order, so both warps see the same values.  Two
// passes over the registers:
//   pass 1  the sum of squares (four packed float-float chains, f32x2
//           arithmetic) and the largest |x * gamma| with its position: the
//           product of two bf16 values is exact in FP32 with its low 8
//           fraction bits zero, so the position rides in those bits and one
//           integer maximum finds both;
//   pass 2  y (packed products), the codes (scalar y * qs, rint) and the
//           exact max |y|.
// amax is taken from the element with the largest exact |x * gamma|: rounding
// can only let an element whose exact product is within a few units in the
// last place overtake it, so pass 2 also tracks max |y| and, when that beats
// the first guess (rare), runs again with it.  The amax pass of the three-pass
// form (rowwise.cu) and its re-read of the row are gone.
#include <cuda_bf16.h>

#include "exactsum.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_quant;

constexpr int kGroupRows = 8;  // one row per consumer warp
constexpr int kConsumerWarps = 2 * kGroupRows;  // two warps per row
constexpr int kThreadsQS = (kConsumerWarps + 1) * 32;
constexpr int kMaxQsStages = 16;
constexpr size_t kRingBytes = 200 * 1024;

struct __align__(8) QsCtrl {
  uint64_t full[kMaxQsStages][kGroupRows];  // one barrier per row slot
  uint64_t empty[kMaxQsStages];
  int abort;
};

// ---- two binary32 values in one 64-bit register, packed f32x2 arithmetic.
// ptxas may contract a packed product feeding a packed sum into one packed
// fused multiply-add (one rounding instead of two), so a product whose
// rounding matters and that feeds a sum is taken with the scalar __fmul_rn,
// which is never contracted.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// the two bf16 values of a 32-bit word as binary32 (exact)
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// TwoSum of (hi, t) per half, the error added to lo (one float-float chain per half)
__device__ __forceinline__ void two_sum2(uint64_t& hi, uint64_t& lo, uint64_t t) {
  const uint64_t s = f2_add(hi, t);
  const uint64_t bb = f2_sub(s, hi);
  const uint64_t e = f2_add(f2_sub(hi, f2_sub(s, bb)), f2_sub(t, bb));
  hi = s;
  lo = f2_add(lo, e);
}
// |p| with the element's position in the low 8 bits (zero in an exact bf16 x bf16 product)
__device__ __forceinline__ uint32_t pos_key(float p, uint32_t pos) {
  return (__float_as_uint(p) & 0x7FFFFFFFu) | pos;
}

__device__ __forceinline__ float bf16_at(const uint4& u, int j) {
  const uint32_t w = (j >> 1) == 0 ? u.x : (j >> 1) == 1 ? u.y : (j >> 1) == 2 ? u.z : u.w;
  return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// Pass 2 over this warp's half of the row: y, codes, stores and the exact
// max |y| of this lane (vectors v = hl + 64 i, hl = the lane's index in the row's 64).
template <bool GAMMA, int VPW>
__device__ __forceinline__ float codes_pass(const uint4 (&xv)[VPW], const uint4* gamma_s, int hl,
                                            int nvec, float rstd, float qs, uint4* ar, uint2* qr) {
  const uint64_t r2 = f2(rstd, rstd);
  float ymax = 0.f;
#pragma unroll
  for (int i = 0; i < VPW; ++i) {
    const int v = hl + 64 * i;
    if (v < nvec) {
      const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
      uint32_t gw[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};  // bf16 1.0
      if (GAMMA) {
        const uint4 g = gamma_s[v];
        gw[0] = g.x;
        gw[1] = g.y;
        gw[2] = g.z;
        gw[3] = g.w;
      }
      uint32_t o[4];
      float c[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint64_t y = f2_mul(bf16x2_to_f2(xw[k]), r2);
        if (GAMMA) y = f2_mul(y, bf16x2_to_f2(gw[k]));
        float y0, y1;
        f2_split(y, y0, y1);
        ymax = fmaxf(ymax, fmaxf(fabsf(y0), fabsf(y1)));
        c[2 * k] = rintf(__fmul_rn(y0, qs));
        c[2 * k + 1] = rintf(__fmul_rn(y1, qs));
        __nv_bfloat162 h = __floats2bfloat162_rn(c[2 * k], c[2 * k + 1]);  // small integers: exact
        o[k] = *reinterpret_cast<uint32_t*>(&h);
      }
      ar[v] = make_uint4(o[0], o[1], o[2], o[3]);
      if (qr != nullptr) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          lo |= (static_cast<uint32_t>(__float2int_rn(c[j])) & 0xFFu) << (8 * j);
          hi |= (static_cast<uint32_t>(__float2int_rn(c[4 + j])) & 0xFFu) << (8 * j);
        }
        qr[v] = make_uint2(lo, hi);
      }
    }
  }
  return ymax;
}

// The float-float total of one warp's eight chains (as ff_warp_total, but
// returning hi and lo unrounded so two warps' halves can be added exactly).
__device__ __forceinline__ void ff_warp_pair(const float (&hs)[8], const float (&ls)[8], float& hi_out,
                                             float& lo_out) {
  float hi = hs[0], lo = ls[0];
#pragma unroll
  for (int j = 1; j < 8; ++j) {
    float sum, e;
    two_sum(hi, hs[j], sum, e);
    lo = __fadd_rn(__fadd_rn(lo, ls[j]), e);
    hi = sum;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    float sum, e;
    two_sum(hi, h2, sum, e);
    lo = __fadd_rn(__fadd_rn(lo, l2), e);
    hi = sum;
  }
  hi_out = hi;
  lo_out = lo;
}

// Values the two warps of a row exchange through shared memory (one set per
// group parity, so a fast pair never overwrites what its partner still reads).
struct __align__(16) PairX {
  float hi[2], lo[2];    // each half's float-float sum of squares
  uint32_t kmax[2];      // each half's keyed max of |x * gamma|
  float guess;           // |y| of the keyed maximum
  uint32_t ymax[2][2];   // each half's max |y|, per pass-2 attempt
};

template <int MODE, bool GAMMA, int VPW>
__global__ void __launch_bounds__(kThreadsQS, 1)
    quant_stream_kernel(const uint8_t* x, const uint4* __restrict__ gamma, int64_t T, int nvec,
                        int stages, float inv_d, float eps, uint4* __restrict__ A,
                        uint2* __restrict__ q_out, float* __restrict__ x_scale) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 127u) & ~127u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
  const uint32_t stage_bytes = kGroupRows * row_bytes;
  uint4* gamma_s = reinterpret_cast<uint4*>(smem + static_cast<size_t>(stages) * stage_bytes);
  QsCtrl* ctrl = reinterpret_cast<QsCtrl*>(smem + static_cast<size_t>(stages) * stage_bytes + row_bytes);
  PairX* px = reinterpret_cast<PairX*>(
      (reinterpret_cast<uintptr_t>(ctrl) + sizeof(QsCtrl) + 15) & ~static_cast<uintptr_t>(15));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t r_begin = static_cast<int64_t>(blockIdx.x) * T / gridDim.x;
  const int64_t r_end = static_cast<int64_t>(blockIdx.x + 1) * T / gridDim.x;
  const int64_t groups = (r_end - r_begin + kGroupRows - 1) / kGroupRows;

  grid_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      for (int r = 0; r < kGroupRows; ++r) mbar_init(smem_u32(&ctrl->full[s][r]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), kConsumerWarps);
    }
    ctrl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();  // everything below may touch the previous kernel's data
  volatile int* abort = &ctrl->abort;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (int64_t g = 0; g < groups; ++g) {
        if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_quant, 51)) break;
        const int64_t row0 = r_begin + g * kGroupRows;
        const int rows = static_cast<int>(r_end - row0 < kGroupRows ? r_end - row0 : kGroupRows);
        const uint32_t dst = base + stage * stage_bytes;
        if (!RNL_DCHECK(&g_err_quant, stages <= kMaxQsStages && stage < static_cast<uint32_t>(stages) &&
                                          static_cast<size_t>(stages) * stage_bytes <= kRingBytes &&
                                          row0 >= 0 && row0 + rows <= T, 53))
          break;
        for (int r = 0; r < rows; ++r) {
          const uint32_t bar = smem_u32(&ctrl->full[stage][r]);
          mbar_arrive_expect_tx(bar, row_bytes);
          bulk_copy_g2s(dst + r * row_bytes, x + (row0 + r) * row_bytes, row_bytes, bar);
        }
        if (++stage == static_cast<uint32_t>(stages)) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  // warps 2r and 2r + 1 share row slot r; sub = which half, hl = the lane's
  // index among the row's 64 lanes; named barrier 2 + r joins the pair
  const int slot = warp >> 1, sub = warp & 1, hl = sub * 32 + lane;
  const uint32_t pair_bar = 2u + static_cast<uint32_t>(slot);
  if (GAMMA) {  // gamma staged once in shared memory for all rows
    for (int v = threadIdx.x; v < nvec; v += kConsumerWarps * 32) gamma_s[v] = __ldg(gamma + v);
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
  }
  uint32_t stage = 0, phase = 0;
  for (int64_t g = 0; g < groups; ++g) {
    const int64_t row = r_begin + g * kGroupRows + slot;
    PairX& x2 = px[slot * 2 + static_cast<int>(g & 1)];
    if (row < r_end) {
      const bool got = mbar_wait(smem_u32(&ctrl->full[stage][slot]), phase, abort, &g_err_quant, 52);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      const uint4* rp = reinterpret_cast<const uint4*>(smem + stage * stage_bytes + slot * row_bytes);
      uint4 xv[VPW];
#pragma unroll
      for (int i = 0; i < VPW; ++i) {
        const int v = hl + 64 * i;
        xv[i] = v < nvec ? rp[v] : make_uint4(0u, 0u, 0u, 0u);
      }
      // pass 1: sum of squares and the keyed max of |x * gamma|
      uint64_t hs[4] = {0, 0, 0, 0}, ls[4] = {0, 0, 0, 0};  // (+0, +0) pairs
      uint32_t kmax = 0;
#pragma unroll
      for (int i = 0; i < VPW; ++i) {
        const int v = hl + 64 * i;
        const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
        uint32_t gw[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
        if (GAMMA && v < nvec) {
          const uint4 gg = gamma_s[v];
          gw[0] = gg.x;
          gw[1] = gg.y;
          gw[2] = gg.z;
          gw[3] = gg.w;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t xx = bf16x2_to_f2(xw[k]);
          // the squares of bf16 values are exact, so a contraction of x * x
          // into the sum changes nothing; the sqrt+div form's (x * x) / K is
          // rounded on its own, as the oracle does
          uint64_t t = f2_mul(xx, xx);
          if (MODE == 1) {
            float t0, t1;
            f2_split(t, t0, t1);
            t = f2(__fmul_rn(t0, inv_d), __fmul_rn(t1, inv_d));
          }
          two_sum2(hs[k], ls[k], t);
          float p0, p1;
          f2_split(GAMMA ? f2_mul(xx, bf16x2_to_f2(gw[k])) : xx, p0, p1);
          // position: element 2k (+1) of vector i, in this half
          const uint32_t pos = static_cast<uint32_t>(sub * 128 + 8 * i + 2 * k);
          if (v < nvec) kmax = max(kmax, max(pos_key(p0, pos), pos_key(p1, pos + 1)));
        }
      }
      // the chains: pair k holds the terms of elements 2k and 2k + 1 of each vector
      float h8[8], l8[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        f2_split(hs[k], h8[2 * k], h8[2 * k + 1]);
        f2_split(ls[k], l8[2 * k], l8[2 * k + 1]);
      }
      float whi, wlo;
      ff_warp_pair(h8, l8, whi, wlo);
      const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, kmax);
      if (lane == 0) {
        x2.hi[sub] = whi;
        x2.lo[sub] = wlo;
        x2.kmax[sub] = wk;
      }
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      // both halves added in the same order in both warps: identical totals
      float tot, e;
      two_sum(x2.hi[0], x2.hi[1], tot, e);
      const float rest = __fadd_rn(__fadd_rn(x2.lo[0], x2.lo[1]), e);
      const float rstd = rstd_of_sum<MODE>(__fadd_rn(tot, rest), inv_d, eps);
      // amax guess: y of the element with the largest exact |x * gamma|
      const uint32_t kbest = max(x2.kmax[0], x2.kmax[1]);
      const uint32_t pos = kbest & 0xFFu;
      if (static_cast<int>(pos >> 7) == sub) {
        const int i = static_cast<int>((pos & 127u) >> 3), j = static_cast<int>(pos & 7u);
        const uint32_t owner = __ffs(__ballot_sync(0xFFFFFFFFu, kmax == kbest)) - 1;
        if (lane == static_cast<int>(owner)) {
          const int v = hl + 64 * i;
          float y = __fmul_rn(bf16_at(rp[v], j), rstd);
          if (GAMMA) y = __fmul_rn(y, bf16_at(gamma_s[v], j));
          x2.guess = fabsf(y);
        }
      }
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      float amax = x2.guess;
      // the row is in registers: this warp's share of the slot goes back
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->empty[stage]));
      uint4* ar = A + row * nvec;
      uint2* qr = q_out != nullptr ? q_out + row * nvec : nullptr;
      if (!RNL_DCHECK(&g_err_quant, row < T && nvec <= 64 * VPW, 54)) break;
      // pass 2, again with the exact max when a rounding beat the guess
      for (int attempt = 0; attempt < 2; ++attempt) {
        const bool zero_row = !(amax > 0.f);
        const float qs = zero_row ? 0.f : __fdiv_rn(127.0f, amax);
        // non-negative binary32 values order like their bit patterns
        const uint32_t yb = __reduce_max_sync(
            0xFFFFFFFFu, __float_as_uint(codes_pass<GAMMA, VPW>(xv, gamma_s, hl, nvec, rstd, qs, ar, qr)));
        if (lane == 0) x2.ymax[attempt][sub] = yb;
        asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
        const float ytrue = __uint_as_float(max(x2.ymax[attempt][0], x2.ymax[attempt][1]));
        if (!(ytrue > amax)) break;  // the guess was the maximum
        amax = ytrue;
      }
      if (sub == 0 && lane == 0) x_scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
    } else {
      // no row for this pair in the group: its slot share is released all the same
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->empty[stage]));
    }
    if (++stage == static_cast<uint32_t>(stages)) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

template <int MODE, bool GAMMA, int VPW>
rnl_status launch_qs(const void* x, const void* gamma, int64_t T, int nvec, int stages, float inv_d,
                     float eps, void* A, int8_t* q_out, float* x_scale, size_t smem,
                     const DeviceInfo& dev, cudaStream_t s) {
  auto kern = quant_stream_kernel<MODE, GAMMA, VPW>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device,
                       kRingBytes + 128 + 8192 + sizeof(QsCtrl) + 16 + 2 * kGroupRows * sizeof(PairX)) !=
          RNL_OK)
    return RNL_ERR_LAUNCH;
  const int64_t groups = (T + kGroupRows - 1) / kGroupRows;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(groups < dev.sm_count ? groups : dev.sm_count), 1, 1);
  cfg.blockDim = dim3(kThreadsQS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(x),
                                           static_cast<const uint4*>(gamma), T, nvec, stages, inv_d, eps,
                                           static_cast<uint4*>(A), reinterpret_cast<uint2*>(q_out), x_scale);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

template <int VPW>
rnl_status dispatch_mode(const void* x, const void* gamma, int64_t T, int nvec, int stages, float inv_d,
                         float eps, void* A, int8_t* q, float* xs, size_t smem, const DeviceInfo& dev,
                         cudaStream_t s, int mode) {
  if (mode == RNL_NORM_RSQRT)
    return gamma ? launch_qs<0, true, VPW>(x, gamma, T, nvec, stages, inv_d, eps, A, q, xs, smem, dev, s)
                 : launch_qs<0, false, VPW>(x, gamma, T, nvec, stages, inv_d, eps, A, q, xs, smem, dev, s);
  return gamma ? launch_qs<1, true, VPW>(x, gamma, T, nvec, stages, inv_d, eps, A, q, xs, smem, dev, s)
               : launch_qs<1, false, VPW>(x, gamma, T, nvec, stages, inv_d, eps, A, q, xs, smem, dev, s);
}

}  // namespace

bool quant_stream_fits(int64_t K) { return K > 0 && K <= 4096 && K % 8 == 0; }

rnl_status launch_quant_stream(const void* x, const void* gamma, int64_t T, int64_t K, float eps, int mode,
                               void* A, int8_t* q_out, float* x_scale, cudaStream_t s) {
  if (T == 0) return RNL_OK;
  if (!quant_stream_fits(K)) return RNL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const int nvec = static_cast<int>(K / 8);
  const size_t stage = static_cast<size_t>(kGroupRows) * static_cast<size_t>(K) * 2;
  int stages = static_cast<int>(kRingBytes / stage);
  if (stages > kMaxQsStages) stages = kMaxQsStages;
  // ring, then the gamma row, the barriers and the pairs' exchange slots
  const size_t smem = 128 + static_cast<size_t>(stages) * stage + static_cast<size_t>(K) * 2 + sizeof(QsCtrl) +
                      16 + 2 * kGroupRows * sizeof(PairX);
  const float inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  trace_before(s);
  const int vpw = (nvec + 63) / 64;  // vectors a lane holds (two warps per row)
  if (vpw <= 2)
    st = dispatch_mode<2>(x, gamma, T, nvec, stages, inv_d, eps, A, q_out, x_scale, smem, dev, s, mode);
  else if (vpw <= 4)
    st = dispatch_mode<4>(x, gamma, T, nvec, stages, inv_d, eps, A, q_out, x_scale, smem, dev, s, mode);
  else
    st = dispatch_mode<8>(x, gamma, T, nvec, stages, inv_d, eps, A, q_out, x_scale, smem, dev, s, mode);
  trace_after(s, "w8a8_quant");
  return st;
}

rnl_status read_clear_error_quant(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_quant, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_quant, &zero, sizeof zero) != cudaSuccess) return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
