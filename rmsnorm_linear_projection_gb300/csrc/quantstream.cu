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
// contiguous range of rows; a producer thread bulk-copies each row into a
// ring of shared-memory row slots, and 16 consumer warps, in pairs, take one
// row per pair (rows j, j + 8, ... of the CTA's range; lane l of half h
// holds the 16-byte vectors 32 h + l + 64 i of the row).  Each warp copies
// its half of the row from the slot into registers and hands its share of
// the slot straight back, so nearly the whole ring holds rows still to come
// and the bulk copies run far enough ahead of the warps (a slot held through
// the arithmetic left most warps waiting for their next row; a whole row in
// one warp's registers did not fit beside 16 warps).  Three passes over the
// registers, the halves exchanged through shared memory in a fixed order so
// that both warps hold the same totals:
//   pass 1  the sum of squares: four packed float-float chains per lane
//           (f32x2 arithmetic, TwoSum per term), merged across the warp,
//           then the two halves;
//   pass 2  amax, the exact max |y| of the row;
//   pass 3  the codes (y * qs, rint) and their stores.
// VPL, the vectors a lane holds, is a compile-time count (the register
// array); a slot is VPL * 64 vectors long, its tail past the row zeroed once
// (as is gamma's), so every load is unconditional and the zeros add nothing
// to the sum or the maximum.  The row reads bound the kernel: on the
// hardware it was tuned on, reads alone stream at about 3.6 TB/s (a copy
// reaches its 6.8 TB/s only with as many writes), and the arithmetic per
// element (about 16 instructions) is of the same order.
#include <cuda_bf16.h>

#include "exactsum.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_quant;

constexpr int kConsumerWarps = 16;  // two per row
constexpr int kThreadsQS = (kConsumerWarps + 1) * 32;
constexpr int kMaxSlots = 32;
constexpr size_t kRingBytes = 200 * 1024;
constexpr int kMaxVpl = 8;  // rows of up to 64 * 8 vectors of 8 elements

constexpr int kPairs = kConsumerWarps / 2;
struct __align__(8) QsCtrl {
  uint64_t full[kMaxSlots];   // a row landed in the slot
  uint64_t empty[kMaxSlots];  // both warps of the slot's pair have the row in registers
  float hi[kPairs][2], lo[kPairs][2];  // each half's float-float sum of squares
  uint32_t amax[kPairs][2];            // each half's max |y|
  int ok[kPairs][2];                   // each warp's row arrived
  uint32_t gmax[kConsumerWarps + 1];   // each warp's max |gamma| over its staged part
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
// merges chain pair (h1, l1) into (h0, l0), both halves at once
__device__ __forceinline__ void ff_merge2(uint64_t& h0, uint64_t& l0, uint64_t h1, uint64_t l1) {
  two_sum2(h0, l0, h1);
  l0 = f2_add(l0, l1);
}
__device__ __forceinline__ uint32_t vec_word(const uint4& u, int k) {
  return k == 0 ? u.x : k == 1 ? u.y : k == 2 ? u.z : u.w;
}
// gamma of the elements of word k of a vector, from its two float4 halves
__device__ __forceinline__ uint64_t g_pair(const float4& a, const float4& b, int k) {
  return k == 0 ? f2(a.x, a.y) : k == 1 ? f2(a.z, a.w) : k == 2 ? f2(b.x, b.y) : f2(b.z, b.w);
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Pass 1: this warp's half of the row's sum of squares as an unrounded
// float-float pair (the same on every lane).  The terms are x * x, or
// (x * x) * (1/K) in the sqrt+div form.
template <int MODE, int VPL>
__device__ __forceinline__ void pass_sum(const uint4 (&xv)[VPL], float inv_d, float& hi_out, float& lo_out) {
  uint64_t hs[4] = {0, 0, 0, 0}, ls[4] = {0, 0, 0, 0};  // (+0, +0) pairs
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t xx = bf16x2_to_f2(vec_word(xv[i], k));
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
    }
  }
  // the lane's eight chains: packed pairs first, then the two halves
  ff_merge2(hs[0], ls[0], hs[1], ls[1]);
  ff_merge2(hs[2], ls[2], hs[3], ls[3]);
  ff_merge2(hs[0], ls[0], hs[2], ls[2]);
  float h0, h1, l0, l1;
  f2_split(hs[0], h0, h1);
  f2_split(ls[0], l0, l1);
  float hi, e;
  two_sum(h0, h1, hi, e);
  float lo = __fadd_rn(__fadd_rn(l0, l1), e);
  ff_warp_merge(hi, lo);
  hi_out = hi;
  lo_out = lo;
}

// y of one vector: (x * rstd) * gamma, each product rounded once (products
// only: nothing to contract)
template <bool GAMMA>
__device__ __forceinline__ void y_vec(const uint4& xv, const float4& ga, const float4& gb, uint64_t r2,
                                      uint64_t (&y)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    y[k] = f2_mul(bf16x2_to_f2(vec_word(xv, k)), r2);
    if (GAMMA) y[k] = f2_mul(y[k], g_pair(ga, gb, k));
  }
}

// Pass 2: the exact max |y| of this warp's half of the row (the same value
// on every lane).  Vector i of the lane is v = lane + 64 i past the half's
// first vector (ga_s, gb_s point there too).
template <bool GAMMA, int VPL>
__device__ __forceinline__ float pass_amax(const uint4 (&xv)[VPL], const float4* ga_s, const float4* gb_s,
                                           int lane, float rstd) {
  const uint64_t r2 = f2(rstd, rstd);
  float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int v = lane + 64 * i;
    float4 ga, gb;
    if (GAMMA) {
      ga = ga_s[v];
      gb = gb_s[v];
    }
    uint64_t y[4];
    y_vec<GAMMA>(xv[i], ga, gb, r2, y);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float y0, y1;
      f2_split(y[k], y0, y1);
      m[k] = max3(m[k], fabsf(y0), fabsf(y1));
    }
  }
  const float lm = max3(m[0], m[1], fmaxf(m[2], m[3]));
  // non-negative binary32 values order like their bit patterns
  return __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(lm)));
}

// Pass 3: the codes of this warp's half, to A as bf16 integers and to q_out
// as int8 (ar, qr and nvec counted from the half's first vector).
template <bool GAMMA, int VPL>
__device__ __forceinline__ void pass_codes(const uint4 (&xv)[VPL], const float4* ga_s, const float4* gb_s,
                                           int nvec, int lane, float rstd, float qs, uint4* __restrict__ ar,
                                           uint2* __restrict__ qr) {
  const uint64_t r2 = f2(rstd, rstd), qs2 = f2(qs, qs);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int v = lane + 64 * i;
    float4 ga, gb;
    if (GAMMA) {
      ga = ga_s[v];
      gb = gb_s[v];
    }
    uint64_t y[4];
    y_vec<GAMMA>(xv[i], ga, gb, r2, y);
    uint32_t o[4];
    float c[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // y * qs feeds no sum, so the packed product stays one rounding
      f2_split(f2_mul(y[k], qs2), c[2 * k], c[2 * k + 1]);
      c[2 * k] = rintf(c[2 * k]);
      c[2 * k + 1] = rintf(c[2 * k + 1]);
      __nv_bfloat162 h = __floats2bfloat162_rn(c[2 * k], c[2 * k + 1]);  // small integers: exact
      o[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    if (v < nvec) {
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
}

template <int MODE, bool GAMMA, int VPL>
__global__ void __launch_bounds__(kThreadsQS, 1)
    quant_stream_kernel(const uint8_t* x, const uint4* __restrict__ gamma, int64_t T, int nvec,
                        int slots, float inv_d, float eps, uint4* __restrict__ A,
                        uint2* __restrict__ q_out, float* __restrict__ x_scale,
                        float* __restrict__ gmax_out) {
  constexpr uint32_t kSlotBytes = 64u * VPL * 16u;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 127u) & ~127u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
  // gamma as binary32: elements 0-3 of each 16-byte vector of the row, then
  // elements 4-7 (a lane's 16-byte reads of either half are contiguous across
  // the warp), each 32 * VPL vectors long; then the barriers
  float4* ga_s = reinterpret_cast<float4*>(smem + static_cast<size_t>(slots) * kSlotBytes);
  float4* gb_s = ga_s + 64 * VPL;
  QsCtrl* ctrl = reinterpret_cast<QsCtrl*>(gb_s + 64 * VPL);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t r_begin = static_cast<int64_t>(blockIdx.x) * T / gridDim.x;
  const int64_t rows = static_cast<int64_t>(blockIdx.x + 1) * T / gridDim.x - r_begin;

  grid_launch_dependents();
  // zeros past the row in every slot (the bulk copies never write there)
  if (row_bytes < kSlotBytes) {
    const uint32_t pad = (kSlotBytes - row_bytes) / 16u;
    for (uint32_t i = threadIdx.x; i < static_cast<uint32_t>(slots) * pad; i += blockDim.x)
      reinterpret_cast<uint4*>(smem + (i / pad) * kSlotBytes + row_bytes)[i % pad] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < slots; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 2);
    }
    ctrl->abort = 0;
    fence_mbar_init();
  }
  grid_dependency_wait();  // everything below may touch the previous kernel's data
  if (GAMMA) {  // gamma staged once in shared memory for all rows, widened to binary32, zero past the row
    uint32_t gm = 0;  // max |gamma| of this thread's part (non-negative binary32 values order like their bits)
    for (int v = threadIdx.x; v < 64 * VPL; v += blockDim.x) {
      const uint4 g = v < nvec ? __ldg(gamma + v) : make_uint4(0u, 0u, 0u, 0u);
      ga_s[v] = make_float4(__uint_as_float(g.x << 16), __uint_as_float(g.x & 0xFFFF0000u),
                            __uint_as_float(g.y << 16), __uint_as_float(g.y & 0xFFFF0000u));
      gb_s[v] = make_float4(__uint_as_float(g.z << 16), __uint_as_float(g.z & 0xFFFF0000u),
                            __uint_as_float(g.w << 16), __uint_as_float(g.w & 0xFFFF0000u));
      gm = max(gm, max(max((g.x << 16) & 0x7FFFFFFFu, g.x & 0x7FFF0000u), max((g.y << 16) & 0x7FFFFFFFu, g.y & 0x7FFF0000u)));
      gm = max(gm, max(max((g.z << 16) & 0x7FFFFFFFu, g.z & 0x7FFF0000u), max((g.w << 16) & 0x7FFFFFFFu, g.w & 0x7FFF0000u)));
    }
    gm = __reduce_max_sync(0xFFFFFFFFu, gm);
    if (lane == 0) ctrl->gmax[warp] = gm;
  }
  __syncthreads();
  volatile int* abort = &ctrl->abort;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // row j of the range goes to slot j % slots, its (j / slots)-th use
    if (lane == 0) {
      for (int64_t j = 0; j < rows; ++j) {
        const uint32_t s = static_cast<uint32_t>(j % slots);
        const uint32_t use = static_cast<uint32_t>(j / slots);
        if (!mbar_wait(smem_u32(&ctrl->empty[s]), (use & 1u) ^ 1u, abort, &g_err_quant, 51)) break;
        if (!RNL_DCHECK(&g_err_quant, slots <= kMaxSlots && r_begin + j < T && row_bytes <= kSlotBytes &&
                                          static_cast<size_t>(slots) * kSlotBytes <= kRingBytes, 53))
          break;
        const uint32_t bar = smem_u32(&ctrl->full[s]);
        mbar_arrive_expect_tx(bar, row_bytes);
        bulk_copy_g2s(base + s * kSlotBytes, x + (r_begin + j) * row_bytes, row_bytes, bar);
      }
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  // warps 2p and 2p + 1 share row slot p: sub = which half (vectors
  // 32 sub + lane + 64 i); named barrier 1 + p joins the pair
  const int pair = warp >> 1, sub = warp & 1;
  const uint32_t pbar = 1u + static_cast<uint32_t>(pair);
  // max |gamma| for the integer GEMM's exactness bound (gemm_pair.cu), from
  // one thread of the grid (every CTA stages all of gamma)
  if (GAMMA && gmax_out != nullptr && blockIdx.x == 0 && warp == 0 && lane == 0) {
    uint32_t gm = ctrl->gmax[0];
    for (int i = 1; i <= kConsumerWarps; ++i) gm = max(gm, ctrl->gmax[i]);
    *gmax_out = __uint_as_float(gm);
  }
  for (int64_t j = pair; j < rows; j += kPairs) {
    const uint32_t s = static_cast<uint32_t>(j % slots);
    const uint32_t use = static_cast<uint32_t>(j / slots);
    const int64_t row = r_begin + j;
    bool ok = mbar_wait(smem_u32(&ctrl->full[s]), use & 1u, abort, &g_err_quant, 52);
    ok = __all_sync(0xFFFFFFFFu, ok) &&
         RNL_DCHECK(&g_err_quant, row < T && s < static_cast<uint32_t>(slots) && nvec <= 64 * VPL, 54);
    const uint4* rp = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(s) * kSlotBytes) + 32 * sub;
    uint4 xv[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) xv[i] = rp[lane + 64 * i];
    // this half of the row is in registers: the warp's share of the slot goes back
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctrl->empty[s]));
    float whi, wlo;
    pass_sum<MODE, VPL>(xv, inv_d, whi, wlo);
    if (lane == 0) {
      ctrl->hi[pair][sub] = whi;
      ctrl->lo[pair][sub] = wlo;
      ctrl->ok[pair][sub] = ok ? 1 : 0;
    }
    asm volatile("bar.sync %0, 64;" ::"r"(pbar) : "memory");
    if (!(ctrl->ok[pair][0] && ctrl->ok[pair][1])) break;  // both warps leave together
    // both halves added in the same order in both warps: identical totals
    float tot, e;
    two_sum(ctrl->hi[pair][0], ctrl->hi[pair][1], tot, e);
    const float rest = __fadd_rn(__fadd_rn(ctrl->lo[pair][0], ctrl->lo[pair][1]), e);
    const float rstd = rstd_of_sum<MODE>(__fadd_rn(tot, rest), inv_d, eps);
    const float wmax = pass_amax<GAMMA, VPL>(xv, ga_s + 32 * sub, gb_s + 32 * sub, lane, rstd);
    if (lane == 0) ctrl->amax[pair][sub] = __float_as_uint(wmax);
    asm volatile("bar.sync %0, 64;" ::"r"(pbar) : "memory");
    const float amax = __uint_as_float(max(ctrl->amax[pair][0], ctrl->amax[pair][1]));
    const float qs = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    pass_codes<GAMMA, VPL>(xv, ga_s + 32 * sub, gb_s + 32 * sub, nvec - 32 * sub, lane, rstd, qs,
                           A + row * nvec + 32 * sub,
                           q_out != nullptr ? q_out + row * nvec + 32 * sub : nullptr);
    if (lane == 0 && sub == 0) {
      x_scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
    }

  }
}

// shared memory of one launch: alignment slack, the ring, gamma's two halves, the barriers
size_t qs_smem(int vpl, int slots) {
  return 128 + static_cast<size_t>(slots) * 1024u * vpl + static_cast<size_t>(vpl) * 2048u + sizeof(QsCtrl);
}

template <int MODE, bool GAMMA, int VPL>
rnl_status launch_qs(const void* x, const void* gamma, int64_t T, int nvec, float inv_d, float eps, void* A,
                     int8_t* q_out, float* x_scale, float* gmax_out, const DeviceInfo& dev, cudaStream_t s) {
  int slots = static_cast<int>(kRingBytes / (1024u * VPL));
  if (slots > kMaxSlots) slots = kMaxSlots;
  const size_t smem = qs_smem(VPL, slots);
  auto kern = quant_stream_kernel<MODE, GAMMA, VPL>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, smem) != RNL_OK) return RNL_ERR_LAUNCH;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T < dev.sm_count ? T : dev.sm_count), 1, 1);
  cfg.blockDim = dim3(kThreadsQS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(x),
                                           static_cast<const uint4*>(gamma), T, nvec, slots, inv_d, eps,
                                           static_cast<uint4*>(A), reinterpret_cast<uint2*>(q_out), x_scale,
                                           gmax_out);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

template <int VPL>
rnl_status dispatch_mode(const void* x, const void* gamma, int64_t T, int nvec, float inv_d, float eps, void* A,
                         int8_t* q, float* xs, float* gm, const DeviceInfo& dev, cudaStream_t s, int mode) {
  if (mode == RNL_NORM_RSQRT)
    return gamma ? launch_qs<0, true, VPL>(x, gamma, T, nvec, inv_d, eps, A, q, xs, gm, dev, s)
                 : launch_qs<0, false, VPL>(x, gamma, T, nvec, inv_d, eps, A, q, xs, gm, dev, s);
  return gamma ? launch_qs<1, true, VPL>(x, gamma, T, nvec, inv_d, eps, A, q, xs, gm, dev, s)
               : launch_qs<1, false, VPL>(x, gamma, T, nvec, inv_d, eps, A, q, xs, gm, dev, s);
}

}  // namespace

bool quant_stream_fits(int64_t K) { return K > 0 && K <= 8 * 64 * kMaxVpl && K % 8 == 0; }

rnl_status launch_quant_stream(const void* x, const void* gamma, int64_t T, int64_t K, float eps, int mode,
                               void* A, int8_t* q_out, float* x_scale, float* gmax_out, cudaStream_t s) {
  if (T == 0) return RNL_OK;
  if (!quant_stream_fits(K)) return RNL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const int nvec = static_cast<int>(K / 8);
  const float inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  const int vpl = (nvec + 63) / 64;  // vectors a lane holds (two warps per row)
  trace_before(s);
  if (vpl <= 1)
    st = dispatch_mode<1>(x, gamma, T, nvec, inv_d, eps, A, q_out, x_scale, gmax_out, dev, s, mode);
  else if (vpl <= 2)
    st = dispatch_mode<2>(x, gamma, T, nvec, inv_d, eps, A, q_out, x_scale, gmax_out, dev, s, mode);
  else if (vpl <= 4)
    st = dispatch_mode<4>(x, gamma, T, nvec, inv_d, eps, A, q_out, x_scale, gmax_out, dev, s, mode);
  else
    st = dispatch_mode<8>(x, gamma, T, nvec, inv_d, eps, A, q_out, x_scale, gmax_out, dev, s, mode);
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
