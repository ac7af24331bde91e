// exactsum.cuh -- the binary32 value of a row's exact sum of squares, for the
// quantising front ends (W8A8 and MXFP8), where FP32 values decide integer or
// E4M3 codes and so must not depend on the order of the K-term sum.
//
// Each term (x*x, or (x*x)*(1/K) for the sqrt+div form) is one binary32
// product; the terms are added in float-float (hi + lo, Knuth's TwoSum per
// term and per merge), which carries the sum to about 2^-44 relative, and the
// result is rounded once to binary32.
#pragma once

#include <cstdint>

namespace rnl {

// Error-free transformation of a sum (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Adds the eight terms of one 16-byte bf16 vector to eight float-float chains.
template <int MODE>
__device__ __forceinline__ void ff_add_squares8(const float (&f)[8], float inv_d, float (&hs)[8],
                                                float (&ls)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float t = __fmul_rn(f[j], f[j]);
    if (MODE == 1) t = __fmul_rn(t, inv_d);
    float sum, e;
    two_sum(hs[j], t, sum, e);
    hs[j] = sum;
    ls[j] = __fadd_rn(ls[j], e);
  }
}

// Adds the float-float pairs (hi, lo) of the warp's 32 lanes (butterfly):
// the same pair on every lane.
__device__ __forceinline__ void ff_warp_merge(float& hi, float& lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    float sum, e;
    two_sum(hi, h2, sum, e);
    lo = __fadd_rn(__fadd_rn(lo, l2), e);
    hi = sum;
  }
}

// Merges the eight chains of every lane of the warp into one float-float
// pair (hi, lo), the same on every lane, left unrounded so that several
// warps' pairs can be merged further.
__device__ __forceinline__ void ff_warp_hilo(const float (&hs)[8], const float (&ls)[8], float& hi_out,
                                             float& lo_out) {
  float hi = hs[0], lo = ls[0];
#pragma unroll
  for (int j = 1; j < 8; ++j) {
    float sum, e;
    two_sum(hi, hs[j], sum, e);
    lo = __fadd_rn(__fadd_rn(lo, ls[j]), e);
    hi = sum;
  }
  ff_warp_merge(hi, lo);
  hi_out = hi;
  lo_out = lo;
}

// The binary32 rounding of the warp's total (the same value on every lane).
__device__ __forceinline__ float ff_warp_total(const float (&hs)[8], const float (&ls)[8]) {
  float hi, lo;
  ff_warp_hilo(hs, ls, hi, lo);
  return __fadd_rn(hi, lo);
}

// rstd from the binary32 sum, one correctly rounded operation per step:
// 1 / sqrt(ss * (1/K) + eps) (rsqrt form, MODE 0) or 1 / sqrt(ss + eps)
// (sqrt+div form, whose terms already carry 1/K).
template <int MODE>
__device__ __forceinline__ float rstd_of_sum(float ss, float inv_d, float eps) {
  if (MODE == 0) return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, inv_d), eps)));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ss, eps)));
}

}  // namespace rnl
