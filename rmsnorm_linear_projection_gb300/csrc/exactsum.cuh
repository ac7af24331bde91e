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

// ---- The same float-float sum on packed f32x2 arithmetic: two chains per
// instruction.  Four packed chains per lane (eight scalar chains, one per
// element position of a 16-byte bf16 vector), merged into one pair.  A
// packed product feeding a packed sum could be contracted by ptxas into one
// fused multiply-add, so the terms' products (which must be rounded, in the
// sqrt+div form) are scalar __fmul_rn; the squares of bf16 values are exact.
__device__ __forceinline__ uint64_t ffx2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void ffx2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffx2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t ffx2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t ffx2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// TwoSum of (hi, t) per half, the error added to lo
__device__ __forceinline__ void ffx2_two_sum(uint64_t& hi, uint64_t& lo, uint64_t t) {
  const uint64_t s = ffx2_add(hi, t);
  const uint64_t bb = ffx2_sub(s, hi);
  const uint64_t e = ffx2_add(ffx2_sub(hi, ffx2_sub(s, bb)), ffx2_sub(t, bb));
  hi = s;
  lo = ffx2_add(lo, e);
}
// the eight terms of one 16-byte bf16 vector into the lane's four packed chains
template <int MODE>
__device__ __forceinline__ void ffx2_add_squares8(const uint4& u, float inv_d, uint64_t (&hs)[4],
                                                  uint64_t (&ls)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t xx = ffx2_pack(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
    uint64_t t = ffx2_mul(xx, xx);  // exact: bf16 squares
    if (MODE == 1) {
      float t0, t1;
      ffx2_unpack(t, t0, t1);
      t = ffx2_pack(__fmul_rn(t0, inv_d), __fmul_rn(t1, inv_d));
    }
    ffx2_two_sum(hs[k], ls[k], t);
  }
}
// the binary32 rounding of the warp's total of all lanes' chains
__device__ __forceinline__ float ffx2_warp_total(uint64_t (&hs)[4], uint64_t (&ls)[4]) {
  ffx2_two_sum(hs[0], ls[0], hs[1]);
  ls[0] = ffx2_add(ls[0], ls[1]);
  ffx2_two_sum(hs[2], ls[2], hs[3]);
  ls[2] = ffx2_add(ls[2], ls[3]);
  ffx2_two_sum(hs[0], ls[0], hs[2]);
  ls[0] = ffx2_add(ls[0], ls[2]);
  float h0, h1, l0, l1;
  ffx2_unpack(hs[0], h0, h1);
  ffx2_unpack(ls[0], l0, l1);
  float hi, e;
  two_sum(h0, h1, hi, e);
  float lo = __fadd_rn(__fadd_rn(l0, l1), e);
  ff_warp_merge(hi, lo);
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
