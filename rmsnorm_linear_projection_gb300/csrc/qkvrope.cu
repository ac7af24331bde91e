// qkvrope.cu -- the V stage after the qkv projection (AT-10 pattern page,
// sec. 6, Qwen3PreAttn: the projection output is split into Q, K and V, and
// Q and K each get a per-head RMSNorm and the rotary embedding):
//
//   y [T, (Hq + 2 Hkv) * D] bf16: q heads, then k heads, then v heads
//   q / k head row h:  r = rsqrt(mean(h^2) + eps)           (FP32)
//                      z = bf16((h * r) * gamma)            (gamma of size D)
//                      o[i]       = bf16(z[i] c_i - z[i + D/2] s_i)
//                      o[i + D/2] = bf16(z[i + D/2] c_i + z[i] s_i),  i < D/2
//   with (c_i, s_i) read from the caller's angle table [P, D] (cos | sin) at
//   the token's position; v heads are copied unchanged.
//
// One warp per (token, group of 8 heads); each head row is read once and
// written once (HBM bound).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_rope;  // kErrArg | site: a position outside [0, P)

constexpr int kRopeWarps = 8;

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// N consecutive bf16 (N = 1, 2, 4) <-> floats, and N consecutive floats.
template <int N>
__device__ __forceinline__ void load_bf16n(const __nv_bfloat16* p, float (&f)[N]) {
  if constexpr (N == 1) {
    f[0] = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  } else if constexpr (N == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xFFFF0000u);
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xFFFF0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int N>
__device__ __forceinline__ void store_bf16n(__nv_bfloat16* p, const float (&f)[N]) {
  if constexpr (N == 1) {
    *p = __float2bfloat16_rn(f[0]);
  } else if constexpr (N == 2) {
    *reinterpret_cast<uint32_t*>(p) = pack2(f[0], f[1]);
  } else {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack2(f[0], f[1]), pack2(f[2], f[3]));
  }
}

template <int N>
__device__ __forceinline__ void load_f32n(const float* p, float (&f)[N]) {
  if constexpr (N == 1) {
    f[0] = *p;
  } else if constexpr (N == 2) {
    const float2 u = *reinterpret_cast<const float2*>(p);
    f[0] = u.x;
    f[1] = u.y;
  } else {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
  }
}

// Heads per warp: the token's position, its table row and both gammas are
// loaded once per warp, and the heads' rows are all loaded before any is
// processed.
constexpr int kHeadsPerWarp = 8;

// Lane l holds R = D/64 elements of each half of a head row: i in
// [l R, l R + R) and their rotation partners i + D/2, so the rotation needs
// no shuffle, and every load or store instruction of the warp covers a
// contiguous 32 R elements.  The 8 heads' sums of squares are reduced
// together (a reduce-scatter: 4 + 2 + 1 shuffles leave each lane with one
// head's partial over 4 lanes, 2 more finish it), one rsqrt a lane, and
// 8 shuffles hand every head its factor: 17 shuffles and 1 rsqrt for 8
// heads instead of 40 and 8.
template <int D>
__global__ void __launch_bounds__(kRopeWarps * 32)
    qkv_rope_kernel(const __nv_bfloat16* __restrict__ y, int64_t T, int Hq, int Hkv, int groups,
                    const __nv_bfloat16* __restrict__ q_gamma,
                    const __nv_bfloat16* __restrict__ k_gamma, float eps,
                    const int* __restrict__ pos, const float* __restrict__ cs, int P,
                    __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
                    __nv_bfloat16* __restrict__ v) {
  constexpr int R = D / 64;  // values of each half per lane
  constexpr int kHalf = D / 2;
  const int lane = threadIdx.x & 31;
  const int H = Hq + 2 * Hkv;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kRopeWarps + (threadIdx.x >> 5);
  if (wid >= T * groups) return;
  const int64_t t = wid / groups;
  const int h0 = static_cast<int>(wid - t * groups) * kHeadsPerWarp;
  const int nh = H - h0 < kHeadsPerWarp ? H - h0 : kHeadsPerWarp;
  const __nv_bfloat16* yt = y + t * H * D + lane * R;
  // every head row of the group first
  float lo[kHeadsPerWarp][R], hi[kHeadsPerWarp][R];
#pragma unroll
  for (int j = 0; j < kHeadsPerWarp; ++j)
    if (j < nh) {
      load_bf16n<R>(yt + (h0 + j) * D, lo[j]);
      load_bf16n<R>(yt + (h0 + j) * D + kHalf, hi[j]);
    }
  const int nqk = Hq + Hkv;  // heads below this index are normalised and rotated
  const bool any_qk = h0 < nqk;
  bool p_ok = true;
  float c[R], sn[R], gql[R], gqh[R], gkl[R], gkh[R];
  if (any_qk) {
    const int p = __ldg(pos + t);
    p_ok = p >= 0 && p < P;
    if (!p_ok) {  // nothing is read from the table; the caller gets RNL_ERR_ARG
      if (lane == 0) atomicCAS(&g_err_rope, 0u, kErrArg | (40u << 8));
    } else {
      const float* row = cs + static_cast<int64_t>(p) * D + lane * R;
      load_f32n<R>(row, c);
      load_f32n<R>(row + kHalf, sn);
    }
    if (Hq > 0) {
      load_bf16n<R>(q_gamma + lane * R, gql);
      load_bf16n<R>(q_gamma + kHalf + lane * R, gqh);
    }
    if (Hkv > 0) {
      load_bf16n<R>(k_gamma + lane * R, gkl);
      load_bf16n<R>(k_gamma + kHalf + lane * R, gkh);
    }
  }
  float r[kHeadsPerWarp];
  if (any_qk) {
    float ss[kHeadsPerWarp];
#pragma unroll
    for (int j = 0; j < kHeadsPerWarp; ++j) {
      ss[j] = 0.f;
      if (j < nh && h0 + j < nqk) {
#pragma unroll
        for (int e = 0; e < R; ++e) ss[j] = fmaf(lo[j][e], lo[j][e], ss[j]);
#pragma unroll
        for (int e = 0; e < R; ++e) ss[j] = fmaf(hi[j][e], hi[j][e], ss[j]);
      }
    }
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float s4[4], s2[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = b4 ? ss[i] : ss[i + 4];
      s4[i] = (b4 ? ss[i + 4] : ss[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = b3 ? s4[i] : s4[i + 2];
      s2[i] = (b3 ? s4[i + 2] : s4[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float s1 = (b2 ? s2[1] : s2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? s2[0] : s2[1], 4);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    // this lane now holds head ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)
    const float rl = rsqrtf(s1 * (1.0f / D) + eps);
#pragma unroll
    for (int j = 0; j < kHeadsPerWarp; ++j)
      r[j] = __shfl_sync(0xffffffffu, rl, ((j >> 2) & 1) << 4 | ((j >> 1) & 1) << 3 | (j & 1) << 2);
  }
#pragma unroll
  for (int j = 0; j < kHeadsPerWarp; ++j) {
    if (j >= nh) break;
    const int h = h0 + j;
    if (h >= nqk) {  // v head: copied
      __nv_bfloat16* dv = v + (t * Hkv + (h - nqk)) * D + lane * R;
      store_bf16n<R>(dv, lo[j]);
      store_bf16n<R>(dv + kHalf, hi[j]);
      continue;
    }
    if (!p_ok) continue;
    const bool is_q = h < Hq;
    __nv_bfloat16* dst = (is_q ? q + (t * Hq + h) * D : k + (t * Hkv + (h - Hq)) * D) + lane * R;
    float ol[R], oh[R];
#pragma unroll
    for (int e = 0; e < R; ++e) {
      const float zl = bf16_round(__fmul_rn(__fmul_rn(lo[j][e], r[j]), is_q ? gql[e] : gkl[e]));
      const float zh = bf16_round(__fmul_rn(__fmul_rn(hi[j][e], r[j]), is_q ? gqh[e] : gkh[e]));
      ol[e] = __fsub_rn(__fmul_rn(zl, c[e]), __fmul_rn(zh, sn[e]));
      oh[e] = __fadd_rn(__fmul_rn(zh, c[e]), __fmul_rn(zl, sn[e]));
    }
    store_bf16n<R>(dst, ol);
    store_bf16n<R>(dst + kHalf, oh);
  }
}

}  // namespace

bool qkv_rope_head_dim_ok(int64_t D) { return D == 64 || D == 128 || D == 256; }

rnl_status launch_qkv_rope(const void* y, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                           const void* q_gamma, const void* k_gamma, float eps,
                           const int32_t* positions, const float* cos_sin, int64_t max_pos,
                           void* q, void* k, void* v, cudaStream_t s) {
  const int64_t H = Hq + 2 * Hkv;
  if (T * H == 0) return RNL_OK;
  const int groups = static_cast<int>((H + kHeadsPerWarp - 1) / kHeadsPerWarp);
  const int64_t warps = T * groups;
  const unsigned blocks = static_cast<unsigned>((warps + kRopeWarps - 1) / kRopeWarps);
  const auto* yp = static_cast<const __nv_bfloat16*>(y);
  const auto* qg = static_cast<const __nv_bfloat16*>(q_gamma);
  const auto* kg = static_cast<const __nv_bfloat16*>(k_gamma);
  auto* qp = static_cast<__nv_bfloat16*>(q);
  auto* kp = static_cast<__nv_bfloat16*>(k);
  auto* vp = static_cast<__nv_bfloat16*>(v);
  const int hq = static_cast<int>(Hq), hkv = static_cast<int>(Hkv), P = static_cast<int>(max_pos);
  trace_before(s);
  switch (D) {
    case 64:
      qkv_rope_kernel<64><<<blocks, kRopeWarps * 32, 0, s>>>(yp, T, hq, hkv, groups, qg, kg, eps, positions,
                                                             cos_sin, P, qp, kp, vp);
      break;
    case 128:
      qkv_rope_kernel<128><<<blocks, kRopeWarps * 32, 0, s>>>(yp, T, hq, hkv, groups, qg, kg, eps, positions,
                                                              cos_sin, P, qp, kp, vp);
      break;
    default:
      qkv_rope_kernel<256><<<blocks, kRopeWarps * 32, 0, s>>>(yp, T, hq, hkv, groups, qg, kg, eps, positions,
                                                              cos_sin, P, qp, kp, vp);
      break;
  }
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "qkv_rope");
  return st;
}

rnl_status read_clear_error_rope(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_rope, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_rope, &zero, sizeof zero) != cudaSuccess)
    return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
