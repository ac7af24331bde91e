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
// One warp per (token, group of 8 heads): lane l holds D/32 consecutive
// values of each head, the sum of squares is a warp reduction, and the
// rotation partner of element i (i + D/2) sits in lane l ^ 16.  HBM / L2
// bound: each head row is read once and written once.
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

template <int E>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float (&f)[E]) {
  if constexpr (E == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xFFFF0000u);
  } else if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int E>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* p, const float (&f)[E]) {
  if constexpr (E == 2) {
    *reinterpret_cast<uint32_t*>(p) = pack2(f[0], f[1]);
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack2(f[0], f[1]), pack2(f[2], f[3]));
  } else {
    *reinterpret_cast<uint4*>(p) =
        make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  }
}

// Heads per warp: the token's position, its table row and both gammas are
// loaded once per warp, and the heads' rows are all loaded before any is
// processed.
constexpr int kHeadsPerWarp = 8;

template <int E>
__device__ __forceinline__ void load_f32v(const float* p, float (&f)[E]) {
  if constexpr (E == 2) {
    const float2 u = *reinterpret_cast<const float2*>(p);
    f[0] = u.x;
    f[1] = u.y;
  } else if constexpr (E == 4) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
  } else {
    const float4 u0 = *reinterpret_cast<const float4*>(p);
    const float4 u1 = *reinterpret_cast<const float4*>(p + 4);
    f[0] = u0.x; f[1] = u0.y; f[2] = u0.z; f[3] = u0.w;
    f[4] = u1.x; f[5] = u1.y; f[6] = u1.z; f[7] = u1.w;
  }
}

template <int D>
__global__ void __launch_bounds__(kRopeWarps * 32)
    qkv_rope_kernel(const __nv_bfloat16* __restrict__ y, int64_t T, int Hq, int Hkv, int groups,
                    const __nv_bfloat16* __restrict__ q_gamma,
                    const __nv_bfloat16* __restrict__ k_gamma, float eps,
                    const int* __restrict__ pos, const float* __restrict__ cs, int P,
                    __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
                    __nv_bfloat16* __restrict__ v) {
  constexpr int E = D / 32;  // values per lane
  const int lane = threadIdx.x & 31;
  const int H = Hq + 2 * Hkv;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kRopeWarps + (threadIdx.x >> 5);
  if (wid >= T * groups) return;
  const int64_t t = wid / groups;
  const int h0 = static_cast<int>(wid - t * groups) * kHeadsPerWarp;
  const int nh = H - h0 < kHeadsPerWarp ? H - h0 : kHeadsPerWarp;
  const __nv_bfloat16* yt = y + t * H * D + lane * E;
  // every head row of the group first
  float f[kHeadsPerWarp][E];
#pragma unroll
  for (int j = 0; j < kHeadsPerWarp; ++j)
    if (j < nh) load_bf16<E>(yt + (h0 + j) * D, f[j]);
  const bool any_qk = h0 < Hq + Hkv;
  int p = 0;
  bool p_ok = true;
  float c[E], sn[E], gq[E], gk[E];
  if (any_qk) {
    p = __ldg(pos + t);
    p_ok = p >= 0 && p < P;
    if (!p_ok) {  // nothing is read from the table; the caller gets RNL_ERR_ARG
      if (lane == 0) atomicCAS(&g_err_rope, 0u, kErrArg | (40u << 8));
    } else {
      const float* row = cs + static_cast<int64_t>(p) * D + (lane & 15) * E;
      load_f32v<E>(row, c);
      load_f32v<E>(row + D / 2, sn);
    }
    if (Hq > 0) load_bf16<E>(q_gamma + lane * E, gq);
    if (Hkv > 0) load_bf16<E>(k_gamma + lane * E, gk);
  }
#pragma unroll
  for (int j = 0; j < kHeadsPerWarp; ++j) {
    if (j >= nh) break;
    const int h = h0 + j;
    if (h >= Hq + Hkv) {  // v head: copied
      store_bf16<E>(v + (t * Hkv + (h - Hq - Hkv)) * D + lane * E, f[j]);
      continue;
    }
    if (!p_ok) continue;
    const bool is_q = h < Hq;
    __nv_bfloat16* dst = is_q ? q + (t * Hq + h) * D : k + (t * Hkv + (h - Hq)) * D;
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(f[j][e], f[j][e], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss * (1.0f / D) + eps);
    float z[E], zp[E], out[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
      z[e] = bf16_round(__fmul_rn(__fmul_rn(f[j][e], r), is_q ? gq[e] : gk[e]));
#pragma unroll
    for (int e = 0; e < E; ++e) zp[e] = __shfl_xor_sync(0xffffffffu, z[e], 16);
    if (lane < 16) {
#pragma unroll
      for (int e = 0; e < E; ++e) out[e] = __fsub_rn(__fmul_rn(z[e], c[e]), __fmul_rn(zp[e], sn[e]));
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) out[e] = __fadd_rn(__fmul_rn(z[e], c[e]), __fmul_rn(zp[e], sn[e]));
    }
    store_bf16<E>(dst + lane * E, out);
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
