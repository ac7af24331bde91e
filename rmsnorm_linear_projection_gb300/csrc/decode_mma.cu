// decode_mma.cu -- the AT-10 RMSNorm + Linear (bf16 out) for a handful of
// tokens (T <= 4, a decode step) on the tensor cores, bound by one read of
// the weight.
//
// out^T = W a^T: the weight is the MMA's A operand (128-row tiles, K-major,
// as stored) and the normalised tokens a = bf16((x rstd) gamma) the B
// operand, padded with zero rows to N = 16; the fp32 accumulator lives in
// TMEM.  A weight tile's K range is split over S CTAs (S = SMs / tiles, at
// most 8, every CTA resident at once), so that every SM streams its share of
// W: 6144 rows -> 48 tiles x 3 = 144 CTAs.
//
//   warp 0      TMA producer: the CTA's W k-blocks (128 x 64, 128-byte
//               swizzle) into a ring of 16 KB stages (up to 12: most of a
//               CTA's share of W is in flight at once)
//   warps 1-4   the norm: one token row per warp (sum of squares over all of
//               K, rstd as the AT-10 page, sec. 3 defines it, the row's loads
//               issued at once), then the CTA's k-blocks of a in the MMA's B
//               layout from the K slices of x and gamma that the producer
//               bulk-copied ahead of the weight (a prologue behind 25 MB of
//               weight requests took half the kernel); warp 1 then issues
//               the MMAs (M = 128, N = 16, K = 16) and, after the last one,
//               warps 1-4 read the 128 x T partial sums from TMEM
//   K split     ranks 1 .. S-1 of a tile write their fp32 partial sums to
//               the workspace and publish a flag tagged with the launch's
//               epoch; rank 0 waits for them (bounded), adds them in rank
//               order, one fixed order, writes out[t, n] = bf16(sum) and sets
//               the flags back to 0 (a replayed graph waits for its own)
//
// The summation order differs from the other paths, inside the same bf16
// output bound.  (A thread-block cluster per tile would exchange the partial
// sums on chip, but clusters of three CTAs of this size do not all fit at
// once: 46 of the 48 needed on 152 SMs, and the last two ran as a second
// wave.)
#include <cuda_bf16.h>

#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_decmma;

constexpr int kDmTokens = 4;              // tokens (rows of a used; B has 16)
constexpr int kDmN = 16;                  // the MMA's N: tokens padded with zero rows
constexpr int kDmThreads = 160;           // producer warp + four norm / MMA / epilogue warps
constexpr int kDmMaxSplit = 8;            // CTAs per weight tile
constexpr uint32_t kDmStage = 128 * 128;  // one W k-block: 128 rows x 128 bytes
constexpr uint32_t kDmBBlock = kDmN * 128;  // one k-block of a: 16 rows x 128 bytes
constexpr int kDmMaxStages = 12;
constexpr size_t kDmSmemLimit = 227 * 1024;

struct __align__(8) DmCtrl {
  uint64_t full[kDmMaxStages];
  uint64_t empty[kDmMaxStages];
  uint64_t mma_done;
  uint64_t slices;     // this CTA's K slice of the token rows and of gamma landed
  uint64_t loads_out;  // the norm warps' loads of x are in flight
  uint32_t tmem_base;
  int abort;
  float rstd[kDmTokens];
};

// Shared-memory plan of one launch (byte offsets from the 1024-aligned
// base): the ring, a in the B layout, the K slices of the token rows and of
// gamma (kbl_max * 128 bytes each), the control block.
struct DmPlan {
  int stages;
  uint32_t b_off, xk_off, gk_off, ctrl_off;
  size_t bytes;  // dynamic shared memory to request
};

__host__ __device__ inline DmPlan dm_plan(int kbl_max) {
  DmPlan p;
  const uint32_t b_bytes = static_cast<uint32_t>(kbl_max) * kDmBBlock;
  const uint32_t slice = static_cast<uint32_t>(kbl_max) * 128u;
  const uint32_t fixed = 1024 + b_bytes + (kDmTokens + 1) * slice + static_cast<uint32_t>(sizeof(DmCtrl)) + 64;
  int st = fixed >= kDmSmemLimit ? 0 : static_cast<int>((kDmSmemLimit - fixed) / kDmStage);
  if (st > kDmMaxStages) st = kDmMaxStages;
  if (st > kbl_max) st = kbl_max;
  p.stages = st;
  p.b_off = static_cast<uint32_t>(st) * kDmStage;
  p.xk_off = p.b_off + b_bytes;
  p.gk_off = p.xk_off + kDmTokens * slice;
  p.ctrl_off = p.gk_off + slice;
  p.bytes = 1024 + p.ctrl_off + sizeof(DmCtrl);
  return p;
}

__device__ __forceinline__ void tmem_ld_4cols(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier 2 over warps 1-4 (128 threads) with the AND of every
// thread's `ok`: the same answer in all of them.
__device__ __forceinline__ bool epi_sync_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 2, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(ok))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int MODE, bool GAMMA>
__global__ void __launch_bounds__(kDmThreads, 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap map_w, const __nv_bfloat16* __restrict__ x,
                      const __nv_bfloat16* __restrict__ gamma, int T, int K, int N, int split,
                      int kb_total, float inv_d, float eps, __nv_bfloat16* __restrict__ out,
                      float4* __restrict__ part, uint64_t* __restrict__ flags, uint64_t epoch) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tile = static_cast<int>(blockIdx.x) / split;
  const int rank = static_cast<int>(blockIdx.x) % split;
  const int kb0 = rank * kb_total / split;
  const int kb1 = (rank + 1) * kb_total / split;
  const int kbl = kb1 - kb0;
  const int kbl_max = (kb_total + split - 1) / split;
  const DmPlan plan = dm_plan(kbl_max);
  const int stages = plan.stages;
  DmCtrl* ctrl = reinterpret_cast<DmCtrl*>(smem + plan.ctrl_off);
  const uint32_t b_base = base + plan.b_off;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctrl->mma_done), 1);
    mbar_init(smem_u32(&ctrl->slices), 1);
    mbar_init(smem_u32(&ctrl->loads_out), 128);
    ctrl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl->tmem_base), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_launch_dependents();
  const uint32_t tmem = ctrl->tmem_base;
  volatile int* abort = &ctrl->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_w);
      grid_dependency_wait();  // x, gamma and W may come from the previous kernel
      // this CTA's K slice of the token rows and of gamma first, then (once
      // the norm warps' loads of x are out) the weight: x's requests are not
      // queued behind 16 KB stages of W
      const int kspan = min(kbl * 64, K - kb0 * 64);
      const uint32_t slice_bytes = static_cast<uint32_t>(kspan) * 2u;
      const uint32_t sbar = smem_u32(&ctrl->slices);
      if (RNL_DCHECK(&g_err_decmma, kspan > 0 && kbl <= (kb_total + split - 1) / split && T <= kDmTokens, 96)) {
        mbar_arrive_expect_tx(sbar, slice_bytes * static_cast<uint32_t>(T + (GAMMA ? 1 : 0)));
        for (int t = 0; t < T; ++t)
          bulk_copy_g2s(base + plan.xk_off + static_cast<uint32_t>(t) * kbl_max * 128u,
                        x + static_cast<int64_t>(t) * K + kb0 * 64, slice_bytes, sbar);
        if (GAMMA) bulk_copy_g2s(base + plan.gk_off, gamma + kb0 * 64, slice_bytes, sbar);
      }
      mbar_wait(smem_u32(&ctrl->loads_out), 0u, abort, &g_err_decmma, 97);
      uint32_t stage = 0, phase = 0;
      for (int j = 0; j < kbl; ++j) {
        if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_decmma, 91)) break;
        if (!RNL_DCHECK(&g_err_decmma, stage < static_cast<uint32_t>(stages) && kb0 + j < kb_total, 92)) break;
        const uint32_t bar = smem_u32(&ctrl->full[stage]);
        mbar_arrive_expect_tx(bar, kDmStage);
        tma_load_2d(base + stage * kDmStage, &map_w, bar, (kb0 + j) * 64, tile * 128);
        if (++stage == static_cast<uint32_t>(stages)) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else {
    const int w4 = warp - 1;  // 0..3
    const int tid = threadIdx.x - 32;
    grid_dependency_wait();   // x comes from the previous kernel
    // ---- rstd of token row w4: all of K, 16 loads a lane in flight at once
    //      (a row of up to 4096 elements in one round trip); the producer
    //      holds the weight back until every warp's first loads are out
    {
      const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(w4) * K);
      const int nvec = w4 < T ? K / 8 : 0;
      float ss = 0.f;
      for (int v0 = 0; v0 < (w4 < T ? nvec : 1); v0 += 32 * 16) {
        uint4 u[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int v = v0 + 32 * q + lane;
          u[q] = v < nvec ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (v0 == 0) mbar_arrive(smem_u32(&ctrl->loads_out));
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const uint32_t wd[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(wd[i] << 16), hi = __uint_as_float(wd[i] & 0xFFFF0000u);
            ss = MODE == 0 ? fmaf(lo, lo, ss) : fmaf(lo * lo, inv_d, ss);
            ss = MODE == 0 ? fmaf(hi, hi, ss) : fmaf(hi * hi, inv_d, ss);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0 && w4 < T) ctrl->rstd[w4] = MODE == 0 ? rsqrtf(ss * inv_d + eps) : 1.0f / sqrtf(ss + eps);
    }
    // ---- the zero rows T .. 15 of every k-block of a (no loads)
    for (int i = tid; i < kbl * (kDmN - T) * 8; i += 128) {
      const int j = i / ((kDmN - T) * 8), t = T + (i / 8) % (kDmN - T), c = i % 8;
      const uint32_t off = static_cast<uint32_t>(j) * kDmBBlock + static_cast<uint32_t>(t >> 3) * 1024u +
                           static_cast<uint32_t>(t & 7) * 128u + (static_cast<uint32_t>(c ^ (t & 7)) << 4);
      *reinterpret_cast<uint4*>(smem + plan.b_off + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    // ---- rows 0 .. T-1 of this CTA's k-blocks of a in the B layout, from
    //      the K slices in shared memory: item (j, c) is 8 elements of gamma
    //      and of each token row; k-block j at b_base + j * 2 KB, row t at
    //      (t / 8) * 1024 + (t % 8) * 128, 16-byte chunk c at position
    //      c ^ (t % 8) (128-byte swizzle)
    float r[kDmTokens];
#pragma unroll
    for (int t = 0; t < kDmTokens; ++t) r[t] = t < T ? ctrl->rstd[t] : 0.f;
    const bool landed = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctrl->slices), 0u, abort, &g_err_decmma, 98));
    const uint4* xk = reinterpret_cast<const uint4*>(smem + plan.xk_off);  // [t][kbl_max * 8]
    const uint4* gk = reinterpret_cast<const uint4*>(smem + plan.gk_off);
    for (int i = tid; landed && i < kbl * 8; i += 128) {
      const int j = i / 8, c = i % 8;
      const bool in_k = (kb0 + j) * 64 + c * 8 < K;
      const uint4 g = GAMMA && in_k ? gk[i] : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int t = 0; t < kDmTokens; ++t) {
        if (t >= T) break;
        const uint4 u = in_k ? xk[t * kbl_max * 8 + i] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t xw[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float lo = __fmul_rn(__uint_as_float(xw[q] << 16), r[t]);
          float hi = __fmul_rn(__uint_as_float(xw[q] & 0xFFFF0000u), r[t]);
          if (GAMMA) {
            lo = __fmul_rn(lo, __uint_as_float(gw[q] << 16));
            hi = __fmul_rn(hi, __uint_as_float(gw[q] & 0xFFFF0000u));
          }
          o[q] = pack_bf16x2(lo, hi);
        }
        const uint32_t off = static_cast<uint32_t>(j) * kDmBBlock + static_cast<uint32_t>(t >> 3) * 1024u +
                             static_cast<uint32_t>(t & 7) * 128u + (static_cast<uint32_t>(c ^ (t & 7)) << 4);
        *reinterpret_cast<uint4*>(smem + plan.b_off + off) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    fence_proxy_async_shared();  // the generic-proxy writes of a, seen by the tensor core
    asm volatile("bar.sync 1, 128;" ::: "memory");

    if (warp == 1) {
      // -------------------------------------------------------------- MMA
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16(128, kDmN);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int j = 0; j < kbl && ok; ++j) {
          if (!mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_decmma, 93)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = desc_kmajor_sw128(base + stage * kDmStage);
          const uint64_t bdesc = desc_kmajor_sw128(b_base + static_cast<uint32_t>(j) * kDmBBlock);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&ctrl->empty[stage]));
          if (++stage == static_cast<uint32_t>(stages)) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(smem_u32(&ctrl->mma_done));
      }
      __syncwarp();
    }
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // the TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    const int n = tile * 128 + row;
    const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctrl->mma_done), 0u, abort, &g_err_decmma, 94));
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (got) {
      tc_fence_after();
      tmem_ld_4cols(tmem + (static_cast<uint32_t>(quarter * 32) << 16), v);
    }
    // partial sums of rank q (1 .. S-1) of tile g: part[(g * 7 + q - 1) * 128 + row];
    // its flag: flags[g * 7 + q - 1].  Every barrier below is reached by all
    // four warps, and carries the AND of their outcomes.
    if (rank > 0) {
      const int slot = tile * (kDmMaxSplit - 1) + rank - 1;
      if (got) {
        part[static_cast<int64_t>(slot) * 128 + row] = make_float4(v[0], v[1], v[2], v[3]);
        __threadfence();
      }
      if (epi_sync_and(got) && tid == 0) flag_release(flags + slot, epoch);
    } else {
      bool all = got;
      for (int q = 1; q < split && all; ++q)
        all = flag_wait(flags + tile * (kDmMaxSplit - 1) + q - 1, epoch, abort, &g_err_decmma, 95);
      // past this barrier every thread has seen the flags (or failed)
      if (epi_sync_and(all)) {
        for (int q = 1; q < split; ++q) {
          const float4 p = part[static_cast<int64_t>(tile * (kDmMaxSplit - 1) + q - 1) * 128 + row];
          v[0] += p.x;
          v[1] += p.y;
          v[2] += p.z;
          v[3] += p.w;
        }
        if (n < N) {
#pragma unroll
          for (int t = 0; t < kDmTokens; ++t)
            if (t < T) out[static_cast<int64_t>(t) * N + n] = __float2bfloat16_rn(v[t]);
        }
        // the flags go back to 0, so that a replay of this launch (same
        // epoch, in a CUDA graph) waits for its own
        if (tid < split - 1) flags[tile * (kDmMaxSplit - 1) + tid] = 0;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

// CTAs per weight tile: one CTA per SM if the tiles allow (every CTA of the
// grid resident at once: rank 0 waits for the others' flags), at most 8; 0
// when the shape does not fit.
int dm_split(int64_t tiles, int kb_total, int sm_count) {
  int64_t s = tiles > 0 ? sm_count / tiles : 0;
  if (s < 1) s = 1;
  if (s > kDmMaxSplit) s = kDmMaxSplit;
  if (s > kb_total) s = kb_total;
  if (s > 1 && tiles * s > sm_count) return 0;
  // the k-blocks of a must leave room for a ring of at least two stages
  while (dm_plan(static_cast<int>((kb_total + s - 1) / s)).stages < 2) {
    if (s >= kDmMaxSplit || s >= kb_total || tiles * (s + 1) > sm_count) return 0;
    ++s;
  }
  return static_cast<int>(s);
}

// workspace bytes of the K split: partial sums, then the flags
size_t dm_part_bytes(int64_t tiles) { return static_cast<size_t>(tiles) * (kDmMaxSplit - 1) * 128 * 16; }
size_t dm_ws_bytes(int64_t tiles) { return dm_part_bytes(tiles) + static_cast<size_t>(tiles) * (kDmMaxSplit - 1) * 8; }

template <int MODE, bool GAMMA>
rnl_status launch_dm(const void* x, const void* gamma, const void* W, int64_t T, int64_t K, int64_t N,
                     float eps, void* out, void* ws, size_t ws_bytes, const DeviceInfo& dev, cudaStream_t s) {
  const int kb_total = static_cast<int>((K + 63) / 64);
  const int64_t tiles = (N + 127) / 128;
  const int split = dm_split(tiles, kb_total, dev.sm_count);
  if (split == 0) return RNL_ERR_UNSUPPORTED;
  if (split > 1 && (ws == nullptr || ws_bytes < dm_ws_bytes(tiles))) return RNL_ERR_WORKSPACE;
  const DmPlan plan = dm_plan((kb_total + split - 1) / split);
  auto kern = decode_mma_kernel<MODE, GAMMA>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, plan.bytes) != RNL_OK)
    return RNL_ERR_LAUNCH;
  CUtensorMap mw;
  rnl_status st = make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, K, N, K * 2, 64, 128);
  if (st != RNL_OK) return st;
  float4* part = static_cast<float4*>(ws);
  uint64_t* flags = split > 1 ? reinterpret_cast<uint64_t*>(static_cast<char*>(ws) + dm_part_bytes(tiles)) : nullptr;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * split), 1, 1);
  cfg.blockDim = dim3(kDmThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  trace_before(s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mw, static_cast<const __nv_bfloat16*>(x),
                                           static_cast<const __nv_bfloat16*>(gamma), static_cast<int>(T),
                                           static_cast<int>(K), static_cast<int>(N), split, kb_total, inv_d,
                                           eps, static_cast<__nv_bfloat16*>(out), part, flags,
                                           next_flag_epoch());
  trace_after(s, "decode_gemv_mma");
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

}  // namespace

bool decode_mma_fits(int64_t T, int64_t K, int64_t N, int sm_count) {
  if (T < 1 || T > kDmTokens || K < 64 || K % 8 != 0 || N < 1 || K > (int64_t{1} << 30)) return false;
  return dm_split((N + 127) / 128, static_cast<int>((K + 63) / 64), sm_count) > 0;
}

size_t decode_mma_workspace_bytes(int64_t N) { return dm_ws_bytes((N + 127) / 128); }

rnl_status launch_decode_mma(const void* x, const void* gamma, const void* W, int64_t T, int64_t K, int64_t N,
                             float eps, int mode, void* out, void* ws, size_t ws_bytes, cudaStream_t s) {
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  if (!decode_mma_fits(T, K, N, dev.sm_count)) return RNL_ERR_UNSUPPORTED;
  if (mode == RNL_NORM_RSQRT)
    return gamma ? launch_dm<0, true>(x, gamma, W, T, K, N, eps, out, ws, ws_bytes, dev, s)
                 : launch_dm<0, false>(x, gamma, W, T, K, N, eps, out, ws, ws_bytes, dev, s);
  return gamma ? launch_dm<1, true>(x, gamma, W, T, K, N, eps, out, ws, ws_bytes, dev, s)
               : launch_dm<1, false>(x, gamma, W, T, K, N, eps, out, ws, ws_bytes, dev, s);
}

rnl_status read_clear_error_decmma(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_decmma, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_decmma, &zero, sizeof zero) != cudaSuccess) return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
