// gemm_pair.cu -- the C stage on CTA pairs: out = epilogue(A[M,K] @ B[N,K]^T)
// with tcgen05.mma.cta_group::2 (AT-09 "Linear" of the AT-10 pattern page,
// sec. 4: matmul(x, w, dtype, b_trans=True), W stored [N, K]).
//
// Two CTAs of a cluster (on two SMs) compute one 256 x BN output tile: each
// holds its own 128 rows of A and one half (BN/2 rows) of the B tile in
// shared memory, and one thread of the even CTA issues M=256 MMAs that read
// both CTAs' operands; each CTA's TMEM receives the accumulator of its own
// 128 rows over all BN columns.  Per SM and k-block the operands are
// 16 KB of A + BN*64 B of B instead of 16 KB + BN*128 B on one SM, so the
// L2 -> SM traffic per flop drops by 30-40 % and the shared memory holds
// more stages (7 or 8) of the pipeline.
//
// Roles per CTA (320 threads): warp 0 TMA producer (both CTAs load their own
// A rows and B half; the loads complete on the even CTA's "full" barrier),
// warp 1 TMEM allocation (pair-wide) and, in the even CTA, the MMA issuer,
// warps 2-9 epilogue of the CTA's own 128 rows.  The MMA completion is
// multicast to both CTAs' "empty" and "accumulator full" barriers; the odd
// CTA's epilogue warps arrive on the even CTA's "accumulator empty" barrier.
// Every wait is bounded (ptx.cuh).
//
// Work list (persistent, one CTA pair per two SMs): with P pairs and T tiles,
// the first floor(T/P) * P tiles run data-parallel (pair p takes tiles p,
// p+P, ...).  The R = T mod P tiles left over would leave most pairs idle in a
// last partial wave, so each of them is cut along K into S = P / R pieces and
// every pair takes one piece: its partial sums (fp32, or exact int32 in the
// integer mode) go to a workspace, and gemm_pair_fixup_kernel adds the S
// pieces of each tile in a fixed order and applies the epilogue.
#include <cuda_bf16.h>

#include <cstdlib>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

using namespace gemm;

__device__ unsigned int g_err_pair;

constexpr int kEpiWarps = 8;
constexpr int kMaxSplits = 16;  // K pieces per leftover tile (partial volume vs tail length)

template <int BN>
struct PairTile {
  static constexpr int kBHalf = BN / 2;                  // B rows per CTA
  static constexpr uint32_t kBBytes = kBHalf * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages =
      static_cast<int>((kSmemLimit - 1024 - 256) / kStageBytes) < kMaxStages
          ? static_cast<int>((kSmemLimit - 1024 - 256) / kStageBytes)
          : kMaxStages;
};

struct __align__(8) PairCtrl {
  uint64_t full[kMaxStages];   // even CTA: both CTAs' loads of a stage
  uint64_t empty[kMaxStages];  // each CTA: its stage consumed by the pair MMA
  uint64_t tmem_full[2];       // each CTA: accumulator ready
  uint64_t tmem_empty[2];      // even CTA: both CTAs' epilogues drained it
  uint32_t tmem_base;
  int abort;
};

template <int BN>
constexpr size_t pair_smem_bytes() {
  return 1024 + static_cast<size_t>(PairTile<BN>::kStages) * PairTile<BN>::kStageBytes +
         sizeof(PairCtrl);
}

struct Work {
  int tile;  // index in the grouped tile order
  int kb0;   // k-block range [kb0, kb1)
  int kb1;
  int slot;  // partial-sum slot, or -1 for a whole tile written to the output
};

// Item `it` of pair `pair`'s work list (identical in every role).
__device__ __forceinline__ Work work_item(int pair, int it, int num_pairs, int dp_waves,
                                          int splits, int num_kb) {
  Work w;
  if (it < dp_waves) {
    w.tile = pair + it * num_pairs;
    w.kb0 = 0;
    w.kb1 = num_kb;
    w.slot = -1;
  } else {
    const int j = pair % splits;
    w.tile = dp_waves * num_pairs + pair / splits;
    w.kb0 = static_cast<int>((static_cast<int64_t>(j) * num_kb) / splits);
    w.kb1 = static_cast<int>((static_cast<int64_t>(j + 1) * num_kb) / splits);
    w.slot = splits > 1 ? pair : -1;
  }
  return w;
}

template <int EPI, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b, int M, int N, int K, int group_m,
                     int dp_waves, int tail_tiles, int splits, void* __restrict__ out,
                     const float* __restrict__ row_scale, const float* __restrict__ col_scale,
                     uint32_t* __restrict__ partial, const __nv_bfloat16* __restrict__ bias) {
  constexpr bool kInt = (EPI == static_cast<int>(Epi::kDequantBf16) ||
                         EPI == static_cast<int>(Epi::kInt32));
  constexpr int kStages = PairTile<BN>::kStages;
  constexpr uint32_t kStageBytes = PairTile<BN>::kStageBytes;
  constexpr int kBHalf = PairTile<BN>::kBHalf;
  constexpr uint32_t kTmemCols = 512;
  constexpr int kColsPerEpiWarp = BN / 2;
  constexpr int kGroups = kColsPerEpiWarp / 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  PairCtrl* ctrl = reinterpret_cast<PairCtrl*>(smem + kStages * kStageBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int num_m = (M + 2 * BM - 1) / (2 * BM);  // 256-row blocks
  const int num_n = (N + BN - 1) / BN;
  const int num_kb = (K + BK - 1) / BK;
  const int n_items = dp_waves + (pair < tail_tiles * splits ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->tmem_full[b]), 1);
      mbar_init(smem_u32(&ctrl->tmem_empty[b]), 2 * kEpiWarps);
    }
    ctrl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&ctrl->tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised and the pair's TMEM allocated
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  // set-up above overlaps the previous kernel (programmatic dependent launch)
  grid_launch_dependents();
  grid_dependency_wait();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort = &ctrl->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_a);
      tma_prefetch_map(&map_b);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int it = 0; it < n_items && ok; ++it) {
        const Work w = work_item(pair, it, num_pairs, dp_waves, splits, num_kb);
        int mb, nb;
        tile_coords(w.tile, num_m, num_n, group_m, mb, nb);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait_cluster(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_pair, 21)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          const uint32_t full_local = smem_u32(&ctrl->full[stage]);
          const uint32_t full_even = mapa_shared(full_local, 0);
          if (rank == 0) mbar_arrive_expect_tx(full_local, 2 * kStageBytes);
          tma_load_2d_pair(sa, &map_a, full_even, kb * BK, mb * 2 * BM + static_cast<int>(rank) * BM);
          tma_load_2d_pair(sa + kABytes, &map_b, full_even, kb * BK,
                           nb * BN + static_cast<int>(rank) * kBHalf);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(2 * BM, BN);
      uint32_t stage = 0, phase = 0, unit = 0;
      bool ok = true;
      for (int it = 0; it < n_items && ok; ++it) {
        const Work w = work_item(pair, it, num_pairs, dp_waves, splits, num_kb);
        const int kb_per_unit = kInt ? kChunkKBlocks : (w.kb1 - w.kb0);
        const int units = (w.kb1 - w.kb0 + kb_per_unit - 1) / kb_per_unit;
        for (int u = 0; u < units && ok; ++u, ++unit) {
          const uint32_t buf = unit & 1u;
          const uint32_t use = unit >> 1;
          if (!mbar_wait_cluster(smem_u32(&ctrl->tmem_empty[buf]), (use & 1u) ^ 1u, abort,
                                 &g_err_pair, 22)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kAccStride;
          const int kb0 = w.kb0 + u * kb_per_unit;
          const int kb1 = min(w.kb1, kb0 + kb_per_unit);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_cluster(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_pair, 23)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = base + stage * kStageBytes;
            const uint64_t adesc = desc_kmajor_sw128(sa);
            const uint64_t bdesc = desc_kmajor_sw128(sa + kABytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              umma_bf16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                             (kb > kb0 || k > 0) ? 1u : 0u);
            umma_commit_pair(smem_u32(&ctrl->empty[stage]), 0x3);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair(smem_u32(&ctrl->tmem_full[buf]), 0x3);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int half = ew >> 2;      // which half of the BN columns
    const int row_local = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t empty_even_0 = mapa_shared(smem_u32(&ctrl->tmem_empty[0]), 0);
    const uint32_t empty_even_1 = mapa_shared(smem_u32(&ctrl->tmem_empty[1]), 0);
    uint32_t unit = 0;
    bool ok = true;
    for (int it = 0; it < n_items && ok; ++it) {
      const Work w = work_item(pair, it, num_pairs, dp_waves, splits, num_kb);
      const int kb_per_unit = kInt ? kChunkKBlocks : (w.kb1 - w.kb0);
      const int units = (w.kb1 - w.kb0 + kb_per_unit - 1) / kb_per_unit;
      // partial slot of this CTA: [slot][rank][128 rows][BN] 32-bit words
      uint32_t* prow = w.slot >= 0 ? partial + ((static_cast<int64_t>(w.slot) * 2 + rank) * BM + row_local) * BN
                                   : nullptr;
      int mb, nb;
      tile_coords(w.tile, num_m, num_n, group_m, mb, nb);
      const int64_t m = static_cast<int64_t>(mb) * 2 * BM + rank * BM + row_local;
      const int n_base = nb * BN + half * kColsPerEpiWarp;
      const bool row_ok = m < M;
      float rs = 0.f;
      if ((EPI == static_cast<int>(Epi::kRowScaleF32) ||
           EPI == static_cast<int>(Epi::kDequantBf16)) && row_ok)
        rs = __ldg(row_scale + m);
      int iacc[kInt ? kGroups : 1][kInt ? 32 : 1];
      if (kInt) {
#pragma unroll
        for (int c = 0; c < (kInt ? kGroups : 1); ++c)
#pragma unroll
          for (int j = 0; j < (kInt ? 32 : 1); ++j) iacc[c][j] = 0;
      }
      for (int u = 0; u < units; ++u, ++unit) {
        const uint32_t buf = unit & 1u;
        const uint32_t use = unit >> 1;
        const bool got = mbar_wait_cluster(smem_u32(&ctrl->tmem_full[buf]), use & 1u, abort,
                                           &g_err_pair, 24);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kGroups; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(tmem_base + lane_addr + buf * kAccStride + half * kColsPerEpiWarp + c * 32, r);
          tmem_ld_wait();
          const int n0 = n_base + c * 32;
          if constexpr (kInt) {
#pragma unroll
            for (int j = 0; j < 32; ++j) iacc[c][j] += __float2int_rn(__uint_as_float(r[j]));
          } else if (prow != nullptr) {
            uint4* dst = reinterpret_cast<uint4*>(prow + half * kColsPerEpiWarp + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          } else if constexpr (EPI == static_cast<int>(Epi::kBf16)) {
            if (row_ok) {
              if (bias != nullptr)
                store_bf16_bias_32(out, m, n0, N, r, bias);
              else
                store_bf16_32(out, m, n0, N, r);
            }
          } else {
            if (row_ok) store_f32_scaled_32(out, m, n0, N, r, rs);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(smem_u32(&ctrl->tmem_empty[buf]));
          else
            mbar_arrive_cluster(buf ? empty_even_1 : empty_even_0);
        }
      }
      if (!ok) break;
      if constexpr (kInt) {
        if (prow != nullptr) {
#pragma unroll
          for (int c = 0; c < kGroups; ++c) {
            int4* dst = reinterpret_cast<int4*>(prow + half * kColsPerEpiWarp + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_int4(iacc[c][4 * j], iacc[c][4 * j + 1], iacc[c][4 * j + 2], iacc[c][4 * j + 3]);
          }
        } else if (row_ok) {
#pragma unroll
          for (int c = 0; c < kGroups; ++c) {
            if constexpr (EPI == static_cast<int>(Epi::kInt32))
              store_i32_32(out, m, n_base + c * 32, N, iacc[c]);
            else
              store_dequant_32(out, m, n_base + c * 32, N, iacc[c], rs, col_scale, bias);
          }
        }
      }
    }
  }

  // no CTA of the pair leaves (or frees TMEM) while its peer may still signal
  // its barriers or the pair MMA may still read its shared memory
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Adds the S partial pieces of each split tile (in piece order) and applies
// the epilogue.  Thread = (tile, 256-row position, 4 consecutive columns);
// the piece loads are unrolled so several are in flight per thread.
template <int EPI, int BN>
__global__ void __launch_bounds__(256)
    gemm_pair_fixup_kernel(int M, int N, int group_m, int dp_tiles, int tail_tiles, int splits,
                           const uint32_t* __restrict__ partial, void* __restrict__ out,
                           const float* __restrict__ row_scale, const float* __restrict__ col_scale,
                           const __nv_bfloat16* __restrict__ bias) {
  constexpr bool kInt = (EPI == static_cast<int>(Epi::kDequantBf16) ||
                         EPI == static_cast<int>(Epi::kInt32));
  constexpr int kQuadsPerRow = BN / 4;
  grid_dependency_wait();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(tail_tiles) * 2 * BM * kQuadsPerRow;
  if (idx >= total) return;
  const int q = static_cast<int>(idx % kQuadsPerRow);
  const int row = static_cast<int>((idx / kQuadsPerRow) % (2 * BM));  // 0..255 in the pair tile
  const int r = static_cast<int>(idx / (kQuadsPerRow * 2 * BM));
  const int num_m = (M + 2 * BM - 1) / (2 * BM);
  const int num_n = (N + BN - 1) / BN;
  int mb, nb;
  tile_coords(dp_tiles + r, num_m, num_n, group_m, mb, nb);
  const int64_t m = static_cast<int64_t>(mb) * 2 * BM + row;
  const int n0 = nb * BN + q * 4;
  if (m >= M || n0 >= N) return;
  const int rank = row / BM;
  const int row_local = row % BM;
  // word offset of this thread's 4 columns in piece sidx
  const int64_t stride = static_cast<int64_t>(2) * BM * BN;  // words per piece
  const uint4* src = reinterpret_cast<const uint4*>(
      partial + ((static_cast<int64_t>(r) * splits * 2 + rank) * BM + row_local) * BN + q * 4);
  const int64_t vstride = stride / 4;  // in uint4
  uint4 acc_bits;
  if constexpr (kInt) {
    int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
    int sidx = 0;
    for (; sidx + 4 <= splits; sidx += 4) {
      const uint4 v0 = src[(sidx + 0) * vstride], v1 = src[(sidx + 1) * vstride];
      const uint4 v2 = src[(sidx + 2) * vstride], v3 = src[(sidx + 3) * vstride];
      a0 += static_cast<int>(v0.x) + static_cast<int>(v1.x) + static_cast<int>(v2.x) + static_cast<int>(v3.x);
      a1 += static_cast<int>(v0.y) + static_cast<int>(v1.y) + static_cast<int>(v2.y) + static_cast<int>(v3.y);
      a2 += static_cast<int>(v0.z) + static_cast<int>(v1.z) + static_cast<int>(v2.z) + static_cast<int>(v3.z);
      a3 += static_cast<int>(v0.w) + static_cast<int>(v1.w) + static_cast<int>(v2.w) + static_cast<int>(v3.w);
    }
    for (; sidx < splits; ++sidx) {
      const uint4 v = src[sidx * vstride];
      a0 += static_cast<int>(v.x);
      a1 += static_cast<int>(v.y);
      a2 += static_cast<int>(v.z);
      a3 += static_cast<int>(v.w);
    }
    const int a[4] = {a0, a1, a2, a3};
    if constexpr (EPI == static_cast<int>(Epi::kInt32)) {
      int* orow = static_cast<int*>(out) + m * N;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n0 + j < N) orow[n0 + j] = a[j];
    } else {
      const float xs = __ldg(row_scale + m);
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(out) + m * N;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n0 + j < N) {
          float v = static_cast<float>(a[j]) * (xs * __ldg(col_scale + n0 + j));
          if (bias != nullptr) v = __fadd_rn(v, __bfloat162float(bias[n0 + j]));
          orow[n0 + j] = __float2bfloat16_rn(v);
        }
    }
    (void)acc_bits;
  } else {
    // fp32 partial sums added in piece order (pairwise within a group of
    // four pieces, then sequentially), the same order on every run
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int sidx = 0;
    for (; sidx + 4 <= splits; sidx += 4) {
      const uint4 v0 = src[(sidx + 0) * vstride], v1 = src[(sidx + 1) * vstride];
      const uint4 v2 = src[(sidx + 2) * vstride], v3 = src[(sidx + 3) * vstride];
      a0 += (__uint_as_float(v0.x) + __uint_as_float(v1.x)) + (__uint_as_float(v2.x) + __uint_as_float(v3.x));
      a1 += (__uint_as_float(v0.y) + __uint_as_float(v1.y)) + (__uint_as_float(v2.y) + __uint_as_float(v3.y));
      a2 += (__uint_as_float(v0.z) + __uint_as_float(v1.z)) + (__uint_as_float(v2.z) + __uint_as_float(v3.z));
      a3 += (__uint_as_float(v0.w) + __uint_as_float(v1.w)) + (__uint_as_float(v2.w) + __uint_as_float(v3.w));
    }
    for (; sidx < splits; ++sidx) {
      const uint4 v = src[sidx * vstride];
      a0 += __uint_as_float(v.x);
      a1 += __uint_as_float(v.y);
      a2 += __uint_as_float(v.z);
      a3 += __uint_as_float(v.w);
    }
    float a[4] = {a0, a1, a2, a3};
    if constexpr (EPI == static_cast<int>(Epi::kBf16)) {
      if (bias != nullptr) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (n0 + j < N) a[j] = __fadd_rn(a[j], __bfloat162float(bias[n0 + j]));
      }
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(out) + m * N;
      if (n0 + 4 <= N && (N & 3) == 0) {
        uint2 o;
        o.x = bf16x2_bits(a[0], a[1]);
        o.y = bf16x2_bits(a[2], a[3]);
        *reinterpret_cast<uint2*>(orow + n0) = o;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (n0 + j < N) orow[n0 + j] = __float2bfloat16_rn(a[j]);
      }
    } else {
      const float rs = __ldg(row_scale + m);
      float* orow = static_cast<float*>(out) + m * N;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n0 + j < N) orow[n0 + j] = a[j] * rs;
    }
    (void)acc_bits;
  }
}

// Work-list shape for T tiles on P pairs: full data-parallel waves, then the
// leftover tiles cut along K into `splits` pieces (one per pair).
struct Plan {
  int dp_waves = 0;
  int tail_tiles = 0;
  int splits = 1;
};

Plan make_plan(int64_t tiles, int pairs, int num_kb) {
  Plan pl;
  pl.dp_waves = static_cast<int>(tiles / pairs);
  pl.tail_tiles = static_cast<int>(tiles - static_cast<int64_t>(pl.dp_waves) * pairs);
  if (pl.tail_tiles > 0) {
    int sp = pairs / pl.tail_tiles;
    if (sp > kMaxSplits) sp = kMaxSplits;
    if (sp > num_kb) sp = num_kb;
    if (sp * pl.tail_tiles > kMaxPartialSlots) sp = kMaxPartialSlots / pl.tail_tiles;
    pl.splits = sp < 1 ? 1 : sp;
  }
  return pl;
}

template <int EPI, int BN>
rnl_status launch_pair_bn(const GemmArgs& g, const DeviceInfo& dev, int max_pairs, cudaStream_t s,
                          const char* name) {
  static bool attr_set[64] = {};
  auto kern = gemm_pair_kernel<EPI, BN>;
  const size_t smem = pair_smem_bytes<BN>();
  if (!attr_set[dev.device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return RNL_ERR_LAUNCH;
    attr_set[dev.device] = true;
  }
  CUtensorMap ma, mb;
  rnl_status st = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.A, g.K, g.M, g.K * 2, BK, BM);
  if (st != RNL_OK) return st;
  st = make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.B, g.K, g.N, g.K * 2, BK,
                   PairTile<BN>::kBHalf);
  if (st != RNL_OK) return st;
  const int num_m = static_cast<int>((g.M + 2 * BM - 1) / (2 * BM));
  const int num_kb = static_cast<int>((g.K + BK - 1) / BK);
  const int64_t tiles = static_cast<int64_t>(num_m) * ((g.N + BN - 1) / BN);
  const int pairs = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
  Plan pl = make_plan(tiles, pairs, num_kb);
  if (pl.splits > 1 && (g.partial_ws == nullptr ||
                        g.partial_ws_bytes < static_cast<size_t>(pl.tail_tiles) * pl.splits * 2 *
                                                 BM * BN * 4))
    pl.splits = 1;  // no room for partial sums: the leftover tiles run whole
  const int group_m = (g.M * g.K * 2 <= (int64_t{48} << 20)) ? num_m : (num_m < 4 ? num_m : 4);

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  trace_before(s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, static_cast<int>(g.M),
                                     static_cast<int>(g.N), static_cast<int>(g.K), group_m,
                                     pl.dp_waves, pl.tail_tiles, pl.splits, g.out, g.row_scale,
                                     g.col_scale, static_cast<uint32_t*>(g.partial_ws),
                                     static_cast<const __nv_bfloat16*>(g.bias));
  trace_after(s, name);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  if (pl.splits > 1) {
    const int64_t threads = static_cast<int64_t>(pl.tail_tiles) * 2 * BM * (BN / 4);
    cudaLaunchConfig_t fc = {};
    fc.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256), 1, 1);
    fc.blockDim = dim3(256, 1, 1);
    fc.stream = s;
    fc.attrs = &attr[1];
    fc.numAttrs = 1;
    trace_before(s);
    e = cudaLaunchKernelEx(&fc, gemm_pair_fixup_kernel<EPI, BN>, static_cast<int>(g.M),
                           static_cast<int>(g.N), group_m, pl.dp_waves * pairs, pl.tail_tiles,
                           pl.splits, static_cast<const uint32_t*>(g.partial_ws), g.out,
                           g.row_scale, g.col_scale, static_cast<const __nv_bfloat16*>(g.bias));
    trace_after(s, "gemm_pair_fixup");
    if (e != cudaSuccess) {
      cudaGetLastError();
      return RNL_ERR_LAUNCH;
    }
  }
  return RNL_OK;
}

// Largest number of CTA pairs that can be resident at once.
int resident_pairs(const DeviceInfo& dev) {
  static int cached[64] = {};
  if (cached[dev.device] > 0) return cached[dev.device];
  auto kern = gemm_pair_kernel<0, 256>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(pair_smem_bytes<256>())) == cudaSuccess) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pair_smem_bytes<256>();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n <= 0) n = dev.sm_count / 2;
  cached[dev.device] = n;
  return n;
}

template <int EPI>
rnl_status launch_pair_epi(const GemmArgs& g, const DeviceInfo& dev, cudaStream_t s,
                           const char* name) {
  const int pairs = resident_pairs(dev);
  int bn = 256;  // 128- and 192-wide pair tiles measured slower per flop than one-CTA tiles
  if (const char* e = std::getenv("RNL_GEMM_BN")) {
    const int v = std::atoi(e);
    if (v == 128 || v == 192 || v == 256) bn = v;
  }
  switch (bn) {
    case 128: return launch_pair_bn<EPI, 128>(g, dev, pairs, s, name);
    case 192: return launch_pair_bn<EPI, 192>(g, dev, pairs, s, name);
    default: return launch_pair_bn<EPI, 256>(g, dev, pairs, s, name);
  }
}

}  // namespace

// Predicted time of the pair kernel (256-wide tiles, K-split tail) in
// microseconds, from the per-SM rate it sustained on GB300 in full waves
// (1909 TFLOP/s over 152 SMs) plus the tail piece (1/S of a tile and about
// 0.15 of a tile of fill, drain and partial stores) and the fix-up pass.
double predict_pair_us(int64_t M, int64_t N, int64_t K, int sm_count, int pairs_hint) {
  const int pairs = pairs_hint > 0 ? pairs_hint : sm_count / 2;
  const int64_t num_m = (M + 2 * BM - 1) / (2 * BM);
  const int64_t tiles = num_m * ((N + 255) / 256);
  const int p = static_cast<int>(tiles < pairs ? tiles : pairs);
  const int num_kb = static_cast<int>((K + BK - 1) / BK);
  const Plan pl = make_plan(tiles, p, num_kb);
  const double tile_us = 2.0 * BM * 256 * static_cast<double>(K) / 12.56e12 * 1e6;
  double t = pl.dp_waves * tile_us;
  if (pl.tail_tiles > 0) {
    if (pl.splits > 1) {
      const double part_bytes = static_cast<double>(pl.tail_tiles) * pl.splits * 2 * BM * 256 * 4;
      t += (1.0 / pl.splits + 0.15) * tile_us + 3.0 + 2.0 * part_bytes / 6.0e12 * 1e6;
    } else {
      t += tile_us;
    }
  }
  return t;
}

int resident_pairs_for(const DeviceInfo& dev) { return resident_pairs(dev); }

rnl_status launch_gemm_pair(const GemmArgs& g, cudaStream_t s) {
  if (g.M == 0) return RNL_OK;
  if (g.a_rstd != nullptr) return RNL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  switch (g.epi) {
    case Epi::kBf16: return launch_pair_epi<0>(g, dev, s, "gemm_pair_bf16");
    case Epi::kRowScaleF32: return launch_pair_epi<1>(g, dev, s, "gemm_pair_rowscale_f32");
    case Epi::kDequantBf16: return launch_pair_epi<2>(g, dev, s, "gemm_pair_int_dequant");
    case Epi::kInt32: return launch_pair_epi<3>(g, dev, s, "gemm_pair_int_s32");
  }
  return RNL_ERR_ARG;
}

rnl_status read_clear_error_pair(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_pair, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_pair, &zero, sizeof zero) != cudaSuccess)
    return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
