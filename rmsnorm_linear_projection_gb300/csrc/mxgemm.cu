// mxgemm.cu -- scaled_mm(x_fp8, w_fp8, FP32, x_scale, w_scale) of the MXFP8
// mode (AT-10 pattern page, sec. 4: AT-09 quant_mode mxfp8; SK-14 skeleton
// page, GMM-MXFP8: E4M3FN data, E8M0FNU scale factors) on the block-scaled
// tensor cores: out[m, n] = sum_k a[m, k] 2^(sa[m, k/32]) w[n, k] 2^(sw[n, k/32])
// with FP32 accumulation, out bf16 or fp32.
//
// tcgen05.mma kind::mxf8f6f4.block_scale multiplies E4M3 operands straight
// from shared memory (K = 32 per instruction) and applies one E8M0 scale per
// 32 elements of K to each operand row, read from tensor memory.  The page's
// 64-element scale is given to the hardware twice (two 32-element blocks of
// the same scale), which is exact.
//
// Persistent, warp-specialised, one CTA per SM, output tiles of 128 x BN:
//   warp 0     producer: per k-block of 128 codes (one 128-byte swizzle row)
//              a TMA box of A (128 x 128 B) and of B (BN x 128 B), plus the
//              k-block's scale factors by bulk copy: one 512-byte atom for the
//              128 rows of A and ceil(BN / 128) atoms for B.  An atom holds
//              the 4 scale bytes of 128 rows (row r at byte 16 (r % 32) +
//              4 (r / 32) + j, j = the 32-element block within the k-block),
//              the layout one tcgen05.cp 32x128b.warpx4 places in TMEM as
//              the MMA reads it; the front end writes the atoms in that order.
//   warp 1     allocates 512 TMEM columns (two fp32 accumulators of BN
//              columns, then slots of 32 columns for the scale factors:
//              A's atom at +0, B's at +16, +20) and one thread issues, per
//              k-block, the tcgen05.cp of the atoms and four MMAs whose
//              instruction descriptors select scale byte j = 0..3.
//   warps 2-9  epilogue: tcgen05.ld of the accumulator, bf16 or fp32 stores.
// A scale slot is rewritten only after the MMAs that read it have completed
// (the "empty" barrier of their k-block's stage), so the copies never race
// with the tensor core; a copy and the MMAs after it are issued by the same
// thread, which orders them.  Every wait is bounded (ptx.cuh).
//
// The CTA-pair form (tcgen05 cta_group::2, 256 x BN tiles on two SMs): each
// CTA stages its own 128 rows of A, half of B's BN rows, its A atom and all
// of B's atoms (every CTA's tensor core scales all BN columns); one thread of
// the even CTA copies the atoms of both CTAs into their tensor memories
// (tcgen05.cp.cta_group::2) and issues M = 256 MMAs.  Per SM and k-block the
// shared memory then moves 16 KB + BN/2 * 128 B instead of 16 KB + BN * 128 B,
// and the ring holds 7 stages instead of 5: at the FP8 rate the one-CTA form
// is bound by shared-memory traffic and ring depth.  All operands and atoms
// are TMA loads that complete on the even CTA's "full" barrier.
#include <cuda_bf16.h>

#include <atomic>
#include <cstdlib>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

using namespace gemm;

__device__ unsigned int g_err_mx;

constexpr int kMxBK = 128;                  // E4M3 codes per k-block (one 128-byte row)
constexpr uint32_t kMxABytes = BM * kMxBK;  // 16 KB
constexpr uint32_t kAtomBytes = 512;        // scale bytes of 128 rows x 4 blocks of 32

template <int BN>
struct MxTile {
  static constexpr int kAtomsB = (BN + 127) / 128;
  static constexpr uint32_t kBBytes = BN * kMxBK;
  static constexpr uint32_t kStageBytes = kMxABytes + kBBytes;           // multiple of 1024
  static constexpr uint32_t kSfStageBytes = kAtomBytes * (1 + kAtomsB);
  static constexpr int kFit = static_cast<int>((kSmemLimit - 1024 - 256) / (kStageBytes + kSfStageBytes));
  static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
  static constexpr uint32_t kSfBase = (2 * BN + 31) / 32 * 32;  // first scale slot column
  static constexpr int kSfSlots = static_cast<int>((512 - kSfBase) / 32);
  static_assert(kAtomsB <= 4 && kSfSlots >= 2, "TMEM budget");
};

struct __align__(8) MxCtrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint32_t tmem_base;
  int abort;
};

template <int BN>
constexpr size_t mx_smem_bytes() {
  return 1024 + static_cast<size_t>(MxTile<BN>::kStages) *
                    (MxTile<BN>::kStageBytes + MxTile<BN>::kSfStageBytes) +
         sizeof(MxCtrl);
}
static_assert(mx_smem_bytes<192>() <= kSmemLimit && mx_smem_bytes<128>() <= kSmemLimit,
              "shared memory budget");

// EPI 0: bf16 out; 1: fp32 out.
template <int EPI, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb, int M, int N,
                   int K, int group_m, void* __restrict__ out) {
  using Tl = MxTile<BN>;
  constexpr int kStages = Tl::kStages;
  constexpr uint32_t kStageBytes = Tl::kStageBytes;
  constexpr uint32_t kSfStageBytes = Tl::kSfStageBytes;
  constexpr int kSfSlots = Tl::kSfSlots;
  constexpr uint32_t kTmemCols = 512;
  constexpr int kEpiWarps = 8;
  constexpr int kColsPerEpiWarp = BN / 2;
  constexpr int kGroups = kColsPerEpiWarp / 32;
  static_assert(kColsPerEpiWarp % 32 == 0, "epilogue column groups");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t sf_base = base + kStages * kStageBytes;
  MxCtrl* ctrl = reinterpret_cast<MxCtrl*>(smem + kStages * (kStageBytes + kSfStageBytes));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (K + kMxBK - 1) / kMxBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->tmem_full[b]), 1);
      mbar_init(smem_u32(&ctrl->tmem_empty[b]), kEpiWarps);
    }
    ctrl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the set-up above overlaps the front end (programmatic dependent launch)
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
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, group_m, mb, nb);
        bool ok = RNL_DCHECK(&g_err_mx, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 90);
        for (int kb = 0; kb < num_kb && ok; ++kb) {
          if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_mx, 31)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          const uint32_t ss = sf_base + stage * kSfStageBytes;
          if (!RNL_DCHECK(&g_err_mx, stage < static_cast<uint32_t>(kStages), 91)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&ctrl->full[stage]);
          mbar_arrive_expect_tx(bar, kStageBytes + kSfStageBytes);
          tma_load_2d(sa, &map_a, bar, kb * kMxBK, mb * BM);
          tma_load_2d(sa + kMxABytes, &map_b, bar, kb * kMxBK, nb * BN);
          bulk_copy_g2s(ss, sfa + (static_cast<int64_t>(mb) * num_kb + kb) * kAtomBytes, kAtomBytes, bar);
          bulk_copy_g2s(ss + kAtomBytes,
                        sfb + (static_cast<int64_t>(nb) * num_kb + kb) * Tl::kAtomsB * kAtomBytes,
                        Tl::kAtomsB * kAtomBytes, bar);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_mxf8(BM, BN);
      uint32_t stage = 0, phase = 0, unit = 0;
      uint32_t g = 0;  // k-blocks issued so far (all tiles)
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++unit) {
        const uint32_t buf = unit & 1u;
        const uint32_t use = unit >> 1;
        if (!mbar_wait(smem_u32(&ctrl->tmem_empty[buf]), (use & 1u) ^ 1u, abort, &g_err_mx, 32)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          if (!mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_mx, 33)) {
            ok = false;
            break;
          }
          // the scale slot of k-block g was last read by k-block g - kSfSlots:
          // wait for its MMAs (its stage's empty barrier) when fewer slots
          // than stages could let it still be in flight
          if (kSfSlots < kStages && g >= static_cast<uint32_t>(kSfSlots)) {
            const uint32_t prev = g - kSfSlots;
            if (!mbar_wait(smem_u32(&ctrl->empty[prev % kStages]), (prev / kStages) & 1u, abort,
                           &g_err_mx, 34)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t slot = g % kSfSlots;
          const uint32_t sf_tmem = tmem_base + Tl::kSfBase + slot * 32;
          if (!RNL_DCHECK(&g_err_mx, buf * BN + BN <= Tl::kSfBase &&
                                         Tl::kSfBase + slot * 32 + 16 + 4 * Tl::kAtomsB <= kTmemCols &&
                                         stage < static_cast<uint32_t>(kStages), 92)) {
            ok = false;
            break;
          }
          const uint32_t ss = sf_base + stage * kSfStageBytes;
          tmem_cp_32x128b_x4(sf_tmem, desc_plain(ss, 16, 128));
#pragma unroll
          for (int t = 0; t < Tl::kAtomsB; ++t)
            tmem_cp_32x128b_x4(sf_tmem + 16 + 4 * t, desc_plain(ss + kAtomBytes * (1 + t), 16, 128));
          const uint32_t sa = base + stage * kStageBytes;
          const uint64_t adesc = desc_kmajor_sw128(sa);
          const uint64_t bdesc = desc_kmajor_sw128(sa + kMxABytes);
#pragma unroll
          for (int k = 0; k < kMxBK / 32; ++k)  // +32 bytes per 32-code step
            umma_mxf8(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8_id(idesc, k), sf_tmem,
                      sf_tmem + 16, (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&ctrl->empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&ctrl->tmem_full[buf]));
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
    uint32_t unit = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++unit) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      if (!RNL_DCHECK(&g_err_mx, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 93)) break;
      const int m = mb * BM + row_local;
      const int n_base = nb * BN + half * kColsPerEpiWarp;
      const bool row_ok = m < M;
      const uint32_t buf = unit & 1u;
      const uint32_t use = unit >> 1;
      const bool got = mbar_wait(smem_u32(&ctrl->tmem_full[buf]), use & 1u, abort, &g_err_mx, 35);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kGroups; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tmem_base + lane_addr + buf * BN + half * kColsPerEpiWarp + c * 32, r);
        tmem_ld_wait();
        if (row_ok) {
          if constexpr (EPI == 0)
            store_bf16_32(out, m, n_base + c * 32, N, r);
          else
            store_f32_scaled_32(out, m, n_base + c * 32, N, r, 1.0f);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->tmem_empty[buf]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- CTA pairs
template <int BN>
struct MxPairTile {
  static constexpr int kBHalf = BN / 2;
  static constexpr int kAtomsB = (BN + 127) / 128;
  static constexpr uint32_t kBBytes = kBHalf * kMxBK;
  static constexpr uint32_t kStageBytes = kMxABytes + kBBytes;  // multiple of 1024
  static constexpr uint32_t kSfStageBytes = kAtomBytes * (1 + kAtomsB);
  static constexpr int kFit = static_cast<int>((kSmemLimit - 1024 - 256) / (kStageBytes + kSfStageBytes));
  static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
  static constexpr uint32_t kSfBase = (2 * BN + 31) / 32 * 32;
  static constexpr int kSfSlots = static_cast<int>((512 - kSfBase) / 32);
  static_assert(kStageBytes % 1024 == 0 && kAtomsB <= 4 && kSfSlots >= 2, "pair tile budget");
};

template <int BN>
constexpr size_t mx_pair_smem_bytes() {
  return 1024 + static_cast<size_t>(MxPairTile<BN>::kStages) *
                    (MxPairTile<BN>::kStageBytes + MxPairTile<BN>::kSfStageBytes) +
         sizeof(MxCtrl);
}
static_assert(mx_pair_smem_bytes<192>() <= kSmemLimit, "shared memory budget");

template <int EPI, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    mx_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_sfa, const __grid_constant__ CUtensorMap map_sfb,
                   int M, int N, int K, int group_m, void* __restrict__ out) {
  using Tl = MxPairTile<BN>;
  constexpr int kStages = Tl::kStages;
  constexpr uint32_t kStageBytes = Tl::kStageBytes;
  constexpr uint32_t kSfStageBytes = Tl::kSfStageBytes;
  constexpr int kSfSlots = Tl::kSfSlots;
  constexpr uint32_t kTmemCols = 512;
  constexpr int kEpiWarps = 8;
  constexpr int kColsPerEpiWarp = BN / 2;
  constexpr int kGroups = kColsPerEpiWarp / 32;
  static_assert(kColsPerEpiWarp % 32 == 0, "epilogue column groups");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t sf_base = base + kStages * kStageBytes;
  MxCtrl* ctrl = reinterpret_cast<MxCtrl*>(smem + kStages * (kStageBytes + kSfStageBytes));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int num_m = (M + 2 * BM - 1) / (2 * BM);  // 256-row blocks
  const int num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (K + kMxBK - 1) / kMxBK;

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
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  grid_launch_dependents();
  grid_dependency_wait();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort = &ctrl->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_a);
      tma_prefetch_map(&map_b);
      tma_prefetch_map(&map_sfa);
      tma_prefetch_map(&map_sfb);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, group_m, mb, nb);
        if (!RNL_DCHECK(&g_err_mx, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 94)) break;
        const int mb128 = 2 * mb + static_cast<int>(rank);  // this CTA's 128-row block
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_cluster(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_mx, 36)) {
            ok = false;
            break;
          }
          if (!RNL_DCHECK(&g_err_mx, stage < static_cast<uint32_t>(kStages), 95)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          const uint32_t ss = sf_base + stage * kSfStageBytes;
          const uint32_t full_local = smem_u32(&ctrl->full[stage]);
          const uint32_t full_even = mapa_shared(full_local, 0);
          if (rank == 0) mbar_arrive_expect_tx(full_local, 2 * (kStageBytes + kSfStageBytes));
          tma_load_2d_pair(sa, &map_a, full_even, kb * kMxBK, mb128 * BM);
          tma_load_2d_pair(sa + kMxABytes, &map_b, full_even, kb * kMxBK,
                           nb * BN + static_cast<int>(rank) * Tl::kBHalf);
          tma_load_2d_pair(ss, &map_sfa, full_even, 0, mb128 * num_kb + kb);
          tma_load_2d_pair(ss + kAtomBytes, &map_sfb, full_even, 0, (nb * num_kb + kb) * Tl::kAtomsB);
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
      constexpr uint32_t idesc = idesc_mxf8(2 * BM, BN);
      uint32_t stage = 0, phase = 0, unit = 0;
      uint32_t g = 0;  // k-blocks issued so far (all tiles)
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs, ++unit) {
        const uint32_t buf = unit & 1u;
        const uint32_t use = unit >> 1;
        if (!mbar_wait_cluster(smem_u32(&ctrl->tmem_empty[buf]), (use & 1u) ^ 1u, abort, &g_err_mx, 37))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          if (!mbar_wait_cluster(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_mx, 38)) {
            ok = false;
            break;
          }
          // the scale slot's previous k-block must have finished its MMAs
          if (kSfSlots < kStages && g >= static_cast<uint32_t>(kSfSlots)) {
            const uint32_t prev = g - kSfSlots;
            if (!mbar_wait_cluster(smem_u32(&ctrl->empty[prev % kStages]), (prev / kStages) & 1u, abort,
                                   &g_err_mx, 39)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t slot = g % kSfSlots;
          const uint32_t sf_tmem = tmem_base + Tl::kSfBase + slot * 32;
          if (!RNL_DCHECK(&g_err_mx, buf * BN + BN <= Tl::kSfBase &&
                                         Tl::kSfBase + slot * 32 + 16 + 4 * Tl::kAtomsB <= kTmemCols &&
                                         stage < static_cast<uint32_t>(kStages), 96)) {
            ok = false;
            break;
          }
          const uint32_t ss = sf_base + stage * kSfStageBytes;
          tmem_cp_32x128b_x4_pair(sf_tmem, desc_plain(ss, 16, 128));
#pragma unroll
          for (int t = 0; t < Tl::kAtomsB; ++t)
            tmem_cp_32x128b_x4_pair(sf_tmem + 16 + 4 * t, desc_plain(ss + kAtomBytes * (1 + t), 16, 128));
          const uint32_t sa = base + stage * kStageBytes;
          const uint64_t adesc = desc_kmajor_sw128(sa);
          const uint64_t bdesc = desc_kmajor_sw128(sa + kMxABytes);
#pragma unroll
          for (int k = 0; k < kMxBK / 32; ++k)
            umma_mxf8_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8_id(idesc, k), sf_tmem,
                           sf_tmem + 16, (kb > 0 || k > 0) ? 1u : 0u);
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
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const int row_local = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t empty_even_0 = mapa_shared(smem_u32(&ctrl->tmem_empty[0]), 0);
    const uint32_t empty_even_1 = mapa_shared(smem_u32(&ctrl->tmem_empty[1]), 0);
    uint32_t unit = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs, ++unit) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      if (!RNL_DCHECK(&g_err_mx, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 97)) break;
      const int64_t m = static_cast<int64_t>(mb) * 2 * BM + rank * BM + row_local;
      const int n_base = nb * BN + half * kColsPerEpiWarp;
      const bool row_ok = m < M;
      const uint32_t buf = unit & 1u;
      const uint32_t use = unit >> 1;
      const bool got = mbar_wait_cluster(smem_u32(&ctrl->tmem_full[buf]), use & 1u, abort, &g_err_mx, 40);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kGroups; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tmem_base + lane_addr + buf * BN + half * kColsPerEpiWarp + c * 32, r);
        tmem_ld_wait();
        if (row_ok) {
          if constexpr (EPI == 0)
            store_bf16_32(out, m, n_base + c * 32, N, r);
          else
            store_f32_scaled_32(out, m, n_base + c * 32, N, r, 1.0f);
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

// Largest number of CTA pairs of the pair kernel resident at once.
int mx_resident_pairs(const DeviceInfo& dev) {
  static std::atomic<int> cached[64];
  const int c = cached[dev.device].load(std::memory_order_relaxed);
  if (c > 0) return c;
  auto kern = mx_pair_kernel<0, 192>;
  int n = 0;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, mx_pair_smem_bytes<192>()) == RNL_OK) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = mx_pair_smem_bytes<192>();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n <= 0) n = dev.sm_count / 2;
  cached[dev.device].store(n, std::memory_order_relaxed);
  return n;
}

template <int EPI, int BN>
rnl_status launch_mx_pair(const uint8_t* a, const uint8_t* b, const uint8_t* sfa, const uint8_t* sfb,
                          int64_t M, int64_t N, int64_t K, void* out, const DeviceInfo& dev,
                          cudaStream_t s) {
  using Tl = MxPairTile<BN>;
  auto kern = mx_pair_kernel<EPI, BN>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, mx_pair_smem_bytes<BN>()) != RNL_OK)
    return RNL_ERR_LAUNCH;
  const int64_t num_kg = (K + kMxBK - 1) / kMxBK;
  CUtensorMap ma, mb, msa, msb;
  rnl_status st = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, kMxBK, BM);
  if (st != RNL_OK) return st;
  st = make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, N, K, kMxBK, Tl::kBHalf);
  if (st != RNL_OK) return st;
  // the atoms as rows of 128 words: A's [ceil(M / 128) * kgs], B's [tiles * kgs * atoms]
  st = make_map_2d_plain(&msa, CU_TENSOR_MAP_DATA_TYPE_UINT32, sfa, 128, ((M + 127) / 128) * num_kg,
                         kAtomBytes, 128, 1);
  if (st != RNL_OK) return st;
  st = make_map_2d_plain(&msb, CU_TENSOR_MAP_DATA_TYPE_UINT32, sfb, 128,
                         ((N + BN - 1) / BN) * num_kg * Tl::kAtomsB, kAtomBytes, 128, Tl::kAtomsB);
  if (st != RNL_OK) return st;
  const int num_m = static_cast<int>((M + 2 * BM - 1) / (2 * BM));
  const int64_t tiles = static_cast<int64_t>(num_m) * ((N + BN - 1) / BN);
  const int max_pairs = mx_resident_pairs(dev);
  const int pairs = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
  const int group_m = (M * K <= (int64_t{24} << 20)) ? num_m : (num_m < 4 ? num_m : 4);
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
  cfg.dynamicSmemBytes = mx_pair_smem_bytes<BN>();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  trace_before(s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, msa, msb, static_cast<int>(M),
                                           static_cast<int>(N), static_cast<int>(K), group_m, out);
  trace_after(s, "gemm_mxfp8_block_scaled_pair");
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

template <int EPI, int BN>
rnl_status launch_mx_bn(const uint8_t* a, const uint8_t* b, const uint8_t* sfa, const uint8_t* sfb,
                        int64_t M, int64_t N, int64_t K, void* out, const DeviceInfo& dev,
                        cudaStream_t s) {
  auto kern = mx_gemm_kernel<EPI, BN>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, mx_smem_bytes<BN>()) != RNL_OK)
    return RNL_ERR_LAUNCH;
  CUtensorMap ma, mb;
  rnl_status st = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, kMxBK, BM);
  if (st != RNL_OK) return st;
  st = make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, N, K, kMxBK, BN);
  if (st != RNL_OK) return st;
  const int num_m = static_cast<int>((M + BM - 1) / BM);
  const int64_t tiles = static_cast<int64_t>(num_m) * ((N + BN - 1) / BN);
  const unsigned grid = static_cast<unsigned>(tiles < dev.sm_count ? tiles : dev.sm_count);
  // A panels of up to 24 MB stay in L2 whole; larger ones are walked in groups of 8 row blocks
  const int group_m = (M * K <= (int64_t{24} << 20)) ? num_m : (num_m < 8 ? num_m : 8);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = mx_smem_bytes<BN>();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_before(s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, sfa, sfb, static_cast<int>(M),
                                           static_cast<int>(N), static_cast<int>(K), group_m, out);
  trace_after(s, "gemm_mxfp8_block_scaled");
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

}  // namespace

int mx_native_bn() { return 192; }

size_t mx_sf_atoms_bytes(int64_t rows, int64_t K, int rows_per_tile) {
  const int64_t tiles = (rows + rows_per_tile - 1) / rows_per_tile;
  const int64_t kgs = (K + kMxBK - 1) / kMxBK;
  const int64_t atoms = (rows_per_tile + 127) / 128;
  return static_cast<size_t>(tiles * kgs * atoms) * kAtomBytes;
}

rnl_status launch_mx_gemm_native(const uint8_t* a_codes, const uint8_t* b_codes, const uint8_t* sfa,
                                 const uint8_t* sfb, int64_t M, int64_t N, int64_t K, void* out,
                                 int out_dtype, cudaStream_t s) {
  if (M == 0) return RNL_OK;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  // one CTA per tile unless RNL_MXFP8_PAIR=1 (the pair form measured slower:
  // 109.6 against 97.2 us at 4096 x 4096 -> 6144)
  bool pair = false;
  if (const char* e = std::getenv("RNL_MXFP8_PAIR"))
    if (e[0] == '0' || e[0] == '1') pair = e[0] == '1';
  if (pair) {
    if (out_dtype == RNL_OUT_BF16) return launch_mx_pair<0, 192>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s);
    return launch_mx_pair<1, 192>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s);
  }
  if (out_dtype == RNL_OUT_BF16) return launch_mx_bn<0, 192>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s);
  return launch_mx_bn<1, 192>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s);
}

rnl_status read_clear_error_mx(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_mx, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_mx, &zero, sizeof zero) != cudaSuccess) return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
