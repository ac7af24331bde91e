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
// Scale-factor atoms (written by the front end, mxfp8.cu): 512 bytes hold the
// 4 scale bytes of 128 rows for one k-block of 128 codes, row r at byte
// 16 (r % 32) + 4 (r / 32) + j (j = the 32-element block); A's atoms per
// 128-row block and k-block, B's per 192-row output tile, k-block and
// 128-row part.  In tensor memory the MMA reads the scale of A row m from
// lane m % 32 (the same in every 32-lane quarter), column sfa + m / 32, byte
// j chosen by the instruction descriptor; B row n from lane n % 32, column
// sfb + 4 (n / 128) + (n % 128) / 32.  So lane i of every quarter holds the
// 16 bytes at offset 16 i of each atom in 4 consecutive columns.
//
// Persistent, warp-specialised, one CTA per SM, output tiles of 128 x BN:
//   warp 0      producer: per k-block a TMA box of A (128 x 128 codes) and of
//               B (BN x 128), 128-byte swizzle, into a ring of stages.
//   warp 1      allocates 512 TMEM columns (two fp32 accumulators of BN
//               columns, then slots of 32 columns for one k-block's scales:
//               A's atom at +0, B's at +16, +20) and one thread issues the
//               four MMAs of each k-block (scale byte j = 0..3).
//   warps 2-9   epilogue: tcgen05.ld of the accumulator, bf16 or fp32 stores.
//   warps 10-13 scale writers, one per TMEM lane quarter: for each k-block
//               they load the atoms' 16-byte rows from global memory (L2)
//               ahead of time, wait until the slot's previous k-block has
//               finished its MMAs, and tcgen05.st them into the slot.
// Writing the scales from separate warps keeps them off the MMA thread's
// in-order tcgen05 stream: a tcgen05.cp of the atoms before each k-block's
// MMAs (the first form of this kernel) held the tensor pipe for ~16 % of
// the time, and the MMA thread's wait for a free slot for another ~7 %.
//
// The CTA-pair form (tcgen05 cta_group::2, 256 x BN tiles on two SMs,
// RNL_MXFP8_PAIR=1): each CTA stages its own 128 rows of A and half of B's
// BN rows; each CTA's scale writers fill its own TMEM (its A rows, all of B's
// rows: each CTA's tensor core scales all BN columns) and signal the even
// CTA, whose one thread issues M = 256 MMAs.  It halves each SM's B traffic
// but measured slower than the one-CTA form, so it is not the default.
// Every wait is bounded (ptx.cuh).
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
constexpr int kSfWarps = 4;                 // scale writers, one per TMEM lane quarter
constexpr int kMxThreads = kThreads + kSfWarps * 32;
constexpr int kMaxSfSlots = 8;

// PAIR = false: 128 x BN tiles on one CTA; true: 256 x BN tiles on a CTA pair.
template <int BN, bool PAIR>
struct MxTile {
  static constexpr int kAtomsB = (BN + 127) / 128;
  static constexpr int kBRows = PAIR ? BN / 2 : BN;  // B rows staged per CTA
  static constexpr uint32_t kBBytes = kBRows * kMxBK;
  static constexpr uint32_t kStageBytes = kMxABytes + kBBytes;  // multiple of 1024
  static constexpr int kFit = static_cast<int>((kSmemLimit - 1024 - 256) / kStageBytes);
  static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
  static constexpr uint32_t kSfBase = (2 * BN + 31) / 32 * 32;  // first scale slot column
  static constexpr int kSfSlotsFit = static_cast<int>((512 - kSfBase) / 32);
  static constexpr int kSfSlots = kSfSlotsFit < kMaxSfSlots ? kSfSlotsFit : kMaxSfSlots;
  static_assert(kStageBytes % 1024 == 0 && kAtomsB <= 4 && kSfSlots >= 2, "tile budget");
};

struct __align__(8) MxCtrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t sf_full[kMaxSfSlots];   // the slot's scales are in TMEM (even CTA for pairs)
  uint64_t sf_empty[kMaxSfSlots];  // the slot's k-block has finished its MMAs
  uint32_t tmem_base;
  int abort;
};

template <int BN, bool PAIR>
constexpr size_t mx_smem_bytes() {
  return 1024 + static_cast<size_t>(MxTile<BN, PAIR>::kStages) * MxTile<BN, PAIR>::kStageBytes +
         sizeof(MxCtrl);
}
static_assert(mx_smem_bytes<192, false>() <= kSmemLimit && mx_smem_bytes<192, true>() <= kSmemLimit,
              "shared memory budget");

// Bounded wait on one of this CTA's barriers that may be signalled from the
// peer CTA (pairs) or by the tensor core.
__device__ __forceinline__ bool mx_wait(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t site) {
  return mbar_wait_cluster(bar, parity, abort, &g_err_mx, site);
}

// EPI 0: bf16 out; 1: fp32 out.
template <int EPI, int BN, bool PAIR>
__global__ void __launch_bounds__(kMxThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const uint4* __restrict__ sfa, const uint4* __restrict__ sfb, int M, int N, int K,
                   int group_m, void* __restrict__ out) {
  using Tl = MxTile<BN, PAIR>;
  constexpr int kStages = Tl::kStages;
  constexpr uint32_t kStageBytes = Tl::kStageBytes;
  constexpr int kSfSlots = Tl::kSfSlots;
  constexpr uint32_t kTmemCols = 512;
  constexpr int kEpiWarps = 8;
  constexpr int kColsPerEpiWarp = BN / 2;
  constexpr int kGroups = kColsPerEpiWarp / 32;
  constexpr int kRowsPerTile = PAIR ? 2 * BM : BM;
  static_assert(kColsPerEpiWarp % 32 == 0, "epilogue column groups");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  MxCtrl* ctrl = reinterpret_cast<MxCtrl*>(smem + kStages * kStageBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // 0 issues the MMAs
  const int unit_id = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int num_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int num_m = (M + kRowsPerTile - 1) / kRowsPerTile;
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
      mbar_init(smem_u32(&ctrl->tmem_empty[b]), (PAIR ? 2 : 1) * kEpiWarps);
    }
    for (int s = 0; s < kSfSlots; ++s) {
      mbar_init(smem_u32(&ctrl->sf_full[s]), (PAIR ? 2 : 1) * kSfWarps);
      mbar_init(smem_u32(&ctrl->sf_empty[s]), 1);
    }
    ctrl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(&ctrl->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();
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
      bool ok = true;
      for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, group_m, mb, nb);
        if (!RNL_DCHECK(&g_err_mx, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 90)) break;
        const int a_row = mb * kRowsPerTile + static_cast<int>(rank) * BM;
        const int b_row = nb * BN + static_cast<int>(rank) * Tl::kBRows;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mx_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, 31)) {
            ok = false;
            break;
          }
          if (!RNL_DCHECK(&g_err_mx, stage < static_cast<uint32_t>(kStages), 91)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          const uint32_t full_local = smem_u32(&ctrl->full[stage]);
          if (PAIR) {
            const uint32_t full_even = mapa_shared(full_local, 0);
            if (rank == 0) mbar_arrive_expect_tx(full_local, 2 * kStageBytes);
            tma_load_2d_pair(sa, &map_a, full_even, kb * kMxBK, a_row);
            tma_load_2d_pair(sa + kMxABytes, &map_b, full_even, kb * kMxBK, b_row);
          } else {
            mbar_arrive_expect_tx(full_local, kStageBytes);
            tma_load_2d(sa, &map_a, full_local, kb * kMxBK, a_row);
            tma_load_2d(sa + kMxABytes, &map_b, full_local, kb * kMxBK, b_row);
          }
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
      constexpr uint32_t idesc = idesc_mxf8(kRowsPerTile, BN);
      uint32_t stage = 0, phase = 0, unit = 0;
      uint32_t g = 0;  // k-blocks issued so far (all tiles)
      bool ok = true;
      for (int tile = unit_id; tile < num_tiles && ok; tile += num_units, ++unit) {
        const uint32_t buf = unit & 1u;
        const uint32_t use = unit >> 1;
        if (!mx_wait(smem_u32(&ctrl->tmem_empty[buf]), (use & 1u) ^ 1u, abort, 32)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const uint32_t slot = g % kSfSlots;
          if (!mx_wait(smem_u32(&ctrl->full[stage]), phase, abort, 33) ||
              !mx_wait(smem_u32(&ctrl->sf_full[slot]), (g / kSfSlots) & 1u, abort, 34)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_tmem = tmem_base + Tl::kSfBase + slot * 32;
          if (!RNL_DCHECK(&g_err_mx, buf * BN + BN <= Tl::kSfBase &&
                                         Tl::kSfBase + slot * 32 + 16 + 4 * Tl::kAtomsB <= kTmemCols &&
                                         stage < static_cast<uint32_t>(kStages), 92)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          const uint64_t adesc = desc_kmajor_sw128(sa);
          const uint64_t bdesc = desc_kmajor_sw128(sa + kMxABytes);
#pragma unroll
          for (int k = 0; k < kMxBK / 32; ++k) {  // +32 bytes per 32-code step
            if (PAIR)
              umma_mxf8_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8_id(idesc, k), sf_tmem,
                             sf_tmem + 16, (kb > 0 || k > 0) ? 1u : 0u);
            else
              umma_mxf8(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8_id(idesc, k), sf_tmem,
                        sf_tmem + 16, (kb > 0 || k > 0) ? 1u : 0u);
          }
          if (PAIR) {
            umma_commit_pair(smem_u32(&ctrl->empty[stage]), 0x3);
            umma_commit_pair(smem_u32(&ctrl->sf_empty[slot]), 0x3);
          } else {
            umma_commit(smem_u32(&ctrl->empty[stage]));
            umma_commit(smem_u32(&ctrl->sf_empty[slot]));
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR)
          umma_commit_pair(smem_u32(&ctrl->tmem_full[buf]), 0x3);
        else
          umma_commit(smem_u32(&ctrl->tmem_full[buf]));
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int half = ew >> 2;      // which half of the BN columns
    const int row_local = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t empty_even_0 = PAIR ? mapa_shared(smem_u32(&ctrl->tmem_empty[0]), 0) : 0u;
    const uint32_t empty_even_1 = PAIR ? mapa_shared(smem_u32(&ctrl->tmem_empty[1]), 0) : 0u;
    uint32_t unit = 0;
    for (int tile = unit_id; tile < num_tiles; tile += num_units, ++unit) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      if (!RNL_DCHECK(&g_err_mx, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 93)) break;
      const int64_t m = static_cast<int64_t>(mb) * kRowsPerTile + rank * BM + row_local;
      const int n_base = nb * BN + half * kColsPerEpiWarp;
      const bool row_ok = m < M;
      const uint32_t buf = unit & 1u;
      const uint32_t use = unit >> 1;
      const bool got = mx_wait(smem_u32(&ctrl->tmem_full[buf]), use & 1u, abort, 35);
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
        if (!PAIR || rank == 0)
          mbar_arrive(smem_u32(&ctrl->tmem_empty[buf]));
        else
          mbar_arrive_cluster(buf ? empty_even_1 : empty_even_0);
      }
    }
  } else {
    // ------------------------------------------------------- scale writers
    const int quarter = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t g = 0;
    bool ok = true;
    for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      if (!RNL_DCHECK(&g_err_mx, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 94)) break;
      // this CTA's 128-row block of A and B's atoms of the tile, lane i's 16 bytes
      const int a_blk = mb * (kRowsPerTile / BM) + static_cast<int>(rank);
      const uint4* pa = sfa + static_cast<int64_t>(a_blk) * num_kb * (kAtomBytes / 16) + lane;
      const uint4* pb = sfb + static_cast<int64_t>(nb) * num_kb * Tl::kAtomsB * (kAtomBytes / 16) + lane;
      for (int kb = 0; kb < num_kb; ++kb, ++g) {
        // the loads go out before the wait for the slot, so their latency
        // hides behind the MMAs still using it
        const uint4 wa = __ldg(pa + kb * (kAtomBytes / 16));
        uint4 wb[Tl::kAtomsB];
#pragma unroll
        for (int t = 0; t < Tl::kAtomsB; ++t) wb[t] = __ldg(pb + (kb * Tl::kAtomsB + t) * (kAtomBytes / 16));
        const uint32_t slot = g % kSfSlots;
        const bool got = mx_wait(smem_u32(&ctrl->sf_empty[slot]), ((g / kSfSlots) & 1u) ^ 1u, abort, 36);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = Tl::kSfBase + slot * 32;
        if (!RNL_DCHECK(&g_err_mx, col + 16 + 4 * Tl::kAtomsB <= kTmemCols, 95)) {
          ok = false;
          break;
        }
        tmem_st_4cols(tmem_base + lane_addr + col, wa);
#pragma unroll
        for (int t = 0; t < Tl::kAtomsB; ++t) tmem_st_4cols(tmem_base + lane_addr + col + 16 + 4 * t, wb[t]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          const uint32_t bar = smem_u32(&ctrl->sf_full[slot]);
          if (!PAIR || rank == 0)
            mbar_arrive(bar);
          else
            mbar_arrive_cluster(mapa_shared(bar, 0));
        }
      }
    }
  }

  // no CTA leaves (or frees TMEM) while the MMAs may still read its shared
  // memory or, in a pair, its peer may still signal its barriers
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Largest number of CTA pairs of the pair kernel resident at once.
int mx_resident_pairs(const DeviceInfo& dev) {
  static std::atomic<int> cached[64];
  const int c = cached[dev.device].load(std::memory_order_relaxed);
  if (c > 0) return c;
  auto kern = mx_gemm_kernel<0, 192, true>;
  int n = 0;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, mx_smem_bytes<192, true>()) == RNL_OK) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(kMxThreads, 1, 1);
    cfg.dynamicSmemBytes = mx_smem_bytes<192, true>();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n <= 0) n = dev.sm_count / 2;
  cached[dev.device].store(n, std::memory_order_relaxed);
  return n;
}

template <int EPI, int BN, bool PAIR>
rnl_status launch_mx(const uint8_t* a, const uint8_t* b, const uint8_t* sfa, const uint8_t* sfb,
                     int64_t M, int64_t N, int64_t K, void* out, const DeviceInfo& dev, cudaStream_t s) {
  using Tl = MxTile<BN, PAIR>;
  auto kern = mx_gemm_kernel<EPI, BN, PAIR>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, mx_smem_bytes<BN, PAIR>()) != RNL_OK)
    return RNL_ERR_LAUNCH;
  CUtensorMap ma, mb;
  rnl_status st = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, kMxBK, BM);
  if (st != RNL_OK) return st;
  st = make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, N, K, kMxBK, Tl::kBRows);
  if (st != RNL_OK) return st;
  constexpr int kRowsPerTile = PAIR ? 2 * BM : BM;
  const int num_m = static_cast<int>((M + kRowsPerTile - 1) / kRowsPerTile);
  const int64_t tiles = static_cast<int64_t>(num_m) * ((N + BN - 1) / BN);
  const int max_units = PAIR ? mx_resident_pairs(dev) : dev.sm_count;
  const int units = static_cast<int>(tiles < max_units ? tiles : max_units);
  // A panels of up to 24 MB stay in L2 whole; larger ones are walked in groups
  const int group_m = (M * K <= (int64_t{24} << 20)) ? num_m : (num_m < 8 ? num_m : 8);
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((PAIR ? 2 : 1) * units), 1, 1);
  cfg.blockDim = dim3(kMxThreads, 1, 1);
  cfg.dynamicSmemBytes = mx_smem_bytes<BN, PAIR>();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  trace_before(s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, reinterpret_cast<const uint4*>(sfa),
                                           reinterpret_cast<const uint4*>(sfb), static_cast<int>(M),
                                           static_cast<int>(N), static_cast<int>(K), group_m, out);
  trace_after(s, PAIR ? "gemm_mxfp8_block_scaled_pair" : "gemm_mxfp8_block_scaled");
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
  // one CTA per 128 x 192 tile; RNL_MXFP8_PAIR=1 selects the CTA-pair form,
  // which measured slower (224 against 92.6 us at 4096 x 4096 -> 6144: the odd
  // CTA's scale stores into its TMEM stall the pair's MMAs)
  bool pair = false;
  if (const char* e = std::getenv("RNL_MXFP8_PAIR"))
    if (e[0] == '0' || e[0] == '1') pair = e[0] == '1';
  const bool bf16 = out_dtype == RNL_OUT_BF16;
  if (pair)
    return bf16 ? launch_mx<0, 192, true>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s)
                : launch_mx<1, 192, true>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s);
  return bf16 ? launch_mx<0, 192, false>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s)
              : launch_mx<1, 192, false>(a_codes, b_codes, sfa, sfb, M, N, K, out, dev, s);
}

rnl_status read_clear_error_mx(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_mx, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_mx, &zero, sizeof zero) != cudaSuccess) return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
