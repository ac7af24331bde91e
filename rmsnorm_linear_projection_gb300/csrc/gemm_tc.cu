// gemm_tc.cu -- the C stage: out = epilogue(A[M,K] @ B[N,K]^T) on the
// 5th-generation tensor cores (tcgen05), AT-09 "Linear" of the AT-10 pattern
// page (sec. 4: matmul(x, w, dtype, b_trans=True), W stored [N, K]).
//
// Persistent, warp-specialised kernel, one CTA per SM, output tiles of
// 128 x BN (BN = 256, 192 or 128, chosen per shape so the last wave of
// tiles is as full as possible):
//   warp 0      TMA producer: 128x64 A box and BNx64 B box per stage
//               (128-byte swizzle), a ring of 4 (BN=256), 5 (192) or 7 (128)
//               stages filling the 227 KB of shared memory.
//   warp 1      allocates 512 TMEM columns (two fp32 accumulators, 256
//               columns apart) and one thread issues tcgen05.mma
//               (M=128, N=BN, K=16).
//   warps 2-9   epilogue: tcgen05.ld the accumulator (each warp one 32-lane
//               quarter x BN/2 columns), convert, store to global memory.
// Both operands are K-major, the layout the MMA reads directly, so the
// weight needs no transpose (the pages pre-transpose it on the host for the
// same reason).  The two accumulators let the epilogue of tile i overlap the
// main loop of tile i+1.
//
// Exact integer mode (W8A8): A and B hold integers in [-127, 127] as bf16
// (exact).  Every product is an integer of magnitude <= 16129 and the MMA
// accumulates in fp32, which is exact while every partial sum stays below
// 2^24; a chunk of 1024 products keeps |sum| <= 16,516,096 < 2^24.  So the
// K loop is cut into chunks of 16 k-blocks (1024 products); each chunk goes
// to its own accumulator and the epilogue converts it exactly to int32 and
// adds it in registers.
//
// Batched sum mode (QuantMatMulReduceSum, Epi::kDequantBatchSum): the work
// items are (batch b, tile) in b-major order; the producer reads batch b's
// rows of A and B, and the epilogue of item (b, tile) adds its dequantised
// FP32 values to the running sum that item (b - 1, tile) left in global
// memory, after waiting (bounded) for that item's flag: one 64-bit flag per
// (tile, epilogue warp), set with a release store to tag | (b + 1) after the
// warp's sums are written, and set back to 0 by the last batch's item, so a
// replay of the launch with the same tag (a CUDA graph) starts from 0.  Item i waits only for item i - tiles, and every
// CTA takes its items in increasing order with all CTAs resident, so every
// wait ends.
#include <cuda_bf16.h>

#include <cstdlib>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_gemm;

using namespace gemm;

// Tile-width dependent constants (BN = 128, 192 or 256 output columns).
template <int BN>
struct Tile {
  static constexpr uint32_t kBBytes = BN * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages =
      static_cast<int>((kSmemLimit - 1024 - 256) / kStageBytes) < kMaxStages
          ? static_cast<int>((kSmemLimit - 1024 - 256) / kStageBytes)
          : kMaxStages;
  static constexpr uint32_t kTmemCols = 512;  // two accumulators of BN <= 256 columns
};

struct __align__(8) Ctrl {
  uint64_t full[kMaxStages];
  uint64_t xform_full[kMaxStages];  // A stage normalised in place (fused-norm mode)
  uint64_t empty[kMaxStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint32_t tmem_base;
  int abort;
};

template <int BN>
constexpr size_t smem_bytes() {
  return 1024 + static_cast<size_t>(Tile<BN>::kStages) * Tile<BN>::kStageBytes + sizeof(Ctrl);
}
static_assert(smem_bytes<256>() <= kSmemLimit && smem_bytes<192>() <= kSmemLimit &&
                  smem_bytes<128>() <= kSmemLimit,
              "shared memory budget");

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t site) {
  const bool ok = mbar_wait(bar, parity, abort, &g_err_gemm, site);
  return __all_sync(0xFFFFFFFFu, ok);
}

// NORM_A: A is the raw activation x; four transform warps turn each A stage
// into bf16((x * rstd[m]) * gamma[k]) in place before the MMA reads it (the
// AT-10 V stage fused into the C stage's operand path).
template <int EPI, int BN, bool NORM_A>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                int M, int N, int K, int group_m, void* __restrict__ out,
                const float* __restrict__ row_scale, const float* __restrict__ col_scale,
                const float* __restrict__ a_rstd, const uint4* __restrict__ a_gamma,
                const __nv_bfloat16* __restrict__ bias, int acc_mode, void* out_final, int nbatch,
                uint64_t* batch_flags, uint64_t tag) {
  constexpr bool kBatch = EPI == static_cast<int>(Epi::kDequantBatchSum);
  constexpr bool kInt = (EPI == static_cast<int>(Epi::kDequantBf16) ||
                         EPI == static_cast<int>(Epi::kInt32) ||
                         EPI == static_cast<int>(Epi::kDequantAccF32) || kBatch);
  static_assert(!(NORM_A && kInt), "the fused norm feeds the bf16 GEMM only");
  constexpr int kStages = Tile<BN>::kStages;
  constexpr uint32_t kStageBytes = Tile<BN>::kStageBytes;
  constexpr uint32_t kTmemCols = Tile<BN>::kTmemCols;
  constexpr int kEpiWarps = NORM_A ? 4 : 8;
  constexpr int kXformWarps = NORM_A ? 4 : 0;
  static_assert(64 + 32 * (kEpiWarps + kXformWarps) == kThreads, "warp roles");
  constexpr int kColsPerEpiWarp = BN * 4 / kEpiWarps;  // 8 warps: BN/2 each; 4 warps: BN
  constexpr int kGroups = kColsPerEpiWarp / 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kStages * kStageBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_items = num_tiles * (kBatch ? nbatch : 1);
  const int num_kb = (K + BK - 1) / BK;
  const int kb_per_unit = kInt ? kChunkKBlocks : num_kb;
  const int units_per_tile = (num_kb + kb_per_unit - 1) / kb_per_unit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->xform_full[s]), kXformWarps > 0 ? kXformWarps : 1);
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
  // The set-up above overlaps the previous kernel when launched as its
  // programmatic dependent; from here on its outputs (A, row scales) are read.
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
      for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
        const int b = kBatch ? item / num_tiles : 0;
        const int tile = item - b * num_tiles;
        int mb, nb;
        tile_coords(tile, num_m, num_n, group_m, mb, nb);
        bool ok = RNL_DCHECK(&g_err_gemm, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n && b < nbatch, 60);
        for (int kb = 0; kb < num_kb && ok; ++kb) {
          if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_gemm, 1)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          if (!RNL_DCHECK(&g_err_gemm, stage < static_cast<uint32_t>(kStages) &&
                                           sa + kStageBytes <= base + kStages * kStageBytes, 61)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&ctrl->full[stage]);
          mbar_arrive_expect_tx(bar, kStageBytes);
          tma_load_2d(sa, &map_a, bar, kb * BK, b * M + mb * BM);
          tma_load_2d(sa + kABytes, &map_b, bar, kb * BK, b * N + nb * BN);
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
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
      uint32_t stage = 0, phase = 0, unit = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
        for (int u = 0; u < units_per_tile && ok; ++u, ++unit) {
          const uint32_t buf = unit & 1u;
          const uint32_t use = unit >> 1;
          if (!mbar_wait(smem_u32(&ctrl->tmem_empty[buf]), (use & 1u) ^ 1u, abort, &g_err_gemm, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kAccStride;
          if (!RNL_DCHECK(&g_err_gemm, buf * kAccStride + BN <= kTmemCols, 62)) {
            ok = false;
            break;
          }
          const int kb0 = u * kb_per_unit;
          const int kb1 = min(num_kb, kb0 + kb_per_unit);
          for (int kb = kb0; kb < kb1; ++kb) {
            const uint32_t ready = NORM_A ? smem_u32(&ctrl->xform_full[stage]) : smem_u32(&ctrl->full[stage]);
            if (!mbar_wait(ready, phase, abort, &g_err_gemm, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = base + stage * kStageBytes;
            if (!RNL_DCHECK(&g_err_gemm, stage < static_cast<uint32_t>(kStages), 63)) {
              ok = false;
              break;
            }
            const uint64_t adesc = desc_kmajor_sw128(sa);
            const uint64_t bdesc = desc_kmajor_sw128(sa + kABytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              // +32 bytes per 16-element K step inside the 128-byte row
              umma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                        (kb > kb0 || k > 0) ? 1u : 0u);
            }
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
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int half = ew >> 2;      // which half of the columns (8 epilogue warps)
    const int row_local = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t unit = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
      const int b = kBatch ? item / num_tiles : 0;
      const int tile = item - b * num_tiles;
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      if (!RNL_DCHECK(&g_err_gemm, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n && b < nbatch, 64)) {
        ok = false;
        break;
      }
      const int m = mb * BM + row_local;
      const int n_base = nb * BN + half * kColsPerEpiWarp;
      const bool row_ok = m < M;
      float rs = 0.f;
      if ((EPI == static_cast<int>(Epi::kRowScaleF32) || EPI == static_cast<int>(Epi::kDequantBf16) ||
           EPI == static_cast<int>(Epi::kDequantAccF32) || kBatch) && row_ok)
        rs = row_scale != nullptr ? __ldg(row_scale + static_cast<int64_t>(b) * M + m) : 1.0f;
      int iacc[kInt ? kGroups : 1][kInt ? 32 : 1];
      if (kInt) {
#pragma unroll
        for (int c = 0; c < (kInt ? kGroups : 1); ++c)
#pragma unroll
          for (int j = 0; j < (kInt ? 32 : 1); ++j) iacc[c][j] = 0;
      }
      uint64_t* flag = nullptr;
      if constexpr (kBatch) {
        // wait for the running sum of batches 0 .. b-1 (item (b-1, tile),
        // 1.7 waves back, normally long done) and pull this warp's part of it
        // into L2 while the accumulators drain
        flag = batch_flags + static_cast<int64_t>(tile) * kEpiWarps + ew;
        // the host sizes the flags for the 128 x 128 tiling (batch_flag_bytes)
        if (!RNL_DCHECK(&g_err_gemm, static_cast<int64_t>(tile) * kEpiWarps + ew <
                                         static_cast<int64_t>((M + 127) / 128) * ((N + 127) / 128) * 8, 65)) {
          ok = false;
          break;
        }
        if (b > 0) {
          if (!__all_sync(0xFFFFFFFFu, flag_wait(flag, tag | static_cast<uint64_t>(b), abort, &g_err_gemm, 26))) {
            ok = false;
            break;
          }
          if (row_ok) {
            const float* arow = static_cast<const float*>(out) + static_cast<int64_t>(m) * N;
#pragma unroll
            for (int c = 0; c < kGroups; ++c)
              if (n_base + c * 32 < N) prefetch_l2(arow + n_base + c * 32);
          }
        }
      }
      for (int u = 0; u < units_per_tile; ++u, ++unit) {
        const uint32_t buf = unit & 1u;
        const uint32_t use = unit >> 1;
        if (!warp_wait(smem_u32(&ctrl->tmem_full[buf]), use & 1u, abort, 4)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (!RNL_DCHECK(&g_err_gemm, buf * kAccStride + (half + 1) * kColsPerEpiWarp <= kTmemCols &&
                                         kColsPerEpiWarp * (kEpiWarps / 4) <= BN, 66)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < kGroups; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(tmem_base + lane_addr + buf * kAccStride + half * kColsPerEpiWarp + c * 32, r);
          tmem_ld_wait();
          const int n0 = n_base + c * 32;
          if constexpr (kInt) {
#pragma unroll
            for (int j = 0; j < 32; ++j) iacc[c][j] += __float2int_rn(__uint_as_float(r[j]));
          } else if constexpr (EPI == static_cast<int>(Epi::kBf16)) {
            if (row_ok) {
              if (bias != nullptr)
                store_bf16_bias_32(out, m, n0, N, r, bias);
              else
                store_bf16_32(out, m, n0, N, r);
            }
          } else {  // kRowScaleF32
            if (row_ok) store_f32_scaled_32(out, m, n0, N, r, rs);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl->tmem_empty[buf]));
      }
      if (!ok) break;
      if constexpr (kBatch) {
        const int mode = (b > 0 ? 1 : 0) | (b == nbatch - 1 ? 2 : 0);
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < kGroups; ++c)
            store_dequant_acc_32(static_cast<float*>(out), static_cast<__nv_bfloat16*>(out_final), m,
                                 n_base + c * 32, N, iacc[c], rs, col_scale, mode);
        }
        if (b < nbatch - 1) {
          __threadfence();
          __syncwarp();
          if (lane == 0) flag_release(flag, tag | static_cast<uint64_t>(b + 1));
        } else if (b > 0) {
          // the last batch consumed the flag: back to 0, so that a replay of
          // this launch (same tag, in a CUDA graph) waits for its own flags
          __syncwarp();
          if (lane == 0) *flag = 0;
        }
      } else if constexpr (kInt) {
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < kGroups; ++c) {
            if constexpr (EPI == static_cast<int>(Epi::kInt32))
              store_i32_32(out, m, n_base + c * 32, N, iacc[c]);
            else if constexpr (EPI == static_cast<int>(Epi::kDequantAccF32))
              store_dequant_acc_32(static_cast<float*>(out), static_cast<__nv_bfloat16*>(out_final), m,
                                   n_base + c * 32, N, iacc[c], rs, col_scale, acc_mode);
            else
              store_dequant_32(out, m, n_base + c * 32, N, iacc[c], rs, col_scale, bias);
          }
        }
      }
    }
  } else if constexpr (NORM_A) {
    // ------------------------------------------------- A transform (fused norm)
    // Thread t owns row t of every A stage: 64 bf16 in eight 16-byte chunks,
    // logical chunk c stored at chunk c ^ (t % 8) by the 128-byte swizzle.
    // Visiting logical chunks in order keeps the eight threads of a
    // shared-memory wavefront on eight different bank groups.
    const int t = (warp - 2 - kEpiWarps) * 32 + lane;
    const int sw = t & 7;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group_m, mb, nb);
      const int m = mb * BM + t;
      const float rs = m < M ? __ldg(a_rstd + m) : 0.f;
      for (int kb = 0; kb < num_kb; ++kb) {
        const bool got = mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_gemm, 5);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        uint4* rowp = reinterpret_cast<uint4*>(smem + stage * kStageBytes + t * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int k = kb * BK + c * 8;
          uint4* q = rowp + (c ^ sw);
          const uint4 u = *q;
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
          uint32_t gw[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};  // bf16 1.0
          if (a_gamma != nullptr && k < K) {
            const uint4 gv = __ldg(a_gamma + (k >> 3));
            gw[0] = gv.x;
            gw[1] = gv.y;
            gw[2] = gv.z;
            gw[3] = gv.w;
          }
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float x0 = __uint_as_float(w[i] << 16), x1 = __uint_as_float(w[i] & 0xFFFF0000u);
            const float g0 = __uint_as_float(gw[i] << 16), g1 = __uint_as_float(gw[i] & 0xFFFF0000u);
            __nv_bfloat162 h = __floats2bfloat162_rn((x0 * rs) * g0, (x1 * rs) * g1);
            o[i] = *reinterpret_cast<uint32_t*>(&h);
          }
          *q = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl->xform_full[stage]));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int EPI, int BN, bool NORM_A>
rnl_status launch_epi(const GemmArgs& g, const DeviceInfo& dev, cudaStream_t s, const char* name) {
  auto kern = gemm_kernel<EPI, BN, NORM_A>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, smem_bytes<BN>()) != RNL_OK)
    return RNL_ERR_LAUNCH;
  constexpr bool kBatch = EPI == static_cast<int>(Epi::kDequantBatchSum);
  const int64_t nbatch = kBatch ? g.nbatch : 1;
  CUtensorMap ma, mb;
  rnl_status st =
      make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.A, g.K, g.M * nbatch, g.K * 2, BK, BM);
  if (st != RNL_OK) return st;
  st = make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.B, g.K, g.N * nbatch, g.K * 2, BK, BN);
  if (st != RNL_OK) return st;
  const int64_t tiles = ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN) * nbatch;
  const unsigned grid = static_cast<unsigned>(tiles < dev.sm_count ? tiles : dev.sm_count);
  const uint64_t tag = kBatch ? next_flag_epoch() << 16 : 0;
  trace_before(s);
  const int num_m = static_cast<int>((g.M + BM - 1) / BM);
  const int group_m = (g.M * g.K * 2 <= (int64_t{48} << 20)) ? num_m : (num_m < 8 ? num_m : 8);
  // programmatic dependent launch: the CTAs' set-up overlaps the previous kernel
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<BN>();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, static_cast<int>(g.M),
                                           static_cast<int>(g.N), static_cast<int>(g.K), group_m,
                                           g.out, g.row_scale, g.col_scale, g.a_rstd,
                                           static_cast<const uint4*>(g.a_gamma),
                                           static_cast<const __nv_bfloat16*>(g.bias), g.acc_mode,
                                           g.out_final, static_cast<int>(nbatch), g.batch_flags, tag);
  trace_after(s, g.trace_name ? g.trace_name : name);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

// Per-SM throughput of the one-CTA kernel in full waves on GB300 (measured:
// 1627 and 1594 TFLOP/s over 152 SMs at BN = 256 and 192; 128 estimated).
double one_cta_rate(int bn) { return bn == 256 ? 10.70e12 : (bn == 192 ? 10.49e12 : 9.4e12); }

// Predicted one-CTA time (microseconds) at tile width bn: whole waves of tiles.
double predict_one_cta_us(int64_t M, int64_t N, int64_t K, int sm_count, int bn) {
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const int64_t waves = (tiles + sm_count - 1) / sm_count;
  return waves * (2.0 * BM * bn * static_cast<double>(K) / one_cta_rate(bn)) * 1e6;
}

// Output tile width of the one-CTA kernel: the fastest by predict_one_cta_us.
int pick_bn(int64_t M, int64_t N, int64_t K, int sm_count) {
  const int cand[3] = {256, 192, 128};
  int best = 256;
  double best_t = -1.0;
  for (int bn : cand) {
    const double t = predict_one_cta_us(M, N, K, sm_count, bn);
    if (best_t < 0 || t < best_t) {
      best_t = t;
      best = bn;
    }
  }
  return best;
}

// RNL_GEMM_BN=128|192|256 in the environment overrides the choice (tuning and
// tests); any other value is ignored.
int tile_width(int64_t M, int64_t N, int64_t K, int sm_count) {
  if (const char* e = std::getenv("RNL_GEMM_BN")) {
    const int v = std::atoi(e);
    if (v == 128 || v == 192 || v == 256) return v;
  }
  return pick_bn(M, N, K, sm_count);
}

template <int EPI>
rnl_status launch_bn(const GemmArgs& g, const DeviceInfo& dev, cudaStream_t s, const char* name) {
  // the batched sum mode has nbatch times the tiles of one batch
  const int64_t rows = EPI == static_cast<int>(Epi::kDequantBatchSum) ? g.M * g.nbatch : g.M;
  switch (tile_width(rows, g.N, g.K, dev.sm_count)) {
    case 128: return launch_epi<EPI, 128, false>(g, dev, s, name);
    case 192: return launch_epi<EPI, 192, false>(g, dev, s, name);
    default: return launch_epi<EPI, 256, false>(g, dev, s, name);
  }
}

}  // namespace

bool gemm_uses_pair(int64_t M, int64_t N, int64_t K) {
  DeviceInfo dev;
  if (current_device(&dev) != RNL_OK) return false;
  if (const char* e = std::getenv("RNL_GEMM_PAIR"))
    if (e[0] == '0' || e[0] == '1') return e[0] == '1';
  const int bn = pick_bn(M, N, K, dev.sm_count);
  return N >= 256 && predict_pair_us(M, N, K, dev.sm_count, resident_pairs_for(dev)) <
                         predict_one_cta_us(M, N, K, dev.sm_count, bn);
}

rnl_status launch_gemm(const GemmArgs& g, cudaStream_t s) {
  if (g.M == 0) return RNL_OK;
  if (g.epi == Epi::kBf16QkvRope) return launch_gemm_pair(g, s);  // the epilogue exists there only
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  // Kernel choice for plain GEMMs: the CTA-pair kernel (gemm_pair.cu) when its
  // predicted time beats the best one-CTA tile width.  The exact-integer mode
  // in 1024-product chunks stays on one CTA (measured faster there: the
  // per-chunk accumulator hand-off waits on both CTAs of a pair); with the
  // rows of an RMSNorm quantiser (exact_rows) the pair kernel accumulates
  // every tile whose rows pass the exactness bound in one FP32 accumulator,
  // and the prediction is the plain one.  RNL_GEMM_PAIR=0/1 forces the choice; the fused-norm form
  // always runs here.
  if (g.a_rstd == nullptr) {
    const char* e = std::getenv("RNL_GEMM_PAIR");
    bool pair;
    if (e != nullptr && (e[0] == '0' || e[0] == '1')) {
      pair = e[0] == '1';
    } else {
      const bool integer = (g.epi == Epi::kDequantBf16 && (!g.exact_rows || g.chunk_ws == nullptr)) ||
                           g.epi == Epi::kInt32 || g.epi == Epi::kDequantAccF32 ||
                           g.epi == Epi::kDequantBatchSum;
      const int bn = pick_bn(g.M, g.N, g.K, dev.sm_count);
      pair = !integer && g.N >= 256 &&
             predict_pair_us(g.M, g.N, g.K, dev.sm_count, resident_pairs_for(dev)) <
                 predict_one_cta_us(g.M, g.N, g.K, dev.sm_count, bn);
    }
    const bool int_no_scratch = (g.epi == Epi::kDequantBf16 || g.epi == Epi::kInt32) && g.chunk_ws == nullptr;
    if (pair && g.epi != Epi::kDequantAccF32 && g.epi != Epi::kDequantBatchSum && !int_no_scratch)
      return launch_gemm_pair(g, s);  // one CTA only
  }
  if (g.a_rstd != nullptr) {  // fused norm: bf16 epilogue only
    if (g.epi != Epi::kBf16) return RNL_ERR_ARG;
    switch (tile_width(g.M, g.N, g.K, dev.sm_count)) {
      case 128: return launch_epi<0, 128, true>(g, dev, s, "gemm_bf16_fused_norm");
      case 192: return launch_epi<0, 192, true>(g, dev, s, "gemm_bf16_fused_norm");
      default: return launch_epi<0, 256, true>(g, dev, s, "gemm_bf16_fused_norm");
    }
  }
  switch (g.epi) {
    case Epi::kBf16: return launch_bn<0>(g, dev, s, "gemm_bf16");
    case Epi::kRowScaleF32: return launch_bn<1>(g, dev, s, "gemm_rowscale_f32");
    case Epi::kDequantBf16: return launch_bn<2>(g, dev, s, "gemm_int_dequant");
    case Epi::kInt32: return launch_bn<3>(g, dev, s, "gemm_int_s32");
    case Epi::kDequantAccF32: return launch_bn<4>(g, dev, s, "gemm_int_dequant_acc");
    case Epi::kDequantBatchSum:
      if (g.nbatch < 1 || g.nbatch > 65535 || (g.nbatch > 1 && g.batch_flags == nullptr))
        return RNL_ERR_ARG;
      return launch_bn<5>(g, dev, s, "gemm_int_batch_sum");
    case Epi::kBf16QkvRope: return RNL_ERR_UNSUPPORTED;
  }
  return RNL_ERR_ARG;
}

rnl_status read_clear_error_gemm(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_gemm, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_gemm, &zero, sizeof zero) != cudaSuccess)
    return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
