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
// Work list (persistent, one CTA pair per two SMs; P pairs, T tiles): a
// hybrid of data-parallel waves and stream-K.  The first (floor(T/P) - 1) * P
// tiles run data-parallel (pair p takes tiles p, p+P, ..., in the grouped
// order that keeps A and W L2-resident).  The last P to 2P tiles would leave
// most pairs idle in a partial wave, so their k-blocks, flattened tile by
// tile, are cut into P equal contiguous ranges, one per pair (stream-K).  A
// range that starts inside a tile computes a partial sum of that tile (fp32,
// or exact int32 in the integer mode), stores it to its pair's slot of the
// workspace and publishes it with a per-warp flag (a GPU-scope release of a
// per-launch epoch); the pair whose range holds the tile's first k-blocks
// processes that fragment last, waits (bounded) for the flags of the pairs
// that hold the rest and adds their partial sums in its epilogue, in pair
// order.  All pairs of the grid are resident at once (the grid is sized from
// the occupancy of the cluster launch), and a pair only waits for pairs of
// higher index, which never wait on it.
//
// Exact integer mode (W8A8: codes and int8 weights as exact bf16 integers).
// Binary32 holds every integer below 2^24 exactly, so a tile whose rows keep
// 128 sum |q| below 2^24 (the bound on RMSNorm-quantised codes in internal.h,
// kWideRowL1, read from x_scale and max |gamma|) is accumulated over all of K
// in one FP32 accumulator and drained through the FP32 epilogue; any other
// tile is accumulated in chunks of 1024 products, each chunk converted to
// int32 and added into a per-pair scratch slot in global memory.  At the
// start the epilogue warps (idle until their first accumulator) reduce the
// test to one byte per 256-row block and one per work item in shared memory,
// so that the MMA thread reads one byte per item.  Both kinds of tile give
// the exact int32 sums, and the dequant is the same arithmetic on them.
#include <cuda_bf16.h>

#include <atomic>
#include <chrono>
#include <cstdlib>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

using namespace gemm;

__device__ unsigned int g_err_pair;

constexpr int kEpiWarps = 8;

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

// The integer mode's exactness marks (kWideRowL1, internal.h), one byte per
// 256-row block, for up to this many blocks (M <= 262144); larger problems
// run every tile in chunks.  The MMA thread reads them per work item, for the
// first kMaxMarkItems items of its pair from a byte each.
constexpr int kMaxMarkBlocks = 1024;
constexpr int kMaxMarkItems = 256;

struct __align__(8) PairCtrl {
  uint64_t full[kMaxStages];   // even CTA: both CTAs' loads of a stage
  uint64_t empty[kMaxStages];  // each CTA: its stage consumed by the pair MMA
  uint64_t tmem_full[2];       // each CTA: accumulator ready
  uint64_t tmem_empty[2];      // even CTA: both CTAs' epilogues drained it
  uint64_t marks_ready;        // each CTA: block_marks written (one arrival per epilogue warp)
  uint32_t tmem_base;
  int abort;
  uint8_t item_chunked[kMaxMarkItems];  // nonzero: item it of this pair in chunks
  uint8_t block_marks[kMaxMarkBlocks];  // nonzero: a marked row in the 256-row block
};

template <int BN>
constexpr size_t pair_smem_bytes() {
  return 1024 + static_cast<size_t>(PairTile<BN>::kStages) * PairTile<BN>::kStageBytes +
         sizeof(PairCtrl);
}
static_assert(pair_smem_bytes<128>() <= kSmemLimit && pair_smem_bytes<192>() <= kSmemLimit &&
                  pair_smem_bytes<256>() <= kSmemLimit,
              "pipeline stages and control block fit the opt-in shared memory");

// The work list shape (identical in every role and CTA).
struct Sched {
  int num_pairs;
  int dp_tiles;  // tiles [0, dp_tiles) data-parallel, whole
  int sk_tiles;  // tiles [dp_tiles, dp_tiles + sk_tiles) stream-K
  int num_kb;
  __device__ __forceinline__ int dp_items(int pair) const {
    return pair < dp_tiles ? (dp_tiles - pair + num_pairs - 1) / num_pairs : 0;
  }
  // first stream-K unit (k-block of the flattened stream-K tiles) of a pair
  __device__ __forceinline__ int64_t sk_start(int pair) const {
    return static_cast<int64_t>(pair) * sk_tiles * num_kb / num_pairs;
  }
  __device__ __forceinline__ int sk_items(int pair) const {
    const int64_t u0 = sk_start(pair), u1 = sk_start(pair + 1);
    if (u1 <= u0) return 0;
    return static_cast<int>((u1 - 1) / num_kb - u0 / num_kb + 1);
  }
  __device__ __forceinline__ int items(int pair) const { return dp_items(pair) + sk_items(pair); }
};

enum : int {
  kWhole = 0,    // the whole tile: epilogue to the output
  kFinish = 1,   // the tile's first k-blocks: add the other pairs' partial sums, then epilogue
  kPartial = 2,  // a later part of the tile: partial sums to this pair's slot, then the flag
};

struct Work {
  int tile;     // index in the grouped tile order
  int kb0;      // k-block range [kb0, kb1)
  int kb1;
  int kind;
  int sk_tile;  // index among the stream-K tiles, or -1
};

// Item `it` of pair `pair`'s work list.
__device__ __forceinline__ Work work_item(const Sched& sc, int pair, int it) {
  Work w;
  const int ndp = sc.dp_items(pair);
  if (it < ndp) {
    w.tile = pair + it * sc.num_pairs;
    w.kb0 = 0;
    w.kb1 = sc.num_kb;
    w.kind = kWhole;
    w.sk_tile = -1;
    return w;
  }
  const int64_t u0 = sc.sk_start(pair), u1 = sc.sk_start(pair + 1);
  const int t = static_cast<int>(u0 / sc.num_kb) + (it - ndp);
  const int64_t ts = static_cast<int64_t>(t) * sc.num_kb;
  w.kb0 = static_cast<int>(u0 > ts ? u0 - ts : 0);
  w.kb1 = static_cast<int>(u1 < ts + sc.num_kb ? u1 - ts : sc.num_kb);
  w.tile = sc.dp_tiles + t;
  w.sk_tile = t;
  w.kind = w.kb0 > 0 ? kPartial : (w.kb1 < sc.num_kb ? kFinish : kWhole);
  return w;
}

// One past the last pair whose partial sums the finisher `pair` of stream-K
// tile t adds: the pairs after it whose ranges start inside tile t.
__device__ __forceinline__ int partners_end(const Sched& sc, int pair, int t) {
  const int64_t tile_end = static_cast<int64_t>(t + 1) * sc.num_kb;
  int q = pair + 1;
  while (q < sc.num_pairs && sc.sk_start(q) < tile_end) ++q;
  return q;
}

// The QKV split + per-head RMSNorm + RoPE of one 128-wide head of row m, in
// the epilogue (AT-10 pattern page, sec. 6, Qwen3PreAttn): y holds the
// thread's 128 bf16-rounded projection values of the head (columns n_base ..
// n_base + 127).  The same arithmetic as the separate stage (qkvrope.cu):
// r = rsqrt(mean(y^2) + eps), z = bf16((y r) gamma), the rotate-half pairs
// (i, i + 64) are both in this thread; v heads are copied.  A position
// outside [0, P) skips the row's q / k heads and records RNL_ERR_ARG.
__device__ __forceinline__ float bf16r(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// One 128-wide head of one row, read from the accumulator in tensor memory
// (taddr: the warp's lane quarter and column half) with the partners'
// partial sums added (stream-K finishers); ss: the sum of squares of its
// bf16-rounded values (pass 1, during the drain); p: the row's position.  v
// heads are copied; q and k heads are normalised and rotated, two 32-column
// groups (c, c + 2) at a time, so that only 64 values are live.  Called by
// the whole warp: the tensor-memory loads are warp-collective, so every lane
// takes them and only the lanes of valid rows (row_ok, a position inside the
// table) compute and store.
__device__ __forceinline__ void rope_head_tmem(uint32_t taddr, const uint32_t* partial_w, int64_t slot_words,
                                               int q0, int q1, float ss, int p, bool row_ok, int64_t m,
                                               int n_base, int N, const RopeEpiArgs& a, unsigned int* err) {
  constexpr int D = 128;
  if (n_base >= N) return;  // the same on every lane
  const int h = n_base / D;
  const int nqk = a.Hq + a.Hkv;
  auto group = [&](int c, uint32_t (&r)[32]) {
    tmem_ld_32cols(taddr + c * 32, r);  // every lane
    tmem_ld_wait();
    for (int q = q0; q < q1 && row_ok; ++q) {
      const uint32_t* src = partial_w + q * slot_words;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t v[8];
        ld_global_v8(src + (c * 4 + j) * 256, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          r[8 * j + i] = __float_as_uint(__uint_as_float(r[8 * j + i]) + __uint_as_float(v[i]));
      }
    }
  };
  if (h >= nqk) {  // v head: copied
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.v) + (m * a.Hkv + (h - nqk)) * D);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      group(c, r);
      if (!row_ok) continue;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o[i] = bf16x2_bits(__uint_as_float(r[8 * q8 + 2 * i]), __uint_as_float(r[8 * q8 + 2 * i + 1]));
        dst[c * 4 + q8] = make_uint4(o[0], o[1], o[2], o[3]);  // 16-byte stores: q, k, v are 16-byte aligned
      }
    }
    return;
  }
  const bool pos_ok = p >= 0 && p < a.P;
  if (row_ok && !pos_ok) atomicCAS(err, 0u, kErrArg | (40u << 8));
  const bool work = row_ok && pos_ok;  // this lane's row is normalised, rotated and stored
  const bool is_q = h < a.Hq;
  const uint4* g4 = static_cast<const uint4*>(is_q ? a.q_gamma : a.k_gamma);
  const float r = rsqrtf(ss * (1.0f / D) + a.eps);
  const float4* row = reinterpret_cast<const float4*>(a.cos_sin + static_cast<int64_t>(work ? p : 0) * D);
  __nv_bfloat16* dst = is_q ? static_cast<__nv_bfloat16*>(a.q) + (m * a.Hq + h) * D
                            : static_cast<__nv_bfloat16*>(a.k) + (m * a.Hkv + (h - a.Hq)) * D;
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t ylo[32], yhi[32];  // columns 32 c .. and their rotation partners 64 + 32 c ..
    group(c, ylo);
    group(c + 2, yhi);
    if (!work) continue;
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8) {
      const int i0 = c * 32 + q8 * 8;  // elements i0 .. i0 + 7 and their partners + 64
      const uint4 gl = __ldg(g4 + i0 / 8), gh = __ldg(g4 + (i0 + 64) / 8);
      const float4 c0 = __ldg(row + i0 / 4), c1 = __ldg(row + i0 / 4 + 1);
      const float4 s0 = __ldg(row + (i0 + 64) / 4), s1 = __ldg(row + (i0 + 64) / 4 + 1);
      const float co[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const float si[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      const uint32_t glw[4] = {gl.x, gl.y, gl.z, gl.w}, ghw[4] = {gh.x, gh.y, gh.z, gh.w};
      uint32_t ol[4], oh[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        float lo[2], hi[2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          const int e = 2 * e2 + t2;
          const float g_lo = __uint_as_float(t2 ? (glw[e2] & 0xFFFF0000u) : (glw[e2] << 16));
          const float g_hi = __uint_as_float(t2 ? (ghw[e2] & 0xFFFF0000u) : (ghw[e2] << 16));
          const float yl = bf16r(__uint_as_float(ylo[q8 * 8 + e]));
          const float yh = bf16r(__uint_as_float(yhi[q8 * 8 + e]));
          const float zl = bf16r(__fmul_rn(__fmul_rn(yl, r), g_lo));
          const float zh = bf16r(__fmul_rn(__fmul_rn(yh, r), g_hi));
          lo[t2] = __fsub_rn(__fmul_rn(zl, co[e]), __fmul_rn(zh, si[e]));
          hi[t2] = __fadd_rn(__fmul_rn(zh, co[e]), __fmul_rn(zl, si[e]));
        }
        ol[e2] = bf16x2_bits(lo[0], lo[1]);
        oh[e2] = bf16x2_bits(hi[0], hi[1]);
      }
      *reinterpret_cast<uint4*>(dst + i0) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
      *reinterpret_cast<uint4*>(dst + i0 + 64) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    }
  }
}

template <int EPI, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b, int M, int N, int K, int group_m,
                     int dp_tiles, int sk_tiles, void* __restrict__ out,
                     const float* __restrict__ row_scale, const float* __restrict__ col_scale,
                     const float* __restrict__ gamma_max, int exact_rows, uint32_t* chunk_ws,
                     uint32_t* partial, uint64_t* flags, uint64_t epoch,
                     const __nv_bfloat16* __restrict__ bias, const RopeEpiArgs rope) {
  constexpr bool kInt = (EPI == static_cast<int>(Epi::kDequantBf16) ||
                         EPI == static_cast<int>(Epi::kInt32));
  constexpr bool kRope = EPI == static_cast<int>(Epi::kBf16QkvRope);
  static_assert(!kRope || BN == 256, "the rope epilogue takes one 128-wide head per warp");
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
  Sched sc;
  sc.num_pairs = num_pairs;
  sc.dp_tiles = dp_tiles;
  sc.sk_tiles = sk_tiles;
  sc.num_kb = num_kb;
  const int n_items = sc.items(pair);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->tmem_full[b]), 1);
      mbar_init(smem_u32(&ctrl->tmem_empty[b]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(&ctrl->marks_ready), kEpiWarps);
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
        const Work w = work_item(sc, pair, it);
        int mb, nb;
        tile_coords(w.tile, num_m, num_n, group_m, mb, nb);
        if (!RNL_DCHECK(&g_err_pair, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n && w.kb0 >= 0 &&
                                         w.kb0 < w.kb1 && w.kb1 <= num_kb, 70))
          break;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait_cluster(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_pair, 21)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * kStageBytes;
          if (!RNL_DCHECK(&g_err_pair, stage < static_cast<uint32_t>(kStages) &&
                                           sa + kStageBytes <= base + kStages * kStageBytes, 71)) {
            ok = false;
            break;
          }
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
      // the per-item marks, written by this CTA's epilogue warps at the start
      if (kInt && exact_rows)
        ok = mbar_wait(smem_u32(&ctrl->marks_ready), 0u, abort, &g_err_pair, 27);
      for (int it = 0; it < n_items && ok; ++it) {
        const Work w = work_item(sc, pair, it);
        bool chunked = kInt;
        if (kInt && exact_rows) {
          if (it < kMaxMarkItems) {
            chunked = ctrl->item_chunked[it] != 0;
          } else {
            int mb, nb;
            tile_coords(w.tile, num_m, num_n, group_m, mb, nb);
            chunked = ctrl->block_marks[mb] != 0;
          }
        }
        const int kb_per_unit = chunked ? kChunkKBlocks : (w.kb1 - w.kb0);
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
          if (!RNL_DCHECK(&g_err_pair, buf * kAccStride + BN <= kTmemCols, 72)) {
            ok = false;
            break;
          }
          const int kb0 = w.kb0 + u * kb_per_unit;
          const int kb1 = min(w.kb1, kb0 + kb_per_unit);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_cluster(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_pair, 23)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = base + stage * kStageBytes;
            if (!RNL_DCHECK(&g_err_pair, stage < static_cast<uint32_t>(kStages), 73)) {
              ok = false;
              break;
            }
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
    if (kInt && exact_rows) {
      // one byte per 256-row block: does the block hold a row whose x_scale
      // is not above exact_row_floor (a row that may need the chunks)?  The
      // epilogue waits for its first accumulator anyway; four blocks per
      // warp at a time, all loads issued before any vote.
      const float gmx = gamma_max != nullptr ? __ldg(gamma_max) : 1.0f;  // loaded beside the x_scale values
      for (int b0 = ew; b0 < num_m; b0 += 4 * kEpiWarps) {
        float xs[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t r = static_cast<int64_t>(b0 + i * kEpiWarps) * 2 * BM + 8 * lane;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            xs[i][j] = (b0 + i * kEpiWarps < num_m && r + j < M) ? __ldg(row_scale + r + j) : INFINITY;
        }
        const float floor_xs = exact_row_floor(static_cast<float>(K), gmx);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          bool wide = false;
#pragma unroll
          for (int j = 0; j < 8; ++j) wide |= !(xs[i][j] > floor_xs);  // NaN: wide
          const int b = b0 + i * kEpiWarps;
          wide = __any_sync(0xFFFFFFFFu, wide);
          if (b < num_m && lane == 0 && RNL_DCHECK(&g_err_pair, b < kMaxMarkBlocks, 77))
            ctrl->block_marks[b] = wide ? 1 : 0;
        }
      }
      // then one byte per work item of this pair, for the MMA thread (the
      // epilogue warps, 256 threads, meet at named barrier 1 first)
      asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
      for (int i = ew * 32 + lane; i < n_items && i < kMaxMarkItems; i += kEpiWarps * 32) {
        const Work wi = work_item(sc, pair, i);
        int mb, nb;
        tile_coords(wi.tile, num_m, num_n, group_m, mb, nb);
        ctrl->item_chunked[i] = ctrl->block_marks[mb];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->marks_ready));
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&ctrl->marks_ready), 0u, abort, &g_err_pair, 27));
    }
    for (int it = 0; it < n_items && ok; ++it) {
      const Work w = work_item(sc, pair, it);
      int mb, nb;
      tile_coords(w.tile, num_m, num_n, group_m, mb, nb);
      if (!RNL_DCHECK(&g_err_pair, mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, 75)) {
        ok = false;
        break;
      }
      // the integer mode accumulates in 1024-product chunks only where a row
      // of the tile may need it (the MMA thread takes the same decision)
      const bool chunked = kInt && (!exact_rows || ctrl->block_marks[mb] != 0);
      const int kb_per_unit = chunked ? kChunkKBlocks : (w.kb1 - w.kb0);
      const int units = (w.kb1 - w.kb0 + kb_per_unit - 1) / kb_per_unit;
      // partial slots: [pair][rank][epilogue warp][32-byte chunk][lane] words,
      // lane-major so that one warp instruction moves 1 KB of contiguous
      // memory; only the same warp and lane of the finisher read a chunk back
      const int64_t slot_words = static_cast<int64_t>(2) * BM * BN;
      const int64_t warp_off = (static_cast<int64_t>(rank) * kEpiWarps + ew) * 32 * kColsPerEpiWarp +
                               lane * 8;
      uint32_t* prow = w.kind == kPartial ? partial + pair * slot_words + warp_off : nullptr;
      // a finisher adds the partial sums of pairs [pair + 1, q_end)
      const int q_end = w.kind == kFinish ? partners_end(sc, pair, w.sk_tile) : pair + 1;
      // the host gives kMaxPartialSlots slots of slot_words words: one per pair
      // (grid <= kMaxPartialSlots - 1 pairs), the flags in the last one; the
      // highest word a warp touches is warp_off + (kGroups * 4 - 1) * 256 + 7
      if (!RNL_DCHECK(&g_err_pair,
                      (w.kind == kWhole || (partial != nullptr && flags != nullptr)) &&
                          (!chunked || chunk_ws != nullptr) &&
                          q_end <= kMaxPartialSlots - 1 && pair < kMaxPartialSlots - 1 &&
                          warp_off + (kGroups * 4 - 1) * 256 + 8 <= slot_words &&
                          (static_cast<int64_t>(q_end) * 2 + 1) * kEpiWarps <= slot_words / 2,
                      74)) {
        ok = false;
        break;
      }
      if (w.kind == kFinish) {
        // this warp reads only the words the same warp of each partner wrote
        bool got = true;
        for (int q = pair + 1; q < q_end && got; ++q)
          got = flag_wait(flags + (static_cast<int64_t>(q) * 2 + rank) * kEpiWarps + ew, epoch, abort,
                          &g_err_pair, 25);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
      }
      const int64_t m = static_cast<int64_t>(mb) * 2 * BM + rank * BM + row_local;
      const int n_base = nb * BN + half * kColsPerEpiWarp;
      const bool row_ok = m < M;
      float rs = 0.f;
      if ((EPI == static_cast<int>(Epi::kRowScaleF32) ||
           EPI == static_cast<int>(Epi::kDequantBf16)) && row_ok)
        rs = row_scale != nullptr ? __ldg(row_scale + m) : 1.0f;
      int rope_p = 0;  // the row's position, loaded before the drain
      if (kRope && row_ok && prow == nullptr) rope_p = __ldg(rope.pos + m);
      // the accumulator of unit u: wait until the pair's MMAs have filled it
      auto acc_wait = [&](uint32_t buf, uint32_t use) -> bool {
        const bool got = mbar_wait_cluster(smem_u32(&ctrl->tmem_full[buf]), use & 1u, abort,
                                           &g_err_pair, 24);
        if (!__all_sync(0xFFFFFFFFu, got)) return false;
        tc_fence_after();
        return RNL_DCHECK(&g_err_pair, buf * kAccStride + (half + 1) * kColsPerEpiWarp <= kTmemCols, 76);
      };
      // ... and hand it back to the MMA thread once drained
      auto acc_release = [&](uint32_t buf) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(smem_u32(&ctrl->tmem_empty[buf]));
          else
            mbar_arrive_cluster(buf ? empty_even_1 : empty_even_0);
        }
      };
      // chunked tiles: the int32 sums of the chunks so far, per thread, in
      // this pair's scratch slot (same lane-major layout as the partials)
      uint32_t* cws = chunked ? chunk_ws + pair * slot_words + warp_off : nullptr;
      float ss = 0.f;  // the rope epilogue's sum of squares of the head's bf16-rounded values
      for (int u = 0; u < units; ++u, ++unit) {
        const uint32_t buf = unit & 1u;
        if (!acc_wait(buf, unit >> 1)) {
          ok = false;
          break;
        }
        if (kInt && chunked) {
          // -------- exact int32 sums of the 1024-product chunks: the running
          // sums in the scratch slot, the last chunk's to the partial slot or
          // (with the partners' partial sums) to the output
          const bool last = u + 1 == units;
          uint32_t* dst = last ? prow : cws;
#pragma unroll
          for (int c = 0; c < kGroups; ++c) {
            uint32_t r[32];
            tmem_ld_32cols(tmem_base + lane_addr + buf * kAccStride + half * kColsPerEpiWarp + c * 32, r);
            tmem_ld_wait();
            // the int32 sums in the same registers (two's complement bits)
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[j])));
            if (u > 0) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t v[8];
                ld_global_v8(cws + (c * 4 + j) * 256, v);
#pragma unroll
                for (int i = 0; i < 8; ++i) r[8 * j + i] += v[i];
              }
            }
            if (dst != nullptr) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = r[8 * j + i];
                st_global_v8(dst + (c * 4 + j) * 256, v);
              }
            } else if (row_ok) {
              // the partners' exact int32 partial sums, in pair order
              for (int q = pair + 1; q < q_end; ++q) {
                const uint32_t* src = partial + q * slot_words + warp_off;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t v[8];
                  ld_global_v8(src + (c * 4 + j) * 256, v);
#pragma unroll
                  for (int i = 0; i < 8; ++i) r[8 * j + i] += v[i];
                }
              }
              const int(&a)[32] = reinterpret_cast<const int(&)[32]>(r);
              if constexpr (EPI == static_cast<int>(Epi::kInt32))
                store_i32_32(out, m, n_base + c * 32, N, a);
              else
                store_dequant_32(out, m, n_base + c * 32, N, a, rs, col_scale, bias);
            }
          }
        } else {
          // -------- one FP32 accumulator (in the integer mode: the exact sum)
#pragma unroll
          for (int c = 0; c < kGroups; ++c) {
            uint32_t r[32];
            tmem_ld_32cols(tmem_base + lane_addr + buf * kAccStride + half * kColsPerEpiWarp + c * 32, r);
            tmem_ld_wait();
            const int n0 = n_base + c * 32;
            if (prow != nullptr) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = r[8 * j + i];
                st_global_v8(prow + (c * 4 + j) * 256, v);
              }
            } else {
              if (row_ok) {
                // the partners' fp32 partial sums, added in pair order (plain
                // loads: they were written during this grid); in the integer
                // mode they are exact integers, and so is every sum of them
                for (int q = pair + 1; q < q_end; ++q) {
                  const uint32_t* src = partial + q * slot_words + warp_off;
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    uint32_t v[8];
                    ld_global_v8(src + (c * 4 + j) * 256, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                      r[8 * j + i] = __float_as_uint(__uint_as_float(r[8 * j + i]) + __uint_as_float(v[i]));
                  }
                }
              }
              if constexpr (kRope) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const float v = bf16r(__uint_as_float(r[j]));
                  ss = fmaf(v, v, ss);
                }
              } else if constexpr (EPI == static_cast<int>(Epi::kBf16)) {
                if (row_ok) {
                  if (bias != nullptr)
                    store_bf16_bias_32(out, m, n0, N, r, bias);
                  else
                    store_bf16_32(out, m, n0, N, r);
                }
              } else if constexpr (EPI == static_cast<int>(Epi::kDequantBf16)) {
                if (row_ok) store_dequant_f32_32(out, m, n0, N, r, rs, col_scale, bias);
              } else if constexpr (EPI == static_cast<int>(Epi::kInt32)) {
                if (row_ok) {
                  int a[32];
#pragma unroll
                  for (int j = 0; j < 32; ++j) a[j] = __float2int_rn(__uint_as_float(r[j]));
                  store_i32_32(out, m, n0, N, a);
                }
              } else {
                if (row_ok) store_f32_scaled_32(out, m, n0, N, r, rs);
              }
            }
          }
        }
        if constexpr (kRope) {  // pass 2, from the accumulator still held (the whole warp)
          if (prow == nullptr)
            rope_head_tmem(tmem_base + lane_addr + buf * kAccStride + half * kColsPerEpiWarp, partial + warp_off,
                           slot_words, pair + 1, q_end, ss, rope_p, row_ok, m, n_base, N, rope, &g_err_pair);
        }
        acc_release(buf);
      }
      if (!ok) break;
      if (w.kind == kFinish) {
        // every flag published in a launch is consumed by exactly one
        // finisher warp, which sets it back to 0 once the partial sums are
        // read: a later launch with the same epoch (a replayed CUDA graph)
        // then waits for flags published in that launch
        __syncwarp();
        if (lane == 0)
          for (int q = pair + 1; q < q_end; ++q)
            flags[(static_cast<int64_t>(q) * 2 + rank) * kEpiWarps + ew] = 0;
      }
      if (w.kind == kPartial) {
        // every lane orders its partial stores, then one lane publishes this
        // warp's flag (release)
        __threadfence();
        __syncwarp();
        if (lane == 0)
          flag_release(flags + (static_cast<int64_t>(pair) * 2 + rank) * kEpiWarps + ew, epoch);
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
// Work-list shape for T tiles on P pairs: (floor(T/P) - 1) full data-parallel
// waves, the remaining P .. 2P - 1 tiles stream-K (every tile then spans at
// most two pairs' ranges, so a finisher adds at most one partner's partial
// sums).  Fewer than 2P tiles: all stream-K.  Without a workspace for the
// partial sums: every tile whole, data-parallel.
struct Plan {
  int dp_tiles = 0;
  int sk_tiles = 0;
};

Plan make_plan(int64_t tiles, int pairs, bool have_partials) {
  Plan pl;
  if (!have_partials) {
    pl.dp_tiles = static_cast<int>(tiles);
    return pl;
  }
  const int64_t waves = tiles / pairs;
  const int64_t dp_waves = waves > 1 ? waves - 1 : 0;
  pl.dp_tiles = static_cast<int>(dp_waves * pairs);
  pl.sk_tiles = static_cast<int>(tiles - pl.dp_tiles);
  return pl;
}

// Pairs to launch: with stream-K every resident pair, as long as each range
// keeps at least 8 k-blocks (fewer pairs for tiny problems); without partial
// sums at most one pair per tile.
int grid_pairs(int64_t tiles, int num_kb, int max_pairs, bool have_partials) {
  int64_t p = tiles;
  if (have_partials) {
    const int64_t by_units = tiles * num_kb / 8;
    p = by_units > tiles ? by_units : tiles;
  }
  if (p > max_pairs) p = max_pairs;
  if (p > kMaxPartialSlots - 1) p = kMaxPartialSlots - 1;
  return static_cast<int>(p < 1 ? 1 : p);
}

// Epoch of each launch: a per-process start value from the clock, then one
// step per launch, so a flag left in a reused workspace by an earlier launch
// (or process) never matches.  A launch captured in a CUDA graph keeps its
// epoch on every replay; there the finishers' reset of every consumed flag
// to 0 is what keeps a replay from reading the previous replay's flags.
template <int EPI, int BN>
rnl_status launch_pair_bn(const GemmArgs& g, const DeviceInfo& dev, int max_pairs, cudaStream_t s,
                          const char* name) {
  auto kern = gemm_pair_kernel<EPI, BN>;
  const size_t smem = pair_smem_bytes<BN>();
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, smem) != RNL_OK)
    return RNL_ERR_LAUNCH;
  CUtensorMap ma, mb;
  rnl_status st = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.A, g.K, g.M, g.K * 2, BK, BM);
  if (st != RNL_OK) return st;
  st = make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.B, g.K, g.N, g.K * 2, BK,
                   PairTile<BN>::kBHalf);
  if (st != RNL_OK) return st;
  const int num_m = static_cast<int>((g.M + 2 * BM - 1) / (2 * BM));
  const int num_kb = static_cast<int>((g.K + BK - 1) / BK);
  const int64_t tiles = static_cast<int64_t>(num_m) * ((g.N + BN - 1) / BN);
  // partial sums: one slot of 2 x 128 x BN words per pair, the flags in the
  // last slot of the workspace (room for kMaxPartialSlots - 1 pairs)
  const size_t slot_bytes = static_cast<size_t>(2) * BM * BN * 4;
  const bool have_partials = g.partial_ws != nullptr &&
                             g.partial_ws_bytes >= kMaxPartialSlots * slot_bytes;
  const int pairs = grid_pairs(tiles, num_kb, max_pairs, have_partials);
  // the exactness marks serve up to kMaxMarkBlocks 256-row blocks
  const int exact_rows = (g.exact_rows && g.row_scale != nullptr && num_m <= kMaxMarkBlocks &&
                          exact_rows_possible(g.K)) ? 1 : 0;
  // the integer mode's chunked tiles keep their running int32 sums in one
  // scratch slot per pair
  constexpr bool kInt = EPI == static_cast<int>(Epi::kDequantBf16) || EPI == static_cast<int>(Epi::kInt32);
  if (kInt && (g.chunk_ws == nullptr || g.chunk_ws_bytes < static_cast<size_t>(pairs) * slot_bytes))
    return RNL_ERR_WORKSPACE;
  const Plan pl = make_plan(tiles, pairs, have_partials);
  uint32_t* partial = static_cast<uint32_t*>(g.partial_ws);
  uint64_t* flags = have_partials ? reinterpret_cast<uint64_t*>(static_cast<char*>(g.partial_ws) +
                                                                (kMaxPartialSlots - 1) * slot_bytes)
                                  : nullptr;
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, static_cast<int>(g.M),
                                           static_cast<int>(g.N), static_cast<int>(g.K), group_m,
                                           pl.dp_tiles, pl.sk_tiles, g.out, g.row_scale,
                                           g.col_scale, g.gamma_max, exact_rows, static_cast<uint32_t*>(g.chunk_ws),
                                           partial, flags, next_flag_epoch(),
                                           static_cast<const __nv_bfloat16*>(g.bias), g.rope);
  trace_after(s, g.trace_name ? g.trace_name : name);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

// Largest number of CTA pairs that can be resident at once.
int resident_pairs(const DeviceInfo& dev) {
  static std::atomic<int> cached[64];  // 0 until measured; racing first calls store the same value
  const int c = cached[dev.device].load(std::memory_order_relaxed);
  if (c > 0) return c;
  auto kern = gemm_pair_kernel<0, 256>;
  int n = 0;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, pair_smem_bytes<256>()) ==
      RNL_OK) {
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
  cached[dev.device].store(n, std::memory_order_relaxed);
  return n;
}

template <int EPI>
rnl_status launch_pair_epi(const GemmArgs& g, const DeviceInfo& dev, cudaStream_t s,
                           const char* name) {
  const int pairs = resident_pairs(dev);
  if constexpr (EPI == static_cast<int>(Epi::kBf16QkvRope)) {
    return launch_pair_bn<EPI, 256>(g, dev, pairs, s, name);  // one 128-wide head per warp
  } else {
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
}

}  // namespace

// Predicted time of the pair kernel (256-wide tiles) in microseconds, from
// the per-SM rate it sustained on GB300 in full waves (1909 TFLOP/s over 152
// SMs): every pair's share of the k-blocks, plus the stream-K hand-off when
// the tiles do not fill whole waves: about 2 us after data-parallel waves (a
// partner's partial is its first, short item), about 20 us when every tile is
// split (fewer than 2P tiles: a partner's partial is its whole range, so the
// finisher waits for it, then drains; measured on the MLA q_a shape,
// 2048 x 1536 x 7168: 43 us against 39 us on one CTA).
double predict_pair_us(int64_t M, int64_t N, int64_t K, int sm_count, int pairs_hint) {
  const int pairs = pairs_hint > 0 ? pairs_hint : sm_count / 2;
  const int64_t num_m = (M + 2 * BM - 1) / (2 * BM);
  const int64_t tiles = num_m * ((N + 255) / 256);
  const int num_kb = static_cast<int>((K + BK - 1) / BK);
  const int p = grid_pairs(tiles, num_kb, pairs, true);
  const double tile_us = 2.0 * BM * 256 * static_cast<double>(K) / 12.56e12 * 1e6;
  const Plan pl = make_plan(tiles, p, true);
  double t = (static_cast<double>(pl.dp_tiles) / p + static_cast<double>(pl.sk_tiles) / p) * tile_us;
  if (pl.sk_tiles % p != 0) t += pl.dp_tiles > 0 ? 2.0 : 20.0;
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
    case Epi::kBf16QkvRope: return launch_pair_epi<6>(g, dev, s, "gemm_pair_qkv_rope");
    case Epi::kDequantAccF32:
    case Epi::kDequantBatchSum: return RNL_ERR_UNSUPPORTED;  // one-CTA kernel only
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

uint64_t next_flag_epoch() {
  static std::atomic<uint64_t> counter{
      static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) * 2654435761ull};
  const uint64_t e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  return e != 0 ? e : 1;  // 0 is the value of a consumed flag
}

}  // namespace rnl
