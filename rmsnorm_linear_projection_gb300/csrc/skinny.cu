// skinny.cu -- the mhc_pre form: huge reduction K x tiny output width N <= 64,
// no gamma, FP32 compute and FP32 output (AT-10 pattern page, sec. 8; the
// "SK-03 Linear Projection (Norm->MatMul)" page, "shape variant: huge
// reduction x tiny output width").
//
// Without gamma the norm is one scalar per row, so it commutes with the
// projection:  sum_k (x[t,k] * rstd_t) * W[n,k] = rstd_t * sum_k x[t,k] * W[n,k].
// One pass over x therefore gives both sum_k x^2 and the N dot products.
// The work is HBM-bound (x is read once; W is small and stays in L2), so the
// kernel is a stream:
//   * the (row tile, k-block) steps are laid out row-major and split into one
//     contiguous range per CTA (one CTA per SM), so every SM streams the same
//     number of 16 KB x tiles whatever T and K are (the split-K of the pages,
//     balanced over the SMs);
//   * warp 0 streams 128x64 x tiles and the 32x64 (or 64x64) W tile by TMA
//     through an 8-stage ring;
//   * warp 1 issues tcgen05.mma (M=128, N=32/64, K=16) into a TMEM
//     accumulator, restarted at each row-tile boundary of the CTA's range;
//   * warps 2-5 (one thread per row) add up x^2 from the same shared-memory
//     tile, and at the end of each row-tile segment write the segment's
//     partial dot products and partial sum of squares to the workspace.
// A second small kernel adds the segments of each row in CTA order
// (deterministic) and applies rstd.  It is launched as the stream kernel's
// programmatic dependent: its CTAs are scheduled while the stream runs and
// wait (griddepcontrol.wait) for the stream grid's completion and memory
// before they read the partial records, so its launch latency is hidden.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_skinny;

constexpr int SM_ROWS = 128;
constexpr int SK = 64;
constexpr int kStages = 8;
constexpr int kStatWarps = 4;
constexpr int kThreads = 64 + kStatWarps * 32;
constexpr uint32_t kXBytes = SM_ROWS * SK * 2;  // 16 KB
constexpr int kMaxCtas = 512;

struct __align__(8) Ctrl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
};

template <int NP>
constexpr uint32_t w_bytes() { return NP * SK * 2; }
template <int NP>
constexpr uint32_t stage_bytes() { return kXBytes + w_bytes<NP>(); }
template <int NP>
constexpr size_t smem_bytes() { return 1024 + static_cast<size_t>(kStages) * stage_bytes<NP>() + sizeof(Ctrl); }

// Partial records: record (cta c, row tile r) lives at index r + c, which is
// unique because each CTA's tiles start at or after the previous CTA's last.
__device__ __forceinline__ int64_t range_begin(int c, int64_t total, int G) {
  return (total * c) / G;
}

template <int NP, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                  int T, int K, float inv_d, float* __restrict__ part) {
  constexpr uint32_t kStage = stage_bytes<NP>();
  constexpr int kRec = NP + 1;  // NP partial dot products + partial sum of squares
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kStages * kStage);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kbpr = (K + SK - 1) / SK;  // k-blocks per row tile
  const int64_t total = static_cast<int64_t>((T + SM_ROWS - 1) / SM_ROWS) * kbpr;
  const int G = gridDim.x;
  const int64_t s_begin = range_begin(blockIdx.x, total, G);
  const int64_t s_end = range_begin(blockIdx.x + 1, total, G);

  grid_launch_dependents();  // the reduce kernel may be scheduled now; it waits for this grid
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1 + kStatWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->acc_full[b]), 1);
      mbar_init(smem_u32(&ctrl->acc_empty[b]), kStatWarps);
    }
    ctrl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl->tmem_base), 2 * NP);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort = &ctrl->abort;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&map_x);
      tma_prefetch_map(&map_w);
      const uint64_t pol_x = l2_policy_evict_first();  // x is read exactly once
      const uint64_t pol_w = l2_policy_evict_last();   // W is re-read by every CTA
      uint32_t stage = 0, phase = 0;
      for (int64_t st = s_begin; st < s_end; ++st) {
        if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_skinny, 11)) break;
        const int r = static_cast<int>(st / kbpr);
        const int kb = static_cast<int>(st - static_cast<int64_t>(r) * kbpr);
        const uint32_t sx = base + stage * kStage;
        if (!RNL_DCHECK(&g_err_skinny, stage < static_cast<uint32_t>(kStages) && st < total &&
                                           r * SM_ROWS < T && kb * SK < K, 80))
          break;
        const uint32_t bar = smem_u32(&ctrl->full[stage]);
        mbar_arrive_expect_tx(bar, kStage);
        tma_load_2d_hint(sx, &map_x, bar, kb * SK, r * SM_ROWS, pol_x);
        tma_load_2d_hint(sx + kXBytes, &map_w, bar, kb * SK, 0, pol_w);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(SM_ROWS, NP);
      uint32_t stage = 0, phase = 0, seg = 0;
      bool ok = true;
      int64_t st = s_begin;
      while (st < s_end && ok) {
        const int r = static_cast<int>(st / kbpr);
        const int64_t seg_end = min(s_end, static_cast<int64_t>(r + 1) * kbpr);
        const uint32_t buf = seg & 1u;
        const uint32_t use = seg >> 1;
        if (!mbar_wait(smem_u32(&ctrl->acc_empty[buf]), (use & 1u) ^ 1u, abort, &g_err_skinny, 12)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * NP;
        for (int64_t s2 = st; s2 < seg_end; ++s2) {
          if (!mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_skinny, 13)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sx = base + stage * kStage;
          const uint64_t adesc = desc_kmajor_sw128(sx);
          const uint64_t bdesc = desc_kmajor_sw128(sx + kXBytes);
#pragma unroll
          for (int k = 0; k < SK / 16; ++k)
            umma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (s2 > st || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&ctrl->empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&ctrl->acc_full[buf]));
        st = seg_end;
        ++seg;
      }
    }
    __syncwarp();
  } else {
    // statistics + segment epilogue: thread = row of the 128-row tile
    const int quarter = warp & 3;
    const int row_local = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t stage = 0, phase = 0, seg = 0;
    bool ok = true;
    int64_t st = s_begin;
    while (st < s_end && ok) {
      const int r = static_cast<int>(st / kbpr);
      const int64_t seg_end = min(s_end, static_cast<int64_t>(r + 1) * kbpr);
      float ss = 0.f;
      for (int64_t s2 = st; s2 < seg_end; ++s2) {
        const bool got = mbar_wait(smem_u32(&ctrl->full[stage]), phase, abort, &g_err_skinny, 14);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        // the row's 128 bytes.  Thread i starts at 16-byte chunk i % 8 so the
        // eight threads served by one shared-memory wavefront hit eight
        // different bank groups (the order of the chunks does not matter for
        // a sum).
        const uint4* rowp = reinterpret_cast<const uint4*>(smem + stage * kStage + row_local * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 u = rowp[c ^ (row_local & 7)];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float a = __uint_as_float(w[i] << 16);
            const float b = __uint_as_float(w[i] & 0xFFFF0000u);
            if (MODE == 0) {
              ss = fmaf(a, a, ss);
              ss = fmaf(b, b, ss);
            } else {
              ss = fmaf(a * a, inv_d, ss);
              ss = fmaf(b * b, inv_d, ss);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl->empty[stage]));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      const uint32_t buf = seg & 1u;
      const uint32_t use = seg >> 1;
      const bool got = mbar_wait(smem_u32(&ctrl->acc_full[buf]), use & 1u, abort, &g_err_skinny, 15);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      float* rec = part + ((static_cast<int64_t>(r) + blockIdx.x) * SM_ROWS + row_local) * kRec;
      // records hold ceil(T / 128) + gridDim.x row tiles (the host's sizing)
      if (!RNL_DCHECK(&g_err_skinny, static_cast<int64_t>(r) + blockIdx.x <
                                         static_cast<int64_t>((T + SM_ROWS - 1) / SM_ROWS) + gridDim.x &&
                                         buf * NP + NP <= 2 * NP, 81))
        break;
#pragma unroll
      for (int c = 0; c < NP / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32cols(tmem_base + lane_addr + buf * NP + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) rec[c * 32 + j] = __uint_as_float(v[j]);
      }
      rec[NP] = ss;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->acc_empty[buf]));
      st = seg_end;
      ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * NP);
  }
}

// out[t, n] = rstd_t * sum over the CTAs covering row t of the partials.
template <int NP, int MODE>
__global__ void __launch_bounds__(128)
    skinny_reduce_kernel(const float* __restrict__ part, int T, int K, int N, int G, float inv_d,
                         float eps, float* __restrict__ out) {
  constexpr int kRec = NP + 1;
  grid_dependency_wait();  // the stream grid has completed and its records are visible
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int kbpr = (K + SK - 1) / SK;
  const int64_t total = static_cast<int64_t>((T + SM_ROWS - 1) / SM_ROWS) * kbpr;
  const int r = t / SM_ROWS;
  const int64_t f0 = static_cast<int64_t>(r) * kbpr, f1 = f0 + kbpr;
  float acc[NP];
#pragma unroll
  for (int j = 0; j < NP; ++j) acc[j] = 0.f;
  float ss = 0.f;
  // CTA c covers steps [floor(total*c/G), floor(total*(c+1)/G)); the CTA
  // holding step s is ceil((s+1)*G/total) - 1.
  const int c_first = static_cast<int>(((f0 + 1) * G + total - 1) / total) - 1;
  const int c_last = static_cast<int>((f1 * G + total - 1) / total) - 1;
  for (int c = c_first; c <= c_last && c < G; ++c) {
    const int64_t b = range_begin(c, total, G), e = range_begin(c + 1, total, G);
    if (e <= f0 || b >= f1) continue;
    const float* rec = part + ((static_cast<int64_t>(r) + c) * SM_ROWS + (t - r * SM_ROWS)) * kRec;
    if (!RNL_DCHECK(&g_err_skinny, static_cast<int64_t>(r) + c < static_cast<int64_t>((T + SM_ROWS - 1) / SM_ROWS) + G,
                    82))
      break;
#pragma unroll
    for (int j = 0; j < NP; ++j) acc[j] += rec[j];
    ss += rec[NP];
  }
  const float rstd = (MODE == 0) ? rsqrtf(ss * inv_d + eps) : 1.0f / sqrtf(ss + eps);
  float* orow = out + static_cast<int64_t>(t) * N;
  for (int j = 0; j < N; ++j) orow[j] = acc[j] * rstd;
}

template <int NP, int MODE>
rnl_status launch_np(const void* x, const void* W, int64_t T, int64_t K, int64_t N, float eps,
                     float* out, float* part, int G, const DeviceInfo& dev, cudaStream_t s) {
  auto kern = skinny_kernel<NP, MODE>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, smem_bytes<NP>()) != RNL_OK)
    return RNL_ERR_LAUNCH;
  CUtensorMap mx, mw;
  rnl_status st = make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, T, K * 2, SK, SM_ROWS);
  if (st != RNL_OK) return st;
  st = make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, K, N, K * 2, SK, NP);
  if (st != RNL_OK) return st;
  const float inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  trace_before(s);
  kern<<<G, kThreads, smem_bytes<NP>(), s>>>(mx, mw, static_cast<int>(T), static_cast<int>(K), inv_d, part);
  trace_after(s, "skinny_stream");
  if (cudaGetLastError() != cudaSuccess) return RNL_ERR_LAUNCH;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((T + 127) / 128), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_before(s);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_reduce_kernel<NP, MODE>, static_cast<const float*>(part),
                                           static_cast<int>(T), static_cast<int>(K), static_cast<int>(N), G,
                                           inv_d, eps, out);
  trace_after(s, "skinny_reduce");
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

int grid_for(int64_t T, int64_t K, int sm_count) {
  const int64_t total = ((T + SM_ROWS - 1) / SM_ROWS) * ((K + SK - 1) / SK);
  int64_t g = sm_count < kMaxCtas ? sm_count : kMaxCtas;
  if (g > total) g = total;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

size_t skinny_workspace_bytes(int64_t T, int64_t K, int64_t N, int /*sm_count*/) {
  (void)K;
  const int64_t np = N <= 32 ? 32 : 64;
  const int64_t tiles = (T + SM_ROWS - 1) / SM_ROWS;
  const int64_t records = tiles + kMaxCtas;  // r + c < tiles + G <= tiles + kMaxCtas
  return static_cast<size_t>(records * SM_ROWS * (np + 1) * sizeof(float));
}

rnl_status launch_skinny(const void* x, const void* W, int64_t T, int64_t K, int64_t N, float eps,
                         int mode, float* out, void* workspace, size_t ws_bytes, int sm_count,
                         cudaStream_t s) {
  if (T == 0) return RNL_OK;
  if (ws_bytes < skinny_workspace_bytes(T, K, N, sm_count)) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const int G = grid_for(T, K, dev.sm_count);
  float* part = static_cast<float*>(workspace);
  if (N <= 32)
    return mode == RNL_NORM_RSQRT ? launch_np<32, 0>(x, W, T, K, N, eps, out, part, G, dev, s)
                                  : launch_np<32, 1>(x, W, T, K, N, eps, out, part, G, dev, s);
  return mode == RNL_NORM_RSQRT ? launch_np<64, 0>(x, W, T, K, N, eps, out, part, G, dev, s)
                                : launch_np<64, 1>(x, W, T, K, N, eps, out, part, G, dev, s);
}

rnl_status read_clear_error_skinny(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_skinny, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_skinny, &zero, sizeof zero) != cudaSuccess)
    return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl

// ---------------------------------------------------------------------------
// Allocation-free variant of the mhc_pre path (rmsnorm_linear_skinny_noalloc).
//
// Its scratch (the split-K partial records) lives in this file-scope device
// array instead of a caller-provided workspace.  Every GPU that loads the
// library holds the array until the process exits; all calls on a device
// share it, so it keeps the previous call's contents (every record the
// reduce kernel reads is written earlier in the same call, so nothing has
// to be cleared), and calls that overlap on the GPU race on it.
// ---------------------------------------------------------------------------
namespace rnl {
namespace {

constexpr size_t kStaticScratchBytes = RNL_NOALLOC_SCRATCH_BYTES;  // 16 MiB
static __device__ __align__(256) unsigned char g_skinny_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of g_skinny_scratch for the current device, looked up once
// per device (with that device current) and cached.
rnl_status static_scratch(int device, void** ptr) {
  if (device < 0 || device >= 64) return RNL_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_skinny_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return RNL_ERR_DEVICE;
    }
    g_scratch_ptr[device] = p;
  }
  *ptr = g_scratch_ptr[device];
  return RNL_OK;
}

}  // namespace
}  // namespace rnl

extern "C" rnl_status rmsnorm_linear_skinny_noalloc(const void* x, const void* W, int64_t T,
                                                    int64_t K, int64_t N, float eps,
                                                    int norm_mode, float* out,
                                                    rnl_stream_t stream) {
  using namespace rnl;
  constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
  if (T < 0 || K <= 0 || N <= 0 || T > kMaxDim || K > kMaxDim) return RNL_ERR_SHAPE;
  if (N > 64) return RNL_ERR_UNSUPPORTED;
  if ((norm_mode != RNL_NORM_RSQRT && norm_mode != RNL_NORM_SQRT_DIV) || !(eps >= 0.f) ||
      !(eps <= 3.4e38f))
    return RNL_ERR_ARG;
  if (T == 0) return RNL_OK;
  if (!x || !W || !out) return RNL_ERR_NULL;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (K % 8 != 0 || misaligned(x) || misaligned(W) || misaligned(out)) return RNL_ERR_ALIGN;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  // records actually used: one per (CTA, row tile) pair, at most tiles + G
  const int G = grid_for(T, K, dev.sm_count);
  const int64_t np = N <= 32 ? 32 : 64;
  const int64_t records = (T + SM_ROWS - 1) / SM_ROWS + G;
  const size_t need = static_cast<size_t>(records * SM_ROWS * (np + 1) * sizeof(float));
  if (need > kStaticScratchBytes) return RNL_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = static_scratch(dev.device, &scratch);
  if (st != RNL_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(scratch);
  if (N <= 32)
    return norm_mode == RNL_NORM_RSQRT ? launch_np<32, 0>(x, W, T, K, N, eps, out, part, G, dev, s)
                                       : launch_np<32, 1>(x, W, T, K, N, eps, out, part, G, dev, s);
  return norm_mode == RNL_NORM_RSQRT ? launch_np<64, 0>(x, W, T, K, N, eps, out, part, G, dev, s)
                                     : launch_np<64, 1>(x, W, T, K, N, eps, out, part, G, dev, s);
}
