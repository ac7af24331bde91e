// normstream.cu -- the AT-10 V stage of the two-kernel form as a persistent
// stream: a = bf16((x * rstd) * gamma) for every token row (AT-10 pattern page,
// sec. 2 compute flow and sec. 3 RMSNorm variants), written as the bf16 A
// operand of the GEMM.
//
// The kernel is HBM-bound (read x once, write A once).  One CTA per SM walks
// groups of 8 rows; one producer thread copies each row of a group into a
// shared-memory ring with one bulk copy per row (cp.async.bulk, completion
// counted on the stage's mbarrier), and 8 consumer warps each normalise one
// row of the group from shared memory and store it with coalesced 16-byte
// stores.  The ring holds up to 200 KB, so each SM keeps several row groups
// in flight whatever the occupancy.  The per-row arithmetic is the same as
// norm_cast_kernel (rowwise.cu), element for element and in the same order.
//
// Consumers keep the current row in registers (rows of up to 4096 elements)
// and read gamma from shared memory, so the inner loops carry no global load.
//
// Launched with programmatic dependent launch: the barrier set-up overlaps the
// previous kernel in the stream, every thread then waits for it
// (griddepcontrol.wait), and the kernel lets the next one be scheduled early.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_norm;

constexpr int kGroupRows = 8;  // one row per consumer warp
constexpr int kConsumerWarps = 8;
constexpr int kThreadsNS = (kConsumerWarps + 1) * 32;
constexpr int kMaxNsStages = 16;
constexpr size_t kRingBytes = 200 * 1024;

struct __align__(8) NsCtrl {
  uint64_t full[kMaxNsStages][kGroupRows];  // one barrier per row slot: a warp starts on its row
  uint64_t empty[kMaxNsStages];
  int abort;
};

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// VPL = 16-byte vectors per lane (row of up to 32 * 8 * VPL elements).  Each
// consumer lane keeps its share of the current row in registers between the
// two passes; gamma is staged once per CTA in shared memory.
template <int MODE, bool GAMMA, int VPL>
__global__ void __launch_bounds__(kThreadsNS, 1)
    norm_cast_stream_kernel(const uint8_t* __restrict__ x, const uint4* __restrict__ gamma,
                            int64_t T, int nvec, int stages, float inv_d, float eps,
                            uint4* __restrict__ A) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 127u) & ~127u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
  const uint32_t stage_bytes = kGroupRows * row_bytes;
  uint4* gamma_s = reinterpret_cast<uint4*>(smem + static_cast<size_t>(stages) * stage_bytes);
  NsCtrl* ctrl = reinterpret_cast<NsCtrl*>(smem + static_cast<size_t>(stages) * stage_bytes + row_bytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t groups = (T + kGroupRows - 1) / kGroupRows;

  grid_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      for (int r = 0; r < kGroupRows; ++r) mbar_init(smem_u32(&ctrl->full[s][r]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), kConsumerWarps);
    }
    ctrl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();  // everything below may touch the previous kernel's data
  volatile int* abort = &ctrl->abort;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
        if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_norm, 31)) break;
        const int64_t row0 = g * kGroupRows;
        const int rows = static_cast<int>(T - row0 < kGroupRows ? T - row0 : kGroupRows);
        const uint32_t dst = base + stage * stage_bytes;
        for (int r = 0; r < rows; ++r) {
          const uint32_t bar = smem_u32(&ctrl->full[stage][r]);
          mbar_arrive_expect_tx(bar, row_bytes);
          bulk_copy_g2s(dst + r * row_bytes, x + (row0 + r) * row_bytes, row_bytes, bar);
        }
        if (++stage == static_cast<uint32_t>(stages)) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    if (GAMMA) {  // gamma staged once in shared memory for all rows
      for (int v = threadIdx.x; v < nvec; v += kConsumerWarps * 32) gamma_s[v] = __ldg(gamma + v);
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    }
    uint32_t stage = 0, phase = 0;
    for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
      const int64_t row = g * kGroupRows + warp;
      if (row < T) {
        const bool got = mbar_wait(smem_u32(&ctrl->full[stage][warp]), phase, abort, &g_err_norm, 32);
        if (!__all_sync(0xFFFFFFFFu, got)) break;
        const uint4* rp = reinterpret_cast<const uint4*>(smem + stage * stage_bytes + warp * row_bytes);
        uint4 xv[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int v = lane + 32 * i;
          xv[i] = v < nvec ? rp[v] : make_uint4(0u, 0u, 0u, 0u);
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          float f[8];
          unpack8(xv[i], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (MODE == 0)
              s = fmaf(f[j], f[j], s);
            else
              s = fmaf(f[j] * f[j], inv_d, s);
          }
        }
        s = warp_sum(s);
        const float rstd = (MODE == 0) ? rsqrtf(s * inv_d + eps) : 1.0f / sqrtf(s + eps);
        uint4* ar = A + row * nvec;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int v = lane + 32 * i;
          if (v >= nvec) break;
          float f[8];
          unpack8(xv[i], f);
          if (GAMMA) {
            float gg[8];
            unpack8(gamma_s[v], gg);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = (f[j] * rstd) * gg[j];
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = f[j] * rstd;
          }
          uint4 o;
          o.x = pack_bf16x2(f[0], f[1]);
          o.y = pack_bf16x2(f[2], f[3]);
          o.z = pack_bf16x2(f[4], f[5]);
          o.w = pack_bf16x2(f[6], f[7]);
          ar[v] = o;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->empty[stage]));
      if (++stage == static_cast<uint32_t>(stages)) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
}

template <int MODE, bool GAMMA, int VPL>
rnl_status launch_ns(const void* x, const void* gamma, int64_t T, int nvec, int stages, float inv_d,
                     float eps, void* A, size_t smem, const DeviceInfo& dev, cudaStream_t s) {
  static bool attr_set[64] = {};
  auto kern = norm_cast_stream_kernel<MODE, GAMMA, VPL>;
  if (!attr_set[dev.device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kRingBytes + 128 + 8192 + sizeof(NsCtrl))) != cudaSuccess)
      return RNL_ERR_LAUNCH;
    attr_set[dev.device] = true;
  }
  const int64_t groups = (T + kGroupRows - 1) / kGroupRows;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(groups < dev.sm_count ? groups : dev.sm_count), 1, 1);
  cfg.blockDim = dim3(kThreadsNS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(x),
                                           static_cast<const uint4*>(gamma), T, nvec, stages,
                                           inv_d, eps, static_cast<uint4*>(A));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

template <int VPL>
rnl_status dispatch_mode(const void* x, const void* gamma, int64_t T, int nvec, int stages,
                         float inv_d, float eps, void* A, size_t smem, const DeviceInfo& dev,
                         cudaStream_t s, int mode) {
  if (mode == RNL_NORM_RSQRT)
    return gamma ? launch_ns<0, true, VPL>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s)
                 : launch_ns<0, false, VPL>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s);
  return gamma ? launch_ns<1, true, VPL>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s)
               : launch_ns<1, false, VPL>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s);
}

}  // namespace

// Rows of up to 4096 elements (16 vectors per lane in registers).
bool norm_cast_stream_fits(int64_t K) { return K % 8 == 0 && K <= 4096; }

rnl_status launch_norm_cast_stream(const void* x, const void* gamma, int64_t T, int64_t K,
                                   float eps, int mode, void* A, cudaStream_t s) {
  if (T == 0) return RNL_OK;
  if (!norm_cast_stream_fits(K)) return RNL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const int nvec = static_cast<int>(K / 8);
  const size_t stage = static_cast<size_t>(kGroupRows) * static_cast<size_t>(K) * 2;
  int stages = static_cast<int>(kRingBytes / stage);
  if (stages > kMaxNsStages) stages = kMaxNsStages;
  const size_t smem = 128 + static_cast<size_t>(stages) * stage + static_cast<size_t>(K) * 2 +
                      sizeof(NsCtrl);
  const float inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  trace_before(s);
  const int vpl = (nvec + 31) / 32;
  if (vpl <= 2)
    st = dispatch_mode<2>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s, mode);
  else if (vpl <= 4)
    st = dispatch_mode<4>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s, mode);
  else if (vpl <= 8)
    st = dispatch_mode<8>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s, mode);
  else
    st = dispatch_mode<16>(x, gamma, T, nvec, stages, inv_d, eps, A, smem, dev, s, mode);
  trace_after(s, "norm_cast");
  return st;
}

rnl_status read_clear_error_norm(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_norm, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_norm, &zero, sizeof zero) != cudaSuccess)
    return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl
