// normstream.cu -- the AT-10 V stage of the two-kernel form as a persistent
// stream: a = bf16((x * rstd) * gamma) for every token row (AT-10 pattern page,
// sec. 2 compute flow and sec. 3 RMSNorm variants), written as the bf16 A
// operand of the GEMM.
//
// The kernel is HBM-bound (read x once, write A once).  One CTA per SM walks
// its own contiguous range of about T / (number of SMs) rows (equal bytes per
// SM) in groups of 8 rows; one producer thread copies each row of a group into a
// shared-memory ring with one bulk copy per row (cp.async.bulk, completion
// counted on the stage's mbarrier), and 8 consumer warps each normalise one
// row of the group from shared memory and store it with coalesced 16-byte
// stores.  The ring holds up to 200 KB, so each SM keeps several row groups
// in flight whatever the occupancy; where a CTA's whole share of rows fits in
// shared memory, the ring holds all of it and every row is requested at
// once.  The per-row arithmetic is the same as norm_cast_kernel
// (rowwise.cu), element for element and in the same order.
//
// Consumers keep the current row in registers (rows of up to 4096 elements)
// and read gamma from shared memory, so the inner loops carry no global load.
//
// Launched with programmatic dependent launch: the barrier set-up overlaps the
// previous kernel in the stream, every thread then waits for it
// (griddepcontrol.wait), and the kernel lets the next one be scheduled early.
#include <cuda_bf16.h>

#include <algorithm>

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
constexpr size_t kNsSmemLimit = 232448;  // 227 KB opt-in shared memory per block

struct __align__(8) NsCtrl {
  uint64_t full[kMaxNsStages][kGroupRows];  // one barrier per row slot: a warp starts on its row
  uint64_t empty[kMaxNsStages];
  int abort;
};

// Options of the extended form (EXT = true; every pointer may be null): the
// residual row is added first (x_add = bf16(x + residual)), x_add is written
// to x_sum, beta is added after gamma, rstd is written per row.  Each
// consumer warp loads the residual row of its next row from global memory as
// soon as the current row's first pass has used its own, so the load
// overlaps the output pass and the wait for the next x row (the ring holds x
// rows only and keeps its depth).  x_add then replaces the x row in the warp's ring
// slot and the output pass reads it from there, so no row is held in
// registers across the two passes.
struct NsExt {
  const uint4* residual;
  uint4* x_sum;
  const uint4* beta;
  float* rstd_out;
};

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
template <int MODE, bool GAMMA, int VPL, bool EXT>
__global__ void __launch_bounds__(kThreadsNS, 1)
    norm_cast_stream_kernel(const uint8_t* x, const uint4* __restrict__ gamma, int64_t T,
                            int nvec, int stages, int ring_rows, float inv_d, float eps,
                            uint4* __restrict__ A,
                            const NsExt ext) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 127u) & ~127u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
  const uint32_t stage_bytes = kGroupRows * row_bytes;
  const bool has_res = EXT && ext.residual != nullptr;
  const bool has_beta = EXT && ext.beta != nullptr;
  // the ring holds ring_rows rows (stage s, row r at row s * kGroupRows + r)
  uint4* gamma_s = reinterpret_cast<uint4*>(smem + static_cast<size_t>(ring_rows) * row_bytes);
  uint4* beta_s = gamma_s + nvec;  // EXT only
  NsCtrl* ctrl = reinterpret_cast<NsCtrl*>(smem + static_cast<size_t>(ring_rows) * row_bytes +
                                           (EXT ? 2 : 1) * row_bytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // this CTA's rows: a contiguous range of T / gridDim.x rows (rounded), so
  // every SM moves the same number of bytes; groups of 8 within the range,
  // the last one possibly partial
  const int64_t r_begin = static_cast<int64_t>(blockIdx.x) * T / gridDim.x;
  const int64_t r_end = static_cast<int64_t>(blockIdx.x + 1) * T / gridDim.x;
  const int64_t groups = (r_end - r_begin + kGroupRows - 1) / kGroupRows;

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
      for (int64_t g = 0; g < groups; ++g) {
        if (!mbar_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, abort, &g_err_norm, 31)) break;
        const int64_t row0 = r_begin + g * kGroupRows;
        const int rows = static_cast<int>(r_end - row0 < kGroupRows ? r_end - row0 : kGroupRows);
        const uint32_t dst = base + stage * stage_bytes;
        if (!RNL_DCHECK(&g_err_norm, stages <= kMaxNsStages && stage < static_cast<uint32_t>(stages) &&
                                         static_cast<int>(stage) * kGroupRows + rows <= ring_rows &&
                                         row0 >= 0 && row0 + rows <= T, 50))
          break;
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
    if (GAMMA || has_beta) {  // gamma (and beta) staged once in shared memory for all rows
      for (int v = threadIdx.x; v < nvec; v += kConsumerWarps * 32) {
        if (GAMMA) gamma_s[v] = __ldg(gamma + v);
        if (has_beta) beta_s[v] = __ldg(ext.beta + v);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    }
    uint32_t stage = 0, phase = 0;
    // the residual row of this warp's next row, loaded while the current one
    // is finished (plain loads: x_sum may be the residual itself; the next
    // row is never the one being written)
    uint4 rv[EXT ? VPL : 1];
    auto load_residual = [&](int64_t r) {
      const uint4* qr = ext.residual + r * nvec;
#pragma unroll
      for (int i = 0; i < (EXT ? VPL : 1); ++i) {
        const int v = lane + 32 * i;
        rv[i] = v < nvec ? qr[v] : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    if (EXT && has_res && r_begin + warp < r_end) load_residual(r_begin + warp);
    for (int64_t g = 0; g < groups; ++g) {
      const int64_t row = r_begin + g * kGroupRows + warp;
      if (row < r_end && EXT) {
        const bool got = mbar_wait(smem_u32(&ctrl->full[stage][warp]), phase, abort, &g_err_norm, 32);
        if (!__all_sync(0xFFFFFFFFu, got)) break;
        uint4* rp = reinterpret_cast<uint4*>(smem + stage * stage_bytes + warp * row_bytes);
        uint4* sr = ext.x_sum != nullptr ? ext.x_sum + row * nvec : nullptr;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int v = lane + 32 * i;
          if (v < nvec) {
            uint4 u = rp[v];
            if (has_res) {  // x_add = bf16(x + residual), one rounding of the exact sum
              float a[8], b[8];
              unpack8(u, a);
              unpack8(rv[i], b);
              u = make_uint4(pack_bf16x2(__fadd_rn(a[0], b[0]), __fadd_rn(a[1], b[1])),
                             pack_bf16x2(__fadd_rn(a[2], b[2]), __fadd_rn(a[3], b[3])),
                             pack_bf16x2(__fadd_rn(a[4], b[4]), __fadd_rn(a[5], b[5])),
                             pack_bf16x2(__fadd_rn(a[6], b[6]), __fadd_rn(a[7], b[7])));
              rp[v] = u;
            }
            if (sr != nullptr) sr[v] = u;
            float f[8];
            unpack8(u, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (MODE == 0)
                s = fmaf(f[j], f[j], s);
              else
                s = fmaf(f[j] * f[j], inv_d, s);
            }
          }
        }
        if (has_res && row + kGroupRows < r_end) load_residual(row + kGroupRows);
        s = warp_sum(s);
        const float rstd = (MODE == 0) ? rsqrtf(s * inv_d + eps) : 1.0f / sqrtf(s + eps);
        if (ext.rstd_out != nullptr && lane == 0) ext.rstd_out[row] = rstd;
        uint4* ar = A + row * nvec;
        if (!RNL_DCHECK(&g_err_norm, row < T && nvec <= 32 * VPL, 51)) break;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int v = lane + 32 * i;  // the elements this lane wrote above
          if (v >= nvec) break;
          float f[8];
          unpack8(rp[v], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = f[j] * rstd;
          if (GAMMA) {
            float gg[8];
            unpack8(gamma_s[v], gg);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = f[j] * gg[j];
          }
          if (has_beta) {
            float bb[8];
            unpack8(beta_s[v], bb);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __fadd_rn(f[j], bb[j]);
          }
          ar[v] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                             pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
        }
        // the slot was written through the generic proxy; order that before
        // the next bulk copy (async proxy) refills it
        if (has_res) fence_proxy_async_shared();
      } else if (row < r_end) {
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
        if (!RNL_DCHECK(&g_err_norm, row < T && nvec <= 32 * VPL, 52)) break;
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

template <int MODE, bool GAMMA, int VPL, bool EXT>
rnl_status launch_ns(const void* x, const void* gamma, int64_t T, int nvec, int stages, int ring_rows, float inv_d,
                     float eps, void* A, const NsExt& ext, size_t smem, const DeviceInfo& dev,
                     cudaStream_t s) {
  auto kern = norm_cast_stream_kernel<MODE, GAMMA, VPL, EXT>;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kern), dev.device, smem) != RNL_OK)
    return RNL_ERR_LAUNCH;
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
                                           static_cast<const uint4*>(gamma), T, nvec, stages, ring_rows,
                                           inv_d, eps, static_cast<uint4*>(A), ext);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return RNL_OK;
}

template <int VPL, bool EXT>
rnl_status dispatch_mode(const void* x, const void* gamma, int64_t T, int nvec, int stages, int ring_rows,
                         float inv_d, float eps, void* A, const NsExt& ext, size_t smem,
                         const DeviceInfo& dev, cudaStream_t s, int mode) {
  if (mode == RNL_NORM_RSQRT)
    return gamma ? launch_ns<0, true, VPL, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s)
                 : launch_ns<0, false, VPL, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s);
  return gamma ? launch_ns<1, true, VPL, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s)
               : launch_ns<1, false, VPL, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s);
}

template <bool EXT>
rnl_status dispatch_vpl(const void* x, const void* gamma, int64_t T, int nvec, int stages, int ring_rows,
                        float inv_d, float eps, void* A, const NsExt& ext, size_t smem,
                        const DeviceInfo& dev, cudaStream_t s, int mode) {
  const int vpl = (nvec + 31) / 32;
  if (vpl <= 2) return dispatch_mode<2, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s, mode);
  if (vpl <= 4) return dispatch_mode<4, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s, mode);
  if (vpl <= 8) return dispatch_mode<8, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s, mode);
  return dispatch_mode<16, EXT>(x, gamma, T, nvec, stages, ring_rows, inv_d, eps, A, ext, smem, dev, s, mode);
}

rnl_status launch_stream(const void* x, const void* gamma, int64_t T, int64_t K, float eps,
                         int mode, void* A, const NsExt* ext, cudaStream_t s) {
  if (T == 0) return RNL_OK;
  if (!norm_cast_stream_fits(K)) return RNL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const int nvec = static_cast<int>(K / 8);
  const size_t row_b = static_cast<size_t>(K) * 2;
  const size_t stage = static_cast<size_t>(kGroupRows) * row_b;
  int stages = static_cast<int>(kRingBytes / stage);
  if (stages > kMaxNsStages) stages = kMaxNsStages;
  int64_t ring_rows = static_cast<int64_t>(stages) * kGroupRows;
  // ring, then gamma [, beta] rows, then the barriers
  const size_t fixed = 128 + static_cast<size_t>(ext ? 2 : 1) * row_b + sizeof(NsCtrl);
  // When the fullest CTA's whole share of rows fits in shared memory, the
  // ring holds all of it, one stage a group: every row is requested at once
  // and no slot waits to be refilled.  (At 4096 rows of 4096 a CTA's 27 rows
  // then stream without the last 3 waiting for the first group to be done.)
  const int64_t grid = std::min<int64_t>((T + kGroupRows - 1) / kGroupRows, dev.sm_count);
  const int64_t rows_max = (T + grid - 1) / grid;
  const int64_t groups_max = (rows_max + kGroupRows - 1) / kGroupRows;
  if (groups_max > stages && groups_max <= kMaxNsStages &&
      fixed + static_cast<size_t>(rows_max) * row_b <= kNsSmemLimit) {
    stages = static_cast<int>(groups_max);
    ring_rows = rows_max;
  }
  const size_t smem = fixed + static_cast<size_t>(ring_rows) * row_b;
  const float inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  trace_before(s);
  if (ext)
    st = dispatch_vpl<true>(x, gamma, T, nvec, stages, static_cast<int>(ring_rows), inv_d, eps, A, *ext, smem, dev, s, mode);
  else
    st = dispatch_vpl<false>(x, gamma, T, nvec, stages, static_cast<int>(ring_rows), inv_d, eps, A, NsExt{}, smem, dev, s, mode);
  trace_after(s, ext ? "add_norm_cast" : "norm_cast");
  return st;
}

}  // namespace

// Rows of up to 4096 elements (16 vectors per lane in registers).
bool norm_cast_stream_fits(int64_t K) { return K % 8 == 0 && K <= 4096; }

rnl_status launch_norm_cast_stream(const void* x, const void* gamma, int64_t T, int64_t K,
                                   float eps, int mode, void* A, cudaStream_t s) {
  return launch_stream(x, gamma, T, K, eps, mode, A, nullptr, s);
}

rnl_status launch_add_norm_cast_stream(const void* x, const void* residual, void* x_sum_out,
                                       const void* gamma, const void* beta, int64_t T, int64_t K,
                                       float eps, int mode, void* A, float* rstd_out,
                                       cudaStream_t s) {
  NsExt ext;
  ext.residual = static_cast<const uint4*>(residual);
  ext.x_sum = static_cast<uint4*>(x_sum_out);
  ext.beta = static_cast<const uint4*>(beta);
  ext.rstd_out = rstd_out;
  return launch_stream(x, gamma, T, K, eps, mode, A, &ext, s);
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
