// selftest.cu -- failure-detection self-tests.  The wait test: a kernel waits on an mbarrier
// that nothing ever arrives on, through the same bounded wait every kernel of
// the library uses, with a 1 ms limit.  The wait gives up, records its site
// in this module's device error word and the kernel returns normally; the
// host then reads RNL_ERR_TIMEOUT from rnl_check_device_error() and the CUDA
// context stays usable.  No fault, trap or unbounded wait is involved.
#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

__device__ unsigned int g_err_selftest;

constexpr uint32_t kSelftestSite = 99;
constexpr uint32_t kBoundsSite = 98;

// Two words; the check below treats only the first as in range, so the
// index it refuses still lies inside this array.
__device__ int g_bounds_selftest[2];

__global__ void bounds_check_kernel(int n_valid, int index) {
  if (RNL_DCHECK(&g_err_selftest, index < n_valid, kBoundsSite)) g_bounds_selftest[index] = 1;
}

__global__ void wait_timeout_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 of `bar` never completes: nothing arrives on it
    mbar_wait_limit(smem_u32(&bar), 0u, &abort, &g_err_selftest, kSelftestSite, limit_ns);
  }
  __syncthreads();
}

}  // namespace

rnl_status read_clear_error_selftest(unsigned int* word) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_selftest, sizeof v) != cudaSuccess) return RNL_ERR_LAUNCH;
  if (v != 0 && cudaMemcpyToSymbol(g_err_selftest, &zero, sizeof zero) != cudaSuccess)
    return RNL_ERR_LAUNCH;
  *word = v;
  return RNL_OK;
}

}  // namespace rnl

extern "C" rnl_status rnl_selftest_wait_timeout(rnl_stream_t stream) {
  rnl::DeviceInfo dev;
  rnl_status st = rnl::current_device(&dev);
  if (st != RNL_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rnl::wait_timeout_kernel<<<1, 32, 0, s>>>(1000000ull);  // 1 ms
  return cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
}

extern "C" rnl_status rnl_selftest_bounds_check(rnl_stream_t stream) {
#ifdef RNL_DEBUG
  rnl::DeviceInfo dev;
  rnl_status st = rnl::current_device(&dev);
  if (st != RNL_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rnl::bounds_check_kernel<<<1, 1, 0, s>>>(1, 1);  // index 1 of a 1-word range, inside the array
  return cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
#else
  (void)stream;
  return RNL_ERR_UNSUPPORTED;
#endif
}
