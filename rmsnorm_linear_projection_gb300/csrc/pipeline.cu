// pipeline.cu -- host-buffer executor: the projection calls of rnl.h fed
// from, and answering into, pinned host memory, with the host<->device copies
// of consecutive calls overlapped with the kernels.
//
// A pipeline owns two slots of device staging (an x buffer and an output
// buffer each), one workspace and three non-blocking streams:
//
//   h2d   x_host -> x_dev[slot]        (copy engine)
//   comp  the call's kernels           x_dev[slot] -> out_dev[slot]
//   d2h   out_dev[slot] -> out_host    (copy engine)
//
// Ticket i uses slot i & 1.  Events order the three streams: the kernels of
// ticket i wait for its input copy; the input copy of ticket i waits until
// the kernels of ticket i - 2 have finished reading x_dev[slot]; the kernels
// of ticket i wait until the output copy of ticket i - 2 has drained
// out_dev[slot]; the output copy of ticket i waits for its kernels.  So while
// ticket i computes, ticket i + 1's input and ticket i - 1's output are on
// the link.  One workspace suffices: every kernel runs on `comp`, in order.
// Host code only.
#include <cuda_runtime.h>

#include <cmath>
#include <new>

#include "internal.h"

struct rnl_pipeline {
  int device = -1;
  int op = 0;
  int64_t T = 0, K = 0, N = 0, N2 = 0;
  size_t x_bytes = 0, out_bytes = 0, ws_bytes = 0;
  void* x_dev[2] = {nullptr, nullptr};
  void* out_dev[2] = {nullptr, nullptr};
  void* ws = nullptr;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t ev_in[2] = {nullptr, nullptr};    // input copy of the slot's last ticket done
  cudaEvent_t ev_done[2] = {nullptr, nullptr};  // kernels of the slot's last ticket done
  cudaEvent_t ev_out[2] = {nullptr, nullptr};   // output copy of the slot's last ticket done
  int64_t next_ticket = 0;
  rnl_status failed = RNL_OK;  // a launch error leaves the pipeline unusable
};

namespace rnl {
namespace {

// Makes `dev` current for the scope of one call and restores the caller's.
struct DeviceScope {
  int prev = -1;
  bool ok = false;
  explicit DeviceScope(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceScope() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

void release(rnl_pipeline* p) {
  for (cudaStream_t s : {p->h2d, p->comp, p->d2h})
    if (s) cudaStreamSynchronize(s);
  for (int i = 0; i < 2; ++i) {
    if (p->x_dev[i]) cudaFree(p->x_dev[i]);
    if (p->out_dev[i]) cudaFree(p->out_dev[i]);
    for (cudaEvent_t e : {p->ev_in[i], p->ev_done[i], p->ev_out[i]})
      if (e) cudaEventDestroy(e);
  }
  if (p->ws) cudaFree(p->ws);
  for (cudaStream_t s : {p->h2d, p->comp, p->d2h})
    if (s) cudaStreamDestroy(s);
  cudaGetLastError();
  delete p;
}

// Page-locked host memory (cudaHostAlloc / cudaHostRegister); anything else
// would turn the asynchronous copies into staged synchronous ones.
bool pinned_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The shared part of the three submit calls; `compute` enqueues the kernels
// on the given stream from x_dev to out_dev and returns their status.
template <class F>
rnl_status submit(rnl_pipeline* p, const void* x_host, void* out_host, int64_t* ticket,
                  F&& compute) {
  if (!p || !x_host || !out_host || !ticket) return RNL_ERR_NULL;
  if (p->failed != RNL_OK) return p->failed;
  if (!pinned_host(x_host) || !pinned_host(out_host)) return RNL_ERR_ARG;
  DeviceScope scope(p->device);
  if (!scope.ok) return RNL_ERR_DEVICE;
  const int64_t t = p->next_ticket;
  const int slot = static_cast<int>(t & 1);
  bool ok = true;
  if (t >= 2) ok = ok && cudaStreamWaitEvent(p->h2d, p->ev_done[slot], 0) == cudaSuccess;
  if (p->x_bytes)
    ok = ok && cudaMemcpyAsync(p->x_dev[slot], x_host, p->x_bytes, cudaMemcpyHostToDevice,
                               p->h2d) == cudaSuccess;
  ok = ok && cudaEventRecord(p->ev_in[slot], p->h2d) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(p->comp, p->ev_in[slot], 0) == cudaSuccess;
  if (t >= 2) ok = ok && cudaStreamWaitEvent(p->comp, p->ev_out[slot], 0) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return p->failed = RNL_ERR_LAUNCH;
  }
  const rnl_status st =
      compute(p->x_dev[slot], p->out_dev[slot], reinterpret_cast<rnl_stream_t>(p->comp));
  if (st != RNL_OK) {
    // the input copy is already enqueued: later tickets could not be ordered
    return p->failed = st;
  }
  ok = cudaEventRecord(p->ev_done[slot], p->comp) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(p->d2h, p->ev_done[slot], 0) == cudaSuccess;
  if (p->out_bytes)
    ok = ok && cudaMemcpyAsync(out_host, p->out_dev[slot], p->out_bytes, cudaMemcpyDeviceToHost,
                               p->d2h) == cudaSuccess;
  ok = ok && cudaEventRecord(p->ev_out[slot], p->d2h) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return p->failed = RNL_ERR_LAUNCH;
  }
  *ticket = t;
  p->next_ticket = t + 1;
  return RNL_OK;
}

// Checks done before anything is enqueued, so that an argument error leaves
// the pipeline usable (the entry points repeat them).
rnl_status check_common(float eps, int norm_mode) {
  if (!std::isfinite(eps) || eps < 0.f) return RNL_ERR_ARG;
  if (norm_mode != RNL_NORM_RSQRT && norm_mode != RNL_NORM_SQRT_DIV) return RNL_ERR_ARG;
  return RNL_OK;
}

}  // namespace
}  // namespace rnl

using namespace rnl;

extern "C" {

rnl_status rnl_pipeline_create(int op, int64_t T, int64_t K, int64_t N, int64_t N2,
                               rnl_pipeline** pipe) {
  if (!pipe) return RNL_ERR_NULL;
  *pipe = nullptr;
  if (op != RNL_OP_BF16 && op != RNL_OP_W8A8 && op != RNL_OP_MLA) return RNL_ERR_ARG;
  if (op == RNL_OP_BF16 && N2 != RNL_OUT_BF16 && N2 != RNL_OUT_FP32) return RNL_ERR_ARG;
  const size_t ws_bytes = rnl_workspace_size(op, T, K, N, N2);
  if (ws_bytes == static_cast<size_t>(-1) || K == 0 || N == 0 || (op == RNL_OP_MLA && N2 == 0))
    return RNL_ERR_SHAPE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;

  rnl_pipeline* p = new (std::nothrow) rnl_pipeline;
  if (!p) return RNL_ERR_WORKSPACE;
  p->device = dev.device;
  p->op = op;
  p->T = T;
  p->K = K;
  p->N = N;
  p->N2 = N2;
  p->x_bytes = static_cast<size_t>(T) * K * 2;
  if (op == RNL_OP_MLA)
    p->out_bytes = static_cast<size_t>(T) * N2 * 2;
  else
    p->out_bytes = static_cast<size_t>(T) * N * (op == RNL_OP_BF16 && N2 == RNL_OUT_FP32 ? 4 : 2);
  p->ws_bytes = ws_bytes;

  bool ok = true;
  for (int i = 0; i < 2 && ok; ++i) {
    ok = (p->x_bytes == 0 || cudaMalloc(&p->x_dev[i], p->x_bytes) == cudaSuccess) &&
         (p->out_bytes == 0 || cudaMalloc(&p->out_dev[i], p->out_bytes) == cudaSuccess);
  }
  if (!ok) {
    release(p);
    return RNL_ERR_WORKSPACE;
  }
  if (ws_bytes && cudaMalloc(&p->ws, ws_bytes) != cudaSuccess) {
    release(p);
    return RNL_ERR_WORKSPACE;
  }
  ok = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) == cudaSuccess &&
       cudaStreamCreateWithFlags(&p->comp, cudaStreamNonBlocking) == cudaSuccess &&
       cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; i < 2 && ok; ++i) {
    ok = cudaEventCreateWithFlags(&p->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_out[i], cudaEventDisableTiming) == cudaSuccess;
  }
  if (!ok) {
    release(p);
    return RNL_ERR_LAUNCH;
  }
  *pipe = p;
  return RNL_OK;
}

rnl_status rnl_pipeline_submit_bf16(rnl_pipeline* p, const void* x_host, const void* gamma,
                                    const void* W, float eps, int norm_mode, void* out_host,
                                    int64_t* ticket) {
  if (p && p->op != RNL_OP_BF16) return RNL_ERR_ARG;
  if (!W) return RNL_ERR_NULL;
  rnl_status st = check_common(eps, norm_mode);
  if (st != RNL_OK) return st;
  if (p && p->N2 == RNL_OUT_FP32 && gamma) return RNL_ERR_UNSUPPORTED;
  if (!aligned16(W) || (gamma && !aligned16(gamma))) return RNL_ERR_ALIGN;
  return submit(p, x_host, out_host, ticket, [&](void* x, void* out, rnl_stream_t s) {
    return rmsnorm_linear_bf16(x, gamma, W, p->T, p->K, p->N, eps, norm_mode, out,
                               static_cast<int>(p->N2), p->ws, p->ws_bytes, s);
  });
}

rnl_status rnl_pipeline_submit_w8a8(rnl_pipeline* p, const void* x_host, const void* gamma,
                                    const int8_t* Wq, const float* w_scale, float eps,
                                    int norm_mode, void* out_host, int64_t* ticket) {
  if (p && p->op != RNL_OP_W8A8) return RNL_ERR_ARG;
  if (!Wq || !w_scale) return RNL_ERR_NULL;
  rnl_status st = check_common(eps, norm_mode);
  if (st != RNL_OK) return st;
  if ((p && p->K % 16 != 0) || !aligned16(Wq) || !aligned16(w_scale) ||
      (gamma && !aligned16(gamma)))
    return RNL_ERR_ALIGN;
  return submit(p, x_host, out_host, ticket, [&](void* x, void* out, rnl_stream_t s) {
    return rmsnorm_linear_w8a8(x, gamma, Wq, w_scale, p->T, p->K, p->N, eps, norm_mode, out,
                               nullptr, nullptr, p->ws, p->ws_bytes, s);
  });
}

rnl_status rnl_pipeline_submit_mla(rnl_pipeline* p, const void* x_host, const void* W_qa,
                                   const void* gamma_cq, const void* W_qb, float eps,
                                   int norm_mode, void* out_host, int64_t* ticket) {
  if (p && p->op != RNL_OP_MLA) return RNL_ERR_ARG;
  if (!W_qa || !gamma_cq || !W_qb) return RNL_ERR_NULL;
  rnl_status st = check_common(eps, norm_mode);
  if (st != RNL_OK) return st;
  if ((p && p->N % 8 != 0) || !aligned16(W_qa) || !aligned16(gamma_cq) || !aligned16(W_qb))
    return RNL_ERR_ALIGN;
  return submit(p, x_host, out_host, ticket, [&](void* x, void* out, rnl_stream_t s) {
    return mla_q_chain(x, W_qa, gamma_cq, W_qb, p->T, p->K, p->N, p->N2, eps, norm_mode, out,
                       nullptr, p->ws, p->ws_bytes, s);
  });
}

rnl_status rnl_pipeline_wait(rnl_pipeline* p, int64_t ticket, int* site) {
  if (!p) return RNL_ERR_NULL;
  if (ticket < 0 || ticket >= p->next_ticket) return RNL_ERR_ARG;
  DeviceScope scope(p->device);
  if (!scope.ok) return RNL_ERR_DEVICE;
  // the slot's event was last recorded for `ticket` or a later ticket of the
  // same slot, whose output copy follows ticket's on the d2h stream
  if (cudaEventSynchronize(p->ev_out[ticket & 1]) != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return read_device_errors(site);
}

rnl_status rnl_pipeline_destroy(rnl_pipeline* p) {
  if (!p) return RNL_OK;
  DeviceScope scope(p->device);
  release(p);
  return RNL_OK;
}

}  // extern "C"
