// api.cu -- the C ABI declared in include/rnl.h: argument validation,
// workspace layout, kernel selection by shape, TMA descriptor encoding,
// device error words and the kernel timing trace.  Host code only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <map>
#include <utility>

#include "internal.h"
#include "ptx.cuh"

namespace rnl {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

// ------------------------------------------------------------ device info
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

// ------------------------------------------------------------ TMA encoding
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// ------------------------------------------------------------ trace ring
constexpr int kTraceCap = 16384;
struct TraceRec {
  cudaEvent_t a = nullptr, b = nullptr;
  char name[32] = {0};
};
bool g_trace_on = false;
TraceRec g_trace[kTraceCap];
int g_trace_n = 0;
bool g_trace_pending = false;

// ------------------------------------------------------------ validation
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline bool bad_eps(float eps) { return !std::isfinite(eps) || eps < 0.f; }
inline bool bad_mode(int m) { return m != RNL_NORM_RSQRT && m != RNL_NORM_SQRT_DIV; }
// sizes must stay inside int32 tile / TMA coordinate arithmetic
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
inline bool bad_dim(int64_t v) { return v < 0 || v > kMaxDim; }

struct Carve {
  char* p;
  size_t used = 0;
  explicit Carve(void* base) : p(static_cast<char*>(base)) {}
  void* take(size_t bytes) {
    void* r = p ? p + used : nullptr;
    used += round_up(bytes);
    return r;
  }
};

// Workspace layouts (a null base just measures).
struct BF16Layout {
  void* part = nullptr;   // gemm K-split partial sums (bf16 out; fp32 out with N > 64)
  void* A = nullptr;      // bf16 [T, K] normed activations (bf16 out, two-kernel form)
  float* rstd = nullptr;  // [T] (bf16 out; fp32 out with N > 64)
  void* skinny = nullptr; // skinny partials (fp32 out, N <= 64)
  size_t bytes = 0;
};
BF16Layout bf16_layout(void* ws, int64_t T, int64_t K, int64_t N, int out_dtype) {
  BF16Layout l;
  Carve c(ws);
  if (out_dtype == RNL_OUT_BF16) {
    l.rstd = static_cast<float*>(c.take(static_cast<size_t>(T) * 4));
    l.A = c.take(static_cast<size_t>(T) * K * 2);  // only the two-kernel form uses it
    l.part = c.take(kGemmPartialBytes);
  } else if (N <= 64) {
    l.skinny = c.take(skinny_workspace_bytes(T, K, N, 0));
  } else {
    l.rstd = static_cast<float*>(c.take(static_cast<size_t>(T) * 4));
    l.part = c.take(kGemmPartialBytes);
  }
  l.bytes = c.used;
  return l;
}

struct W8A8Layout {
  void* A = nullptr;        // bf16 [T, K] integer codes
  void* Wb = nullptr;       // bf16 [N, K] widened weight
  float* xs = nullptr;      // [T] x_scale when the caller passes none
  float* gmax = nullptr;    // max |gamma| (the integer GEMM's exactness bound)
  void* part = nullptr;     // gemm K-split partial sums
  void* chunk = nullptr;    // the pair GEMM's running int32 sums of chunked tiles
  size_t bytes = 0;
};
W8A8Layout w8a8_layout(void* ws, int64_t T, int64_t K, int64_t N) {
  W8A8Layout l;
  Carve c(ws);
  l.A = c.take(static_cast<size_t>(T) * K * 2);
  l.Wb = c.take(static_cast<size_t>(N) * K * 2);
  l.xs = static_cast<float*>(c.take(static_cast<size_t>(T) * 4));
  l.gmax = static_cast<float*>(c.take(4));
  l.part = c.take(kGemmPartialBytes);
  l.chunk = c.take(kGemmPartialBytes);
  l.bytes = c.used;
  return l;
}

// rmsnorm_linear_w8a8_prepared: the weight arrives widened, so no Wb
struct W8A8PLayout {
  void* A = nullptr;        // bf16 [T, K] integer codes
  float* xs = nullptr;      // [T] x_scale when the caller passes none
  float* gmax = nullptr;    // max |gamma| (the integer GEMM's exactness bound)
  void* part = nullptr;     // gemm K-split partial sums
  void* chunk = nullptr;    // the pair GEMM's running int32 sums of chunked tiles
  size_t bytes = 0;
};
W8A8PLayout w8a8p_layout(void* ws, int64_t T, int64_t K) {
  W8A8PLayout l;
  Carve c(ws);
  l.A = c.take(static_cast<size_t>(T) * K * 2);
  l.xs = static_cast<float*>(c.take(static_cast<size_t>(T) * 4));
  l.gmax = static_cast<float*>(c.take(4));
  l.part = c.take(kGemmPartialBytes);
  l.chunk = c.take(kGemmPartialBytes);
  l.bytes = c.used;
  return l;
}

struct MLALayout {
  void* qa = nullptr;     // bf16 [T, N1] stage-1 output when the caller passes none
  void* z = nullptr;      // bf16 [T, N1] normed * gamma_cq (two-kernel form)
  float* rstd = nullptr;  // [T] rstd of the stage-1 rows
  void* part = nullptr;   // gemm K-split partial sums (both stages, one after the other)
  size_t bytes = 0;
};
MLALayout mla_layout(void* ws, int64_t T, int64_t N1) {
  MLALayout l;
  Carve c(ws);
  l.qa = c.take(static_cast<size_t>(T) * N1 * 2);
  l.z = c.take(static_cast<size_t>(T) * N1 * 2);
  l.rstd = static_cast<float*>(c.take(static_cast<size_t>(T) * 4));
  l.part = c.take(kGemmPartialBytes);
  l.bytes = c.used;
  return l;
}

struct QmrsLayout {
  void* x1 = nullptr;     // bf16 [B*M, K] widened x1
  void* x2 = nullptr;     // bf16 [B*N, K] transposed, widened x2
  float* ws = nullptr;    // fp32 [N] x2_scale
  float* acc = nullptr;   // fp32 [M, N] running sum over the batch
  uint64_t* flags = nullptr;  // per (output tile, epilogue warp): batch b's sum is written
  size_t bytes = 0;
};
QmrsLayout qmrs_layout(void* ws, int64_t B, int64_t M, int64_t K, int64_t N) {
  QmrsLayout l;
  Carve c(ws);
  l.x1 = c.take(static_cast<size_t>(B) * M * K * 2);
  l.x2 = c.take(static_cast<size_t>(B) * N * K * 2);
  l.ws = static_cast<float*>(c.take(static_cast<size_t>(N) * 4));
  l.acc = static_cast<float*>(c.take(B > 1 ? static_cast<size_t>(M) * N * 4 : 0));
  l.flags = static_cast<uint64_t*>(c.take(B > 1 ? batch_flag_bytes(M, N) : 0));
  l.bytes = c.used;
  return l;
}

// The MXFP8 kernels index 16-code vectors of either operand in 32 bits.
inline bool mx_too_large(int64_t T, int64_t K, int64_t N) {
  return T * K / 16 >= (int64_t{1} << 32) || N * K / 16 >= (int64_t{1} << 32);
}

struct MxLayout {
  uint8_t* codes = nullptr;  // E4M3 [T, K] activation codes when the caller takes none
  uint8_t* sfa = nullptr;    // scale atoms of the activations (block-scaled GEMM)
  uint8_t* sfb = nullptr;    // scale atoms of the weight
  void* A = nullptr;         // bf16 [T, K] dequantised activations (emulation path)
  void* Wb = nullptr;        // bf16 [N, K] dequantised weight (emulation path)
  void* part = nullptr;
  size_t bytes = 0;
};
MxLayout mx_layout(void* ws, int64_t T, int64_t K, int64_t N) {
  MxLayout l;
  Carve c(ws);
  l.codes = static_cast<uint8_t*>(c.take(static_cast<size_t>(T) * K));
  // A's atoms cover whole 256-row tiles (the CTA-pair GEMM reads both halves)
  l.sfa = static_cast<uint8_t*>(c.take(mx_sf_atoms_bytes((T + 255) / 256 * 256, K, 128)));
  l.sfb = static_cast<uint8_t*>(c.take(mx_sf_atoms_bytes(N, K, mx_native_bn())));
  l.A = c.take(static_cast<size_t>(T) * K * 2);
  l.Wb = c.take(static_cast<size_t>(N) * K * 2);
  l.part = c.take(kGemmPartialBytes);
  l.bytes = c.used;
  return l;
}

// The GEMM of both MXFP8 entry points: bf16 operands, bf16 out or fp32 out
// (the fp32 epilogue with no row scale).
rnl_status mx_gemm(const MxLayout& l, int64_t T, int64_t K, int64_t N, void* out, int out_dtype,
                   cudaStream_t s) {
  GemmArgs g;
  g.A = l.A;
  g.B = l.Wb;
  g.M = T;
  g.N = N;
  g.K = K;
  g.out = out;
  g.epi = out_dtype == RNL_OUT_BF16 ? Epi::kBf16 : Epi::kRowScaleF32;
  g.partial_ws = l.part;
  g.partial_ws_bytes = kGemmPartialBytes;
  g.trace_name = "gemm_mxfp8";
  return launch_gemm(g, s);
}

struct S8Layout {
  void* A = nullptr;
  void* B = nullptr;
  void* part = nullptr;
  void* chunk = nullptr;  // the pair GEMM's running int32 sums of chunked tiles
  size_t bytes = 0;
};
S8Layout s8_layout(void* ws, int64_t M, int64_t K, int64_t N) {
  S8Layout l;
  Carve c(ws);
  l.A = c.take(static_cast<size_t>(M) * K * 2);
  l.B = c.take(static_cast<size_t>(N) * K * 2);
  l.part = c.take(kGemmPartialBytes);
  l.chunk = c.take(kGemmPartialBytes);
  l.bytes = c.used;
  return l;
}

inline cudaStream_t cs(rnl_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// The W8A8 front end's quantising part: the streamed form (each row read
// once into registers, quantstream.cu) for rows of up to 4096 elements, else
// the three-read row kernels (rowwise.cu).  RNL_W8A8_STREAM=0 forces the
// latter; both give the same codes and scales.  The streamed form also
// writes max |gamma| (into *gmax when gamma is given) for the integer GEMM's
// exactness bound (*exact = true); after the row kernels the GEMM takes
// every tile in chunks (*exact = false).
rnl_status w8a8_quantise(const void* x, const void* gamma, int64_t T, int64_t K, float eps, int mode,
                         void* A, int8_t* q_out, float* xs, float* gmax, bool* exact, cudaStream_t s) {
  const char* e = std::getenv("RNL_W8A8_STREAM");
  *exact = false;
  if (quant_stream_fits(K) && (e == nullptr || e[0] != '0')) {
    *exact = true;
    return launch_quant_stream(x, gamma, T, K, eps, mode, A, q_out, xs, gamma ? gmax : nullptr, s);
  }
  return launch_norm_quant(x, gamma, T, K, eps, mode, A, q_out, xs, s);
}

// The exact integer GEMM with the dequant epilogue: out = bf16(float(A Wb^T) * (xs * w_scale)).
// With the streamed quantiser's exactness bound (exact: rows of RMSNorm
// codes, gmax = max |gamma| or null) the CTA-pair kernel takes it where it is
// predicted faster (gemm_tc.cu launch_gemm).
rnl_status w8a8_gemm(const void* A, const void* Wb, int64_t T, int64_t K, int64_t N, const float* xs,
                     const float* w_scale, bool exact, const float* gmax, void* out, void* part,
                     void* chunk, cudaStream_t s) {
  GemmArgs g;
  g.A = A;
  g.B = Wb;
  g.M = T;
  g.N = N;
  g.K = K;
  g.out = out;
  g.row_scale = xs;
  g.col_scale = w_scale;
  g.exact_rows = exact;
  g.gamma_max = gmax;
  g.chunk_ws = chunk;
  g.chunk_ws_bytes = kGemmPartialBytes;
  g.epi = Epi::kDequantBf16;
  g.partial_ws = part;
  g.partial_ws_bytes = kGemmPartialBytes;
  return launch_gemm(g, s);
}

// Two forms of the normalise-and-cast step compute the same values:
//   two-kernel (default): a row pass writes the bf16 A operand [T, K], the
//     GEMM streams it by TMA;
//   fused (RNL_FUSED_NORM=1): a row pass writes only rstd [T]; four
//     transform warps in the GEMM rewrite each TMA-loaded x stage in shared
//     memory as bf16((x * rstd) * gamma) before the MMA reads it.
// The fused form redoes the transform for every N tile of a row block (32
// times for a 6144-wide output with 192-wide tiles) and measured 2.7x slower
// on GB300, so it is opt-in.
bool fused_norm() {
  const char* e = std::getenv("RNL_FUSED_NORM");
  return e != nullptr && e[0] == '1';
}

// The MXFP8 mode multiplies on the block-scaled tensor cores
// (tcgen05.mma kind::mxf8f6f4.block_scale, mxgemm.cu) straight from the E4M3
// codes; RNL_MXFP8_NATIVE=0 selects the exact emulation instead (operands
// dequantised to bf16, the bf16 GEMM).  Both give results within the same
// FP32-accumulation bound.
bool mx_native() {
  const char* e = std::getenv("RNL_MXFP8_NATIVE");
  return e == nullptr || e[0] != '0';
}

// Up to 4 tokens against a weight of at least 1024 rows (a decode step) run
// as a matrix-vector product that spreads the weight over every SM, on the
// CUDA cores (decode.cu), or with RNL_DECODE_MMA=1 on the tensor cores with
// the weight streamed by TMA and the K ranges split over several CTAs
// (decode_mma.cu: as fast at a 50 MB weight, slower at 12.6 and 101 MB);
// RNL_DECODE=0 sends them to the GEMM path.
bool decode_path() {
  const char* e = std::getenv("RNL_DECODE");
  return e == nullptr || e[0] != '0';
}
bool decode_mma() {
  const char* e = std::getenv("RNL_DECODE_MMA");
  return e != nullptr && e[0] == '1';
}

// The QKV split + per-head norm + RoPE runs in the CTA-pair GEMM's epilogue
// when head_dim is 128 and the projection runs on CTA pairs; otherwise (and
// with RNL_QKV_ROPE_EPILOGUE=0) the projection writes y and the separate
// stage (qkvrope.cu) reads it.  Both give results within the same bounds.
bool qkv_rope_in_epilogue() {
  const char* e = std::getenv("RNL_QKV_ROPE_EPILOGUE");
  return e == nullptr || e[0] != '0';
}

}  // namespace

// ------------------------------------------------------------ shared helpers
rnl_status current_device(DeviceInfo* info) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return RNL_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.device < 0) {
    DeviceInfo n;
    n.device = dev;
    if (cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return RNL_ERR_DEVICE;
    }
    if (n.major != 10 || n.minor != 3) return RNL_ERR_DEVICE;  // built for sm_103a only
    d = n;
  }
  *info = d;
  return RNL_OK;
}

namespace {
rnl_status encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                     uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                     CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return RNL_ERR_DEVICE;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? RNL_OK : RNL_ERR_ARG;
}
}  // namespace

rnl_status make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                       uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                       uint32_t box_outer) {
  return encode_2d(map, dtype, base, inner, outer, row_bytes, box_inner, box_outer,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

rnl_status make_map_2d_plain(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                             uint64_t inner, uint64_t outer, uint64_t row_bytes,
                             uint32_t box_inner, uint32_t box_outer) {
  return encode_2d(map, dtype, base, inner, outer, row_bytes, box_inner, box_outer,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
}

namespace {
std::mutex g_attr_mu;
std::map<std::pair<const void*, int>, size_t> g_attr_done;  // the dynamic shared memory each kernel may use
}  // namespace

rnl_status ensure_smem_attr(const void* kernel, int device, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_attr_mu);
  const auto key = std::make_pair(kernel, device);
  const auto it = g_attr_done.find(key);
  if (it != g_attr_done.end() && it->second >= bytes) return RNL_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  g_attr_done[key] = bytes;
  return RNL_OK;
}

void trace_before(cudaStream_t s) {
  if (!g_trace_on || g_trace_n >= kTraceCap) return;
  TraceRec& t = g_trace[g_trace_n];
  if (t.a == nullptr) {
    cudaEventCreate(&t.a);
    cudaEventCreate(&t.b);
  }
  cudaEventRecord(t.a, s);
  g_trace_pending = true;
}

void trace_after(cudaStream_t s, const char* name) {
  if (!g_trace_on || !g_trace_pending || g_trace_n >= kTraceCap) return;
  TraceRec& t = g_trace[g_trace_n];
  cudaEventRecord(t.b, s);
  std::snprintf(t.name, sizeof t.name, "%s", name);
  ++g_trace_n;
  g_trace_pending = false;
}

rnl_status read_device_errors(int* site) {
  unsigned int words[10] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
  if (read_clear_error_rowwise(&words[0]) != RNL_OK || read_clear_error_gemm(&words[1]) != RNL_OK ||
      read_clear_error_skinny(&words[2]) != RNL_OK || read_clear_error_pair(&words[3]) != RNL_OK ||
      read_clear_error_norm(&words[4]) != RNL_OK || read_clear_error_selftest(&words[5]) != RNL_OK ||
      read_clear_error_rope(&words[6]) != RNL_OK || read_clear_error_mx(&words[7]) != RNL_OK ||
      read_clear_error_quant(&words[8]) != RNL_OK || read_clear_error_decmma(&words[9]) != RNL_OK)
    return RNL_ERR_LAUNCH;
  for (unsigned int w : words) {
    if (w != 0) {
      if (site) *site = static_cast<int>((w >> 8) & 0xFFu);
      // a failed bounds check (debug builds) comes first: a wait that then
      // timed out is its consequence
      if (w & kErrBounds) return RNL_ERR_BOUNDS;
      return (w & kErrTimeout) ? RNL_ERR_TIMEOUT : RNL_ERR_ARG;
    }
  }
  if (site) *site = 0;
  return RNL_OK;
}

}  // namespace rnl

using namespace rnl;

extern "C" {

int rnl_version(void) { return 100; }

int rnl_debug_build(void) {
#ifdef RNL_DEBUG
  return 1;
#else
  return 0;
#endif
}

const char* rnl_status_string(rnl_status s) {
  switch (s) {
    case RNL_OK: return "ok";
    case RNL_ERR_NULL: return "null pointer";
    case RNL_ERR_SHAPE: return "bad shape";
    case RNL_ERR_ALIGN: return "misaligned pointer or K";
    case RNL_ERR_ARG: return "bad argument";
    case RNL_ERR_WORKSPACE: return "workspace too small";
    case RNL_ERR_LAUNCH: return "CUDA launch error";
    case RNL_ERR_TIMEOUT: return "device wait timed out";
    case RNL_ERR_UNSUPPORTED: return "unsupported argument combination";
    case RNL_ERR_DEVICE: return "no sm_103 device or driver entry point";
    case RNL_ERR_BOUNDS: return "device bounds check failed (debug build)";
  }
  return "unknown status";
}

size_t rnl_workspace_size(int op, int64_t T, int64_t K, int64_t N, int64_t N2) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || bad_dim(N2)) return static_cast<size_t>(-1);
  switch (op) {
    case RNL_OP_BF16:
      if (N2 != RNL_OUT_BF16 && N2 != RNL_OUT_FP32) return static_cast<size_t>(-1);
      return bf16_layout(nullptr, T, K, N, static_cast<int>(N2)).bytes;
    case RNL_OP_W8A8: return w8a8_layout(nullptr, T, K, N).bytes;
    case RNL_OP_W8A8_PREPARED: return w8a8p_layout(nullptr, T, K).bytes;
    case RNL_OP_MLA: return mla_layout(nullptr, T, N).bytes;
    case RNL_OP_GEMM_S8: return s8_layout(nullptr, T, K, N).bytes;
    case RNL_OP_QMRS:
      if (N2 <= 0) return static_cast<size_t>(-1);
      return qmrs_layout(nullptr, N2, T, K, N).bytes;
    case RNL_OP_MXFP8: return mx_layout(nullptr, T, K, N).bytes;
    case RNL_OP_QKV_ROPE:
      return bf16_layout(nullptr, T, K, N, RNL_OUT_BF16).bytes + round_up(static_cast<size_t>(T) * N * 2);
  }
  return static_cast<size_t>(-1);
}

rnl_status rmsnorm_linear_bf16(const void* x, const void* gamma, const void* W, int64_t T,
                               int64_t K, int64_t N, float eps, int norm_mode, void* out,
                               int out_dtype, void* workspace, size_t workspace_bytes,
                               rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (bad_mode(norm_mode) || bad_eps(eps) ||
      (out_dtype != RNL_OUT_BF16 && out_dtype != RNL_OUT_FP32))
    return RNL_ERR_ARG;
  if (out_dtype == RNL_OUT_FP32 && gamma != nullptr) return RNL_ERR_UNSUPPORTED;
  if (T == 0) return RNL_OK;
  if (!x || !W || !out) return RNL_ERR_NULL;
  if (K % 8 != 0 || !aligned16(x) || !aligned16(W) || !aligned16(out) ||
      (gamma && !aligned16(gamma)) || (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const BF16Layout need = bf16_layout(nullptr, T, K, N, out_dtype);
  if (need.bytes > 0 && (!workspace || workspace_bytes < need.bytes)) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const BF16Layout l = bf16_layout(workspace, T, K, N, out_dtype);
  cudaStream_t s = cs(stream);

  if (out_dtype == RNL_OUT_BF16 && decode_path() && !fused_norm() && decode_fits(T, K, N)) {
    if (decode_mma() && decode_mma_fits(T, K, N, dev.sm_count) &&
        decode_mma_workspace_bytes(N) <= kGemmPartialBytes)
      return launch_decode_mma(x, gamma, W, T, K, N, eps, norm_mode, out, l.part, kGemmPartialBytes, s);
    return launch_decode(x, gamma, W, T, K, N, eps, norm_mode, out, dev.sm_count, s);
  }
  if (out_dtype == RNL_OUT_BF16) {
    GemmArgs g;
    g.B = W;
    g.M = T;
    g.N = N;
    g.K = K;
    g.out = out;
    g.epi = Epi::kBf16;
    g.partial_ws = l.part;
    g.partial_ws_bytes = kGemmPartialBytes;
    if (fused_norm()) {
      st = launch_row_rstd(x, T, K, eps, norm_mode, l.rstd, s);
      if (st != RNL_OK) return st;
      g.A = x;
      g.a_rstd = l.rstd;
      g.a_gamma = gamma;
    } else {
      st = norm_cast_stream_fits(K) ? launch_norm_cast_stream(x, gamma, T, K, eps, norm_mode, l.A, s)
                                    : launch_norm_cast(x, gamma, T, K, eps, norm_mode, l.A, nullptr, s);
      if (st != RNL_OK) return st;
      g.A = l.A;
    }
    return launch_gemm(g, s);
  }
  if (N <= 64)
    return launch_skinny(x, W, T, K, N, eps, norm_mode, static_cast<float*>(out), l.skinny,
                         skinny_workspace_bytes(T, K, N, dev.sm_count), dev.sm_count, s);
  st = launch_row_rstd(x, T, K, eps, norm_mode, l.rstd, s);
  if (st != RNL_OK) return st;
  GemmArgs g;
  g.A = x;
  g.B = W;
  g.M = T;
  g.N = N;
  g.K = K;
  g.out = out;
  g.row_scale = l.rstd;
  g.epi = Epi::kRowScaleF32;
  g.partial_ws = l.part;
  g.partial_ws_bytes = kGemmPartialBytes;
  return launch_gemm(g, s);
}

rnl_status rmsnorm_linear_bf16_ex(const void* x, const void* residual, void* x_sum_out,
                                  const void* gamma, const void* beta, const void* W,
                                  const void* bias, int64_t T, int64_t K, int64_t N, float eps,
                                  int norm_mode, void* out, float* rstd_out, void* workspace,
                                  size_t workspace_bytes, rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (bad_mode(norm_mode) || bad_eps(eps)) return RNL_ERR_ARG;
  if (x_sum_out && !residual) return RNL_ERR_ARG;  // nothing to write back
  if (x_sum_out && x_sum_out != x && x_sum_out != residual) {
    // x_sum_out is either one of the inputs (in place) or disjoint from both
    const uintptr_t o = reinterpret_cast<uintptr_t>(x_sum_out);
    const uintptr_t n = static_cast<uintptr_t>(T) * static_cast<uintptr_t>(K) * 2;
    for (const void* in : {x, residual}) {
      const uintptr_t i = reinterpret_cast<uintptr_t>(in);
      if (in && o < i + n && i < o + n) return RNL_ERR_ARG;
    }
  }
  if (T == 0) return RNL_OK;
  if (!x || !W || !out) return RNL_ERR_NULL;
  if (K % 8 != 0 || !aligned16(x) || !aligned16(W) || !aligned16(out) ||
      (residual && !aligned16(residual)) || (x_sum_out && !aligned16(x_sum_out)) ||
      (gamma && !aligned16(gamma)) || (beta && !aligned16(beta)) || (bias && !aligned16(bias)) ||
      (rstd_out && (reinterpret_cast<uintptr_t>(rstd_out) & 3u)) ||
      (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const BF16Layout need = bf16_layout(nullptr, T, K, N, RNL_OUT_BF16);
  if (need.bytes > 0 && (!workspace || workspace_bytes < need.bytes)) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const BF16Layout l = bf16_layout(workspace, T, K, N, RNL_OUT_BF16);
  cudaStream_t s = cs(stream);
  // with no residual, beta or rstd output this is the plain AT-10 V stage
  if (!residual && !beta && !rstd_out && norm_cast_stream_fits(K))
    st = launch_norm_cast_stream(x, gamma, T, K, eps, norm_mode, l.A, s);
  else if (norm_cast_stream_fits(K))
    st = launch_add_norm_cast_stream(x, residual, x_sum_out, gamma, beta, T, K, eps, norm_mode,
                                     l.A, rstd_out, s);
  else
    st = launch_add_norm_cast(x, residual, x_sum_out, gamma, beta, T, K, eps, norm_mode, l.A,
                              rstd_out, s);
  if (st != RNL_OK) return st;
  GemmArgs g;
  g.A = l.A;
  g.B = W;
  g.M = T;
  g.N = N;
  g.K = K;
  g.out = out;
  g.epi = Epi::kBf16;
  g.bias = bias;
  g.partial_ws = l.part;
  g.partial_ws_bytes = kGemmPartialBytes;
  return launch_gemm(g, s);
}

rnl_status rnl_qkv_rope(const void* y, int64_t T, int64_t n_q_heads, int64_t n_kv_heads,
                        int64_t head_dim, const void* q_gamma, const void* k_gamma, float eps,
                        const int32_t* positions, const float* cos_sin, int64_t max_pos,
                        void* q_out, void* k_out, void* v_out, rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(n_q_heads) || bad_dim(n_kv_heads) || bad_dim(max_pos) ||
      n_q_heads + 2 * n_kv_heads == 0 || max_pos == 0 || bad_dim(T * (n_q_heads + 2 * n_kv_heads)))
    return RNL_ERR_SHAPE;
  if (!qkv_rope_head_dim_ok(head_dim)) return RNL_ERR_UNSUPPORTED;
  if (bad_eps(eps)) return RNL_ERR_ARG;
  if (T == 0) return RNL_OK;
  if (!y || !positions || !cos_sin || (n_q_heads && (!q_gamma || !q_out)) ||
      (n_kv_heads && (!k_gamma || !k_out || !v_out)))
    return RNL_ERR_NULL;
  if (!aligned16(y) || !aligned16(cos_sin) || (q_gamma && !aligned16(q_gamma)) ||
      (k_gamma && !aligned16(k_gamma)) || (q_out && !aligned16(q_out)) ||
      (k_out && !aligned16(k_out)) || (v_out && !aligned16(v_out)) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return RNL_ERR_ALIGN;
  DeviceInfo dev;
  const rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  return launch_qkv_rope(y, T, n_q_heads, n_kv_heads, head_dim, q_gamma, k_gamma, eps, positions,
                         cos_sin, max_pos, q_out, k_out, v_out, cs(stream));
}

rnl_status rmsnorm_linear_qkv_rope(const void* x, const void* gamma, const void* W, int64_t T,
                                   int64_t K, int64_t n_q_heads, int64_t n_kv_heads,
                                   int64_t head_dim, float eps, int norm_mode,
                                   const void* q_gamma, const void* k_gamma, float head_eps,
                                   const int32_t* positions, const float* cos_sin,
                                   int64_t max_pos, void* q_out, void* k_out, void* v_out,
                                   void* workspace, size_t workspace_bytes, rnl_stream_t stream) {
  if (bad_dim(n_q_heads) || bad_dim(n_kv_heads) || bad_dim(head_dim)) return RNL_ERR_SHAPE;
  const int64_t N = (n_q_heads + 2 * n_kv_heads) * head_dim;
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || K == 0 || N == 0 || bad_dim(max_pos) || max_pos == 0)
    return RNL_ERR_SHAPE;
  if (!qkv_rope_head_dim_ok(head_dim)) return RNL_ERR_UNSUPPORTED;
  if (bad_mode(norm_mode) || bad_eps(eps) || bad_eps(head_eps)) return RNL_ERR_ARG;
  const size_t need = rnl_workspace_size(RNL_OP_QKV_ROPE, T, K, N, 0);
  if (T == 0) return RNL_OK;
  if (!workspace || workspace_bytes < need) return RNL_ERR_WORKSPACE;
  if (!aligned16(workspace)) return RNL_ERR_ALIGN;
  const size_t proj = bf16_layout(nullptr, T, K, N, RNL_OUT_BF16).bytes;
  void* y = static_cast<char*>(workspace) + proj;
  // check the V-stage arguments before anything is enqueued
  if (!positions || !cos_sin || (n_q_heads && (!q_gamma || !q_out)) ||
      (n_kv_heads && (!k_gamma || !k_out || !v_out)))
    return RNL_ERR_NULL;
  if (!aligned16(cos_sin) || (q_gamma && !aligned16(q_gamma)) || (k_gamma && !aligned16(k_gamma)) ||
      (q_out && !aligned16(q_out)) || (k_out && !aligned16(k_out)) || (v_out && !aligned16(v_out)) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return RNL_ERR_ALIGN;
  if (head_dim == 128 && !fused_norm() && qkv_rope_in_epilogue() && gemm_uses_pair(T, N, K)) {
    // the stage in the CTA-pair GEMM's epilogue: y is never written
    if (!x || !W) return RNL_ERR_NULL;
    if (K % 8 != 0 || !aligned16(x) || !aligned16(W) || (gamma && !aligned16(gamma)))
      return RNL_ERR_ALIGN;
    DeviceInfo dev;
    rnl_status st = current_device(&dev);
    if (st != RNL_OK) return st;
    const BF16Layout l = bf16_layout(workspace, T, K, N, RNL_OUT_BF16);
    cudaStream_t s = cs(stream);
    st = norm_cast_stream_fits(K) ? launch_norm_cast_stream(x, gamma, T, K, eps, norm_mode, l.A, s)
                                  : launch_norm_cast(x, gamma, T, K, eps, norm_mode, l.A, nullptr, s);
    if (st != RNL_OK) return st;
    GemmArgs g;
    g.A = l.A;
    g.B = W;
    g.M = T;
    g.N = N;
    g.K = K;
    g.epi = Epi::kBf16QkvRope;
    g.partial_ws = l.part;
    g.partial_ws_bytes = kGemmPartialBytes;
    g.rope.Hq = static_cast<int>(n_q_heads);
    g.rope.Hkv = static_cast<int>(n_kv_heads);
    g.rope.q_gamma = q_gamma;
    g.rope.k_gamma = k_gamma;
    g.rope.eps = head_eps;
    g.rope.pos = positions;
    g.rope.cos_sin = cos_sin;
    g.rope.P = static_cast<int>(max_pos);
    g.rope.q = q_out;
    g.rope.k = k_out;
    g.rope.v = v_out;
    return launch_gemm(g, s);
  }
  rnl_status st = rmsnorm_linear_bf16(x, gamma, W, T, K, N, eps, norm_mode, y, RNL_OUT_BF16,
                                      workspace, proj, stream);
  if (st != RNL_OK) return st;
  return rnl_qkv_rope(y, T, n_q_heads, n_kv_heads, head_dim, q_gamma, k_gamma, head_eps,
                      positions, cos_sin, max_pos, q_out, k_out, v_out, stream);
}

rnl_status quant_matmul_reduce_sum(const int8_t* x1, const int8_t* x2, const float* x1_scale,
                                   const void* x2_scale, int64_t B, int64_t M, int64_t K,
                                   int64_t N, void* out, void* workspace, size_t workspace_bytes,
                                   rnl_stream_t stream) {
  if (bad_dim(B) || bad_dim(M) || bad_dim(K) || bad_dim(N) || B == 0 || B > 65535 || K == 0 ||
      N == 0 || bad_dim(B * M) || bad_dim(B * N))
    return RNL_ERR_SHAPE;
  if (M == 0) return RNL_OK;
  if (!x1 || !x2 || !x1_scale || !x2_scale || !out) return RNL_ERR_NULL;
  if (K % 16 != 0 || N % 16 != 0 || !aligned16(x1) || !aligned16(x2) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(x1_scale) & 3u) || (reinterpret_cast<uintptr_t>(x2_scale) & 1u) ||
      (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const QmrsLayout need = qmrs_layout(nullptr, B, M, K, N);
  if (!workspace || workspace_bytes < need.bytes) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const QmrsLayout l = qmrs_layout(workspace, B, M, K, N);
  cudaStream_t s = cs(stream);
  st = launch_qmrs_prep(x1, x2, x2_scale, B, M, K, N, l.x1, l.x2, l.ws, s);
  if (st != RNL_OK) return st;
  // all batches in one launch: items (b, tile), each adding its FP32 values to
  // the running sum of batches 0 .. b-1 of the same tile (gemm_tc.cu)
  GemmArgs g;
  g.A = l.x1;
  g.B = l.x2;
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = l.acc;
  g.out_final = out;
  g.row_scale = x1_scale;
  g.col_scale = l.ws;
  g.epi = Epi::kDequantBatchSum;
  g.nbatch = static_cast<int>(B);
  g.batch_flags = l.flags;
  return launch_gemm(g, s);
}

rnl_status rmsnorm_linear_w8a8(const void* x, const void* gamma, const int8_t* Wq,
                               const float* w_scale, int64_t T, int64_t K, int64_t N, float eps,
                               int norm_mode, void* out, int8_t* q_out, float* x_scale_out,
                               void* workspace, size_t workspace_bytes, rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (bad_mode(norm_mode) || bad_eps(eps)) return RNL_ERR_ARG;
  if (T == 0) return RNL_OK;
  if (!x || !Wq || !w_scale || !out) return RNL_ERR_NULL;
  if (K % 16 != 0 || !aligned16(x) || !aligned16(Wq) || !aligned16(out) ||
      (gamma && !aligned16(gamma)) || (q_out && !aligned16(q_out)) ||
      (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const W8A8Layout need = w8a8_layout(nullptr, T, K, N);
  if (!workspace || workspace_bytes < need.bytes) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const W8A8Layout l = w8a8_layout(workspace, T, K, N);
  cudaStream_t s = cs(stream);
  float* xs = x_scale_out ? x_scale_out : l.xs;
  bool exact = false;
  if (quant_stream_fits(K)) {
    // the weight widened by its own launch, then the streamed quantiser
    st = launch_s8_to_bf16(Wq, N * K, l.Wb, s);
    if (st == RNL_OK) st = w8a8_quantise(x, gamma, T, K, eps, norm_mode, l.A, q_out, xs, l.gmax, &exact, s);
  } else {
    st = launch_w8a8_front(x, gamma, T, K, eps, norm_mode, l.A, q_out, xs, Wq, N, l.Wb, s);
  }
  if (st != RNL_OK) return st;
  return w8a8_gemm(l.A, l.Wb, T, K, N, xs, w_scale, exact, gamma ? l.gmax : nullptr, out, l.part, l.chunk, s);
}

rnl_status rnl_w8a8_prepare_weight(const int8_t* Wq, int64_t N, int64_t K, void* Wb,
                                   rnl_stream_t stream) {
  if (bad_dim(K) || bad_dim(N) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (!Wq || !Wb) return RNL_ERR_NULL;
  if (K % 16 != 0 || !aligned16(Wq) || !aligned16(Wb)) return RNL_ERR_ALIGN;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  return launch_s8_to_bf16(Wq, N * K, Wb, cs(stream));
}

rnl_status rmsnorm_linear_w8a8_prepared(const void* x, const void* gamma, const void* Wb,
                                        const float* w_scale, int64_t T, int64_t K, int64_t N,
                                        float eps, int norm_mode, void* out, int8_t* q_out,
                                        float* x_scale_out, void* workspace, size_t workspace_bytes,
                                        rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (bad_mode(norm_mode) || bad_eps(eps)) return RNL_ERR_ARG;
  if (T == 0) return RNL_OK;
  if (!x || !Wb || !w_scale || !out) return RNL_ERR_NULL;
  if (K % 16 != 0 || !aligned16(x) || !aligned16(Wb) || !aligned16(out) ||
      (gamma && !aligned16(gamma)) || (q_out && !aligned16(q_out)) ||
      (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const W8A8PLayout need = w8a8p_layout(nullptr, T, K);
  if (!workspace || workspace_bytes < need.bytes) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const W8A8PLayout l = w8a8p_layout(workspace, T, K);
  cudaStream_t s = cs(stream);
  float* xs = x_scale_out ? x_scale_out : l.xs;
  bool exact = false;
  st = w8a8_quantise(x, gamma, T, K, eps, norm_mode, l.A, q_out, xs, l.gmax, &exact, s);
  if (st != RNL_OK) return st;
  return w8a8_gemm(l.A, Wb, T, K, N, xs, w_scale, exact, gamma ? l.gmax : nullptr, out, l.part, l.chunk, s);
}

rnl_status rmsnorm_linear_mxfp8(const void* x, const void* gamma, const uint8_t* w_codes,
                                const uint8_t* w_scale, int64_t T, int64_t K, int64_t N, float eps,
                                int norm_mode, int64_t block, void* out, int out_dtype,
                                uint8_t* x_codes_out, uint8_t* x_scale_out, void* workspace,
                                size_t workspace_bytes, rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (bad_mode(norm_mode) || bad_eps(eps) || !mx_block_ok(block) ||
      (out_dtype != RNL_OUT_BF16 && out_dtype != RNL_OUT_FP32))
    return RNL_ERR_ARG;
  if (K % block != 0 || mx_too_large(T, K, N)) return RNL_ERR_SHAPE;
  if (T == 0) return RNL_OK;
  if (!x || !w_codes || !w_scale || !out) return RNL_ERR_NULL;
  if (!aligned16(x) || !aligned16(w_codes) || !aligned16(out) || (gamma && !aligned16(gamma)) ||
      (x_codes_out && !aligned16(x_codes_out)) || (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const MxLayout need = mx_layout(nullptr, T, K, N);
  if (!workspace || workspace_bytes < need.bytes) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const MxLayout l = mx_layout(workspace, T, K, N);
  cudaStream_t s = cs(stream);
  if (mx_native()) {
    uint8_t* codes = x_codes_out != nullptr ? x_codes_out : l.codes;
    st = launch_mx_front(x, gamma, T, K, eps, norm_mode, block, nullptr, codes, x_scale_out, w_codes,
                         w_scale, N, nullptr, l.sfa, l.sfb, mx_native_bn(), s);
    if (st != RNL_OK) return st;
    return launch_mx_gemm_native(codes, w_codes, l.sfa, l.sfb, T, N, K, out, out_dtype, s);
  }
  st = launch_mx_front(x, gamma, T, K, eps, norm_mode, block, l.A, x_codes_out, x_scale_out,
                       w_codes, w_scale, N, l.Wb, nullptr, nullptr, 0, s);
  if (st != RNL_OK) return st;
  return mx_gemm(l, T, K, N, out, out_dtype, s);
}

rnl_status mxfp8_scaled_mm(const uint8_t* x_codes, const uint8_t* x_scale, const uint8_t* w_codes,
                           const uint8_t* w_scale, int64_t T, int64_t K, int64_t N, int64_t block,
                           void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                           rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (!mx_block_ok(block) || (out_dtype != RNL_OUT_BF16 && out_dtype != RNL_OUT_FP32))
    return RNL_ERR_ARG;
  if (K % block != 0 || mx_too_large(T, K, N)) return RNL_ERR_SHAPE;
  if (T == 0) return RNL_OK;
  if (!x_codes || !x_scale || !w_codes || !w_scale || !out) return RNL_ERR_NULL;
  if (!aligned16(x_codes) || !aligned16(w_codes) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const MxLayout need = mx_layout(nullptr, T, K, N);
  if (!workspace || workspace_bytes < need.bytes) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const MxLayout l = mx_layout(workspace, T, K, N);
  cudaStream_t s = cs(stream);
  if (mx_native()) {
    st = launch_mx_sf_prep(x_scale, T, w_scale, N, K, block, l.sfa, l.sfb, mx_native_bn(), s);
    if (st != RNL_OK) return st;
    return launch_mx_gemm_native(x_codes, w_codes, l.sfa, l.sfb, T, N, K, out, out_dtype, s);
  }
  st = launch_mx_dequant2(x_codes, x_scale, T, w_codes, w_scale, N, K, block, l.A, l.Wb, s);
  if (st != RNL_OK) return st;
  return mx_gemm(l, T, K, N, out, out_dtype, s);
}

rnl_status mla_q_chain(const void* x, const void* W_qa, const void* gamma_cq, const void* W_qb,
                       int64_t T, int64_t K, int64_t N1, int64_t N2, float eps, int norm_mode,
                       void* out, void* qa_out, void* workspace, size_t workspace_bytes,
                       rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(K) || bad_dim(N1) || bad_dim(N2) || K == 0 || N1 == 0 || N2 == 0)
    return RNL_ERR_SHAPE;
  if (bad_mode(norm_mode) || bad_eps(eps)) return RNL_ERR_ARG;
  if (T == 0) return RNL_OK;
  if (!x || !W_qa || !gamma_cq || !W_qb || !out) return RNL_ERR_NULL;
  if (K % 8 != 0 || N1 % 8 != 0 || !aligned16(x) || !aligned16(W_qa) || !aligned16(gamma_cq) ||
      !aligned16(W_qb) || !aligned16(out) || (qa_out && !aligned16(qa_out)) ||
      (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const MLALayout need = mla_layout(nullptr, T, N1);
  if (!workspace || workspace_bytes < need.bytes) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const MLALayout l = mla_layout(workspace, T, N1);
  cudaStream_t s = cs(stream);
  void* qa = qa_out ? qa_out : l.qa;
  GemmArgs g1;
  g1.A = x;
  g1.B = W_qa;
  g1.M = T;
  g1.N = N1;
  g1.K = K;
  g1.out = qa;
  g1.epi = Epi::kBf16;
  g1.partial_ws = l.part;
  g1.partial_ws_bytes = kGemmPartialBytes;
  g1.trace_name = "gemm_mla_stage1";
  st = launch_gemm(g1, s);
  if (st != RNL_OK) return st;
  GemmArgs g2;
  if (fused_norm()) {
    st = launch_row_rstd(qa, T, N1, eps, norm_mode, l.rstd, s);
    if (st != RNL_OK) return st;
    g2.A = qa;
    g2.a_rstd = l.rstd;
    g2.a_gamma = gamma_cq;
  } else {
    st = norm_cast_stream_fits(N1)
             ? launch_norm_cast_stream(qa, gamma_cq, T, N1, eps, norm_mode, l.z, s)
             : launch_norm_cast(qa, gamma_cq, T, N1, eps, norm_mode, l.z, nullptr, s);
    if (st != RNL_OK) return st;
    g2.A = l.z;
  }
  g2.B = W_qb;
  g2.M = T;
  g2.N = N2;
  g2.K = N1;
  g2.out = out;
  g2.epi = Epi::kBf16;
  g2.partial_ws = l.part;
  g2.partial_ws_bytes = kGemmPartialBytes;
  g2.trace_name = "gemm_mla_stage2";
  return launch_gemm(g2, s);
}

rnl_status rnl_head_rmsnorm(const void* y, int64_t T, int64_t n_heads, int64_t head_dim,
                            const void* gamma, float eps, int norm_mode, void* out,
                            rnl_stream_t stream) {
  if (bad_dim(T) || bad_dim(n_heads) || bad_dim(head_dim) || n_heads == 0 ||
      bad_dim(T * n_heads) || bad_dim(n_heads * head_dim))
    return RNL_ERR_SHAPE;
  if (!head_norm_dim_ok(head_dim)) return RNL_ERR_UNSUPPORTED;
  if (bad_mode(norm_mode) || bad_eps(eps)) return RNL_ERR_ARG;
  if (T == 0) return RNL_OK;
  if (!y || !out) return RNL_ERR_NULL;
  if (!aligned16(y) || !aligned16(out) || (gamma && !aligned16(gamma))) return RNL_ERR_ALIGN;
  const uintptr_t bytes = static_cast<uintptr_t>(T) * n_heads * head_dim * 2;
  const uintptr_t yb = reinterpret_cast<uintptr_t>(y), ob = reinterpret_cast<uintptr_t>(out);
  if (yb != ob && yb < ob + bytes && ob < yb + bytes) return RNL_ERR_ARG;  // partial overlap
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  return launch_head_norm(y, T, n_heads, head_dim, gamma, eps, norm_mode, out, cs(stream));
}

rnl_status mla_q_chain_head_norm(const void* x, const void* W_qa, const void* gamma_cq,
                                 const void* W_qb, int64_t T, int64_t K, int64_t N1, int64_t N2,
                                 float eps, int norm_mode, int64_t head_dim, const void* head_gamma,
                                 float head_eps, void* out, void* qa_out, void* workspace,
                                 size_t workspace_bytes, rnl_stream_t stream) {
  if (bad_dim(head_dim) || head_dim == 0 || N2 % head_dim != 0) return RNL_ERR_SHAPE;
  if (!head_norm_dim_ok(head_dim)) return RNL_ERR_UNSUPPORTED;
  if (bad_eps(head_eps)) return RNL_ERR_ARG;
  if (head_gamma && !aligned16(head_gamma)) return RNL_ERR_ALIGN;
  rnl_status st = mla_q_chain(x, W_qa, gamma_cq, W_qb, T, K, N1, N2, eps, norm_mode, out, qa_out,
                              workspace, workspace_bytes, stream);
  if (st != RNL_OK || T == 0) return st;
  return rnl_head_rmsnorm(out, T, N2 / head_dim, head_dim, head_gamma, head_eps, norm_mode, out,
                          stream);
}

rnl_status rnl_gemm_s8s8s32(const int8_t* A, const int8_t* B, int32_t* C, int64_t M, int64_t N,
                            int64_t K, void* workspace, size_t workspace_bytes,
                            rnl_stream_t stream) {
  if (bad_dim(M) || bad_dim(N) || bad_dim(K) || K == 0 || N == 0) return RNL_ERR_SHAPE;
  if (M == 0) return RNL_OK;
  if (!A || !B || !C) return RNL_ERR_NULL;
  if (K % 16 != 0 || !aligned16(A) || !aligned16(B) || !aligned16(C) ||
      (workspace && !aligned16(workspace)))
    return RNL_ERR_ALIGN;
  const S8Layout need = s8_layout(nullptr, M, K, N);
  if (!workspace || workspace_bytes < need.bytes) return RNL_ERR_WORKSPACE;
  DeviceInfo dev;
  rnl_status st = current_device(&dev);
  if (st != RNL_OK) return st;
  const S8Layout l = s8_layout(workspace, M, K, N);
  cudaStream_t s = cs(stream);
  st = launch_s8_to_bf16(A, M * K, l.A, s);
  if (st != RNL_OK) return st;
  st = launch_s8_to_bf16(B, N * K, l.B, s);
  if (st != RNL_OK) return st;
  GemmArgs g;
  g.A = l.A;
  g.B = l.B;
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = C;
  g.epi = Epi::kInt32;
  g.partial_ws = l.part;
  g.partial_ws_bytes = kGemmPartialBytes;
  g.chunk_ws = l.chunk;
  g.chunk_ws_bytes = kGemmPartialBytes;
  return launch_gemm(g, s);
}

rnl_status rnl_check_device_error(rnl_stream_t stream, int* site) {
  if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) {
    cudaGetLastError();
    return RNL_ERR_LAUNCH;
  }
  return read_device_errors(site);
}

rnl_status rnl_trace_enable(int on) {
  g_trace_on = on != 0;
  if (!g_trace_on) g_trace_pending = false;
  return RNL_OK;
}

int rnl_trace_read(char (*names)[32], float* ms, int max) {
  int n = g_trace_n < max ? g_trace_n : max;
  for (int i = 0; i < n; ++i) {
    TraceRec& t = g_trace[i];
    float v = -1.f;
    if (cudaEventSynchronize(t.b) == cudaSuccess && cudaEventElapsedTime(&v, t.a, t.b) == cudaSuccess) {
      ms[i] = v;
    } else {
      cudaGetLastError();
      ms[i] = -1.f;
    }
    if (names) std::memcpy(names[i], t.name, 32);
  }
  g_trace_n = 0;
  g_trace_pending = false;
  return n;
}

}  // extern "C"
