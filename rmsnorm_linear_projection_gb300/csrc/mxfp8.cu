// mxfp8.cu -- the MXFP8 mode of the linear atom (AT-10 pattern page, sec. 4:
// AT-09 quant_mode mxfp8, y = scaled_mm(x_fp8, w_fp8, FP32, x_scale,
// w_scale); SK-14 skeleton page, GMM-MXFP8: E4M3FN data, E8M0FNU scale
// factors, one scale per 64 elements).
//
// Front end, per token row (one warp per row):
//   y      = (x * rstd) * gamma                      FP32, as the W8A8 front end
//   per block of BLK (64, or the OCP MX 32) elements along K:
//   amax   = max |y|
//   X      = floor(log2 amax) - 8, at least -127     (8 = E4M3's largest exponent;
//                                                     an all-zero block gets -127)
//   scale  = X + 127                                 (the E8M0 byte)
//   code   = E4M3(y * 2^-X)                          round to nearest even,
//                                                     saturating to +-448
// The weight [N, K] arrives as E4M3 codes with E8M0 scales [N, K/BLK].
//
// Block-scaled path (the default): the codes go to the block-scaled tensor
// cores as they are (mxgemm.cu); this front end writes the rows' codes and
// their scale atoms (the 512-byte blocks the GEMM copies into tensor memory,
// each 64-element scale given to both 32-element hardware blocks), and its
// weight blocks arrange the weight's scales into atoms of the GEMM's tiles.
//
// Emulation path (RNL_MXFP8_NATIVE=0): A = bf16(value(code) * 2^X), and the
// weight is dequantised the same way.  value(code) * 2^X has four
// significant bits, so it is exact in bf16 whenever it lies in bf16's normal
// range (it can only fall below it for blocks with amax < 2^-116); the bf16
// tcgen05 GEMM on these operands then computes scaled_mm's sum with FP32
// accumulation.
//
// The codes of y * 2^-X come from cuda_fp8.h's saturating E4M3 conversion; y
// * 2^-X is exact (a power-of-two scaling that stays inside binary32's range:
// |y * 2^-X| < 512).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "exactsum.cuh"
#include "internal.h"

namespace rnl {
namespace {

constexpr int kWarps = 8;   // token rows per block
constexpr int kDqVec = 4;   // 16-code vectors per thread in the dequant blocks

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

// 2^e as a binary32 for e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two E4M3 codes (low byte first) -> their values.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t two) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return __half22float2(__half2(r));
}

// Two values -> two E4M3 codes (low byte = a), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2_code(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Quantises the 8 values f of one 16-byte vector of a row (lanes in groups
// of BLK/8 hold one block): writes the dequantised bf16 operand (a_dst, the
// emulation path) and the codes and the block's scale byte when asked, and
// returns the block's scale byte (127 for a lane outside the row).  Every
// lane of the warp calls it (the block maximum is a shuffle); `live` says
// whether this lane's vector is inside the row.
template <int BLK>
__device__ __forceinline__ int quant_vec(const float (&f)[8], bool live, uint4* a_dst,
                                         uint2* q_dst, uint8_t* s_dst) {
  constexpr int kGroup = BLK / 8;  // lanes per block
  float am = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(f[j]));
#pragma unroll
  for (int o = 1; o < kGroup; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const int eb = static_cast<int>((__float_as_uint(am) >> 23) & 0xFFu);
  int X = eb == 0 ? -127 : eb - 127 - 8;  // floor(log2 amax) - 8 for normal amax
  if (X < -127) X = -127;
  if (!live) return 127;
  const float inv = pow2f(-X);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = e4m3x2_code(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv));
  if (a_dst != nullptr) {
    const float p = pow2f(X);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = e4m3x2_value(c[i]);
      o[i] = pack_bf16x2(__fmul_rn(v.x, p), __fmul_rn(v.y, p));
    }
    *a_dst = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (q_dst != nullptr) *q_dst = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  if (s_dst != nullptr && (threadIdx.x & (kGroup - 1)) == 0) *s_dst = static_cast<uint8_t>(X + 127);
  return X + 127;
}

// Scale-factor atoms of the block-scaled GEMM (mxgemm.cu): for a matrix of
// `rows` rows cut into tiles of `rpt` rows, atom (tile, kg, t) holds the
// scale bytes of the tile's rows t * 128 .. t * 128 + 127 for the four
// 32-element blocks of k-block kg (128 elements); row r of the atom at word
// 4 (r % 32) + r / 32, byte j for block j.  A page block of 64 gives the same
// byte to its two 32-element halves; rows past the matrix and blocks past K
// get 127 (scale 1; their codes are zero).
template <int BLK>
__device__ __forceinline__ uint32_t sf_atom_word(const uint8_t* __restrict__ scales, int64_t rows, int K,
                                                 int rpt, int atoms, int num_kg, int64_t w) {
  const int64_t atom = w >> 7;
  const int within = static_cast<int>(w & 127);
  const int r = (within >> 2) + 32 * (within & 3);
  const int t = static_cast<int>(atom % atoms);
  const int64_t rest = atom / atoms;
  const int kg = static_cast<int>(rest % num_kg);
  const int64_t tile = rest / num_kg;
  const int rt = t * 128 + r;
  const int64_t row = tile * rpt + rt;
  if (rt >= rpt || row >= rows) return 0x7F7F7F7Fu;
  const int nb = K / BLK;
  uint32_t word = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k0 = (4 * kg + j) * 32;
    const uint32_t s = k0 < K ? __ldg(scales + row * nb + k0 / BLK) : 127u;
    word |= s << (8 * j);
  }
  return word;
}

struct MxRows {
  const uint4* x;
  const uint4* gamma;  // may be null
  int64_t T;
  int nvec;  // K / 8
  float inv_d, eps;
  uint4* A;           // bf16 [T, K] (emulation path) or null
  uint2* q_out;       // E4M3 [T, K] or null
  uint8_t* s_out;     // E8M0 [T, K / BLK] or null
  const uint4* w;     // E4M3 [N, K]
  const uint8_t* ws;  // E8M0 [N, K / BLK]
  int64_t w_nvec16;   // N * K / 16
  int k_vec16;        // K / 16
  uint4* Wb;          // bf16 [N, K] (emulation path)
  unsigned quant_blocks, dq_blocks;
  // block-scaled path: the weight blocks write the weight's scale atoms
  // instead of dequantising it, the rows write their own atoms
  bool native;
  uint32_t* sfa;      // A atoms (128-row tiles), words
  uint32_t* sfb;      // B atoms (bn-row tiles), words
  int64_t T_pad;      // T rounded up to 256: rows T .. T_pad - 1 get padding atoms
  int num_kg;         // k-blocks of 128
  int64_t N;
  int bn, b_atoms;
  int64_t sfb_words;
};

__device__ __forceinline__ void load_y(const uint4& u, const uint4* gamma, int v, float rstd,
                                       float (&f)[8]) {
  unpack8(u, f);
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], rstd);
  if (gamma != nullptr) {
    float g[8];
    unpack8(__ldg(gamma + v), g);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = __fmul_rn(f[j], g[j]);
  }
}

// The 16 lanes holding the 16 vectors (128 elements) of k-block kg = v / 16
// hand their blocks' scale bytes to the first of them, which writes the row's
// atom word: bytes of the 32-element blocks at lanes +0, +4, +8, +12.  Every
// lane calls it (shuffles).
__device__ __forceinline__ void put_atom_word(uint32_t* sfa_row, int sb, int v, int lane, int num_kg) {
  const int s1 = __shfl_down_sync(0xffffffffu, sb, 4);
  const int s2 = __shfl_down_sync(0xffffffffu, sb, 8);
  const int s3 = __shfl_down_sync(0xffffffffu, sb, 12);
  const int kg = v >> 4;
  if ((lane & 15) == 0 && kg < num_kg)
    sfa_row[static_cast<int64_t>(kg) * 128] = static_cast<uint32_t>(sb) | (static_cast<uint32_t>(s1) << 8) |
                                              (static_cast<uint32_t>(s2) << 16) | (static_cast<uint32_t>(s3) << 24);
}

// One token row.  VPL > 0: the row's vectors stay in registers (K <= 256 *
// VPL); VPL == 0: any K, x read twice (the sum of squares, then the blocks;
// the second read mostly hits L2), each pass with several 16-byte loads in
// flight per lane.
template <int MODE, int VPL, int BLK>
__device__ __forceinline__ void mx_quant_row(unsigned block, const MxRows& p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(block) * kWarps + (threadIdx.x >> 5);
  // the block-scaled path's atom words of this row: word 4 (row % 32) + (row / 32) % 4
  // of atom (row / 128, kg)
  uint32_t* const sfa_row = p.sfa != nullptr
                                ? p.sfa + (row / 128) * p.num_kg * 128 + 4 * (row % 32) + (row / 32) % 4
                                : nullptr;
  if (row >= p.T) {
    if (sfa_row != nullptr && row < p.T_pad)
      for (int kg = lane; kg < p.num_kg; kg += 32) sfa_row[static_cast<int64_t>(kg) * 128] = 0x7F7F7F7Fu;
    return;
  }
  const uint4* xr = p.x + row * p.nvec;
  const int iters = (p.nvec + 31) / 32;  // the same on every lane
  constexpr int kR = VPL > 0 ? VPL : 1;
  uint4 u[kR];
  uint64_t hs[4] = {0, 0, 0, 0}, ls[4] = {0, 0, 0, 0};  // packed float-float chains, (+0, +0)
  if (VPL > 0) {
#pragma unroll
    for (int i = 0; i < kR; ++i) {
      const int v = lane + 32 * i;
      u[i] = v < p.nvec ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kR; ++i) ffx2_add_squares8<MODE>(u[i], p.inv_d, hs, ls);
  } else {
    int v = lane;
    for (; v + 96 < p.nvec; v += 128) {
      uint4 w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = __ldg(xr + v + 32 * j);
#pragma unroll
      for (int j = 0; j < 4; ++j) ffx2_add_squares8<MODE>(w[j], p.inv_d, hs, ls);
    }
    for (; v < p.nvec; v += 32) ffx2_add_squares8<MODE>(__ldg(xr + v), p.inv_d, hs, ls);
  }
  const float rstd = rstd_of_sum<MODE>(ffx2_warp_total(hs, ls), p.inv_d, p.eps);
  const int nb = p.nvec / (BLK / 8);  // blocks per row
  uint4* ar = p.A != nullptr ? p.A + row * p.nvec : nullptr;
  uint2* qr = p.q_out != nullptr ? p.q_out + row * p.nvec : nullptr;
  uint8_t* sr = p.s_out != nullptr ? p.s_out + row * nb : nullptr;
  if (VPL > 0) {
#pragma unroll
    for (int i = 0; i < kR; ++i) {
      if (32 * i >= p.nvec) break;  // warp-uniform
      const int v = lane + 32 * i;
      const bool live = v < p.nvec;
      float f[8];
      load_y(u[i], live ? p.gamma : nullptr, v, rstd, f);
      const int sb = quant_vec<BLK>(f, live, ar ? ar + v : nullptr, qr ? qr + v : nullptr,
                                    sr ? sr + v / (BLK / 8) : nullptr);
      if (sfa_row != nullptr) put_atom_word(sfa_row, sb, v, lane, p.num_kg);
    }
  } else {
    for (int i = 0; i < iters; i += 2) {  // two vectors per lane in flight
      uint4 w[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int v = lane + 32 * (i + j);
        w[j] = (i + j < iters && v < p.nvec) ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (i + j >= iters) break;  // warp-uniform
        const int v = lane + 32 * (i + j);
        const bool live = v < p.nvec;
        float f[8];
        load_y(w[j], live ? p.gamma : nullptr, v, rstd, f);
        const int sb = quant_vec<BLK>(f, live, ar ? ar + v : nullptr, qr ? qr + v : nullptr,
                                      sr ? sr + v / (BLK / 8) : nullptr);
        if (sfa_row != nullptr) put_atom_word(sfa_row, sb, v, lane, p.num_kg);
      }
    }
  }
}

// Dequantises kDqVec x 16 codes per thread: value(code) * 2^(scale - 127) as
// bf16 (scale byte 255, the E8M0 NaN, gives NaN).
template <int BLK>
__device__ __forceinline__ void mx_dequant_block(unsigned block, const uint4* __restrict__ src,
                                                 const uint8_t* __restrict__ scales, int64_t nvec16,
                                                 int k_vec16, uint4* __restrict__ dst) {
  const int64_t base = static_cast<int64_t>(block) * blockDim.x * kDqVec + threadIdx.x;
  uint4 u[kDqVec];
  float sc[kDqVec];
#pragma unroll
  for (int i = 0; i < kDqVec; ++i) {
    const int64_t v = base + static_cast<int64_t>(i) * blockDim.x;
    u[i] = make_uint4(0u, 0u, 0u, 0u);
    sc[i] = 0.f;
    if (v < nvec16) {
      u[i] = __ldg(src + v);
      // row and column of the vector (32-bit division: nvec16 < 2^32 is
      // checked on the host)
      const uint32_t vv = static_cast<uint32_t>(v);
      const uint32_t n = vv / static_cast<uint32_t>(k_vec16);
      const uint32_t kv = vv - n * static_cast<uint32_t>(k_vec16);
      const int64_t nb = static_cast<int64_t>(k_vec16) * 16 / BLK;
      const int s = __ldg(scales + n * nb + kv * 16 / BLK);
      sc[i] = s == 255 ? __uint_as_float(0x7FC00000u) : pow2f(s - 127);
    }
  }
#pragma unroll
  for (int i = 0; i < kDqVec; ++i) {
    const int64_t v = base + static_cast<int64_t>(i) * blockDim.x;
    if (v >= nvec16) continue;
    const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 lo = e4m3x2_value(w[k] & 0xFFFFu);
      const float2 hi = e4m3x2_value(w[k] >> 16);
      o[2 * k] = pack_bf16x2(__fmul_rn(lo.x, sc[i]), __fmul_rn(lo.y, sc[i]));
      o[2 * k + 1] = pack_bf16x2(__fmul_rn(hi.x, sc[i]), __fmul_rn(hi.y, sc[i]));
    }
    dst[2 * v] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * v + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// The front end in one launch: quantising rows of x (ALU bound) and
// dequantising the weight (HBM bound) share no data, so their blocks are
// interleaved (even / odd while both last) and run side by side on every SM.
template <int MODE, int VPL, int BLK>
__global__ void __launch_bounds__(kWarps * 32, 4) mx_front_kernel(MxRows p) {
  const unsigned b = blockIdx.x;
  const unsigned both = p.quant_blocks < p.dq_blocks ? p.quant_blocks : p.dq_blocks;
  bool quant;
  unsigned idx;
  if (b < 2 * both) {
    quant = (b & 1u) == 0;
    idx = b >> 1;
  } else {
    quant = p.quant_blocks > p.dq_blocks;
    idx = b - both;
  }
  if (quant) {
    mx_quant_row<MODE, VPL, BLK>(idx, p);
  } else if (p.native) {
    // the weight's scale atoms: one word a thread
    const int64_t w = static_cast<int64_t>(idx) * blockDim.x + threadIdx.x;
    if (w < p.sfb_words)
      p.sfb[w] = sf_atom_word<BLK>(p.ws, p.N, p.k_vec16 * 16, p.bn, p.b_atoms, p.num_kg, w);
  } else {
    mx_dequant_block<BLK>(idx, p.w, p.ws, p.w_nvec16, p.k_vec16, p.Wb);
  }
}

// Both operands' scale atoms from scale bytes in the page's layout [rows,
// K / BLK] (scaled_mm on codes that were quantised elsewhere): one word a
// thread, A's atoms (128-row tiles) first.
template <int BLK>
__global__ void __launch_bounds__(256)
    mx_sf_prep_kernel(const uint8_t* __restrict__ a_scale, int64_t M, uint32_t* __restrict__ sfa,
                      int64_t a_words, const uint8_t* __restrict__ b_scale, int64_t N,
                      uint32_t* __restrict__ sfb, int64_t b_words, int K, int num_kg, int bn,
                      int b_atoms) {
  const int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (w < a_words)
    sfa[w] = sf_atom_word<BLK>(a_scale, M, K, 128, 1, num_kg, w);
  else if (w - a_words < b_words)
    sfb[w - a_words] = sf_atom_word<BLK>(b_scale, N, K, bn, b_atoms, num_kg, w - a_words);
}

// Dequantisation of two operands (activation codes, then weight codes).
template <int BLK>
__global__ void __launch_bounds__(256)
    mx_dequant2_kernel(const uint4* __restrict__ a, const uint8_t* __restrict__ as, int64_t a_nvec16,
                       uint4* __restrict__ a_dst, unsigned a_blocks, const uint4* __restrict__ b,
                       const uint8_t* __restrict__ bs, int64_t b_nvec16, uint4* __restrict__ b_dst,
                       int k_vec16) {
  if (blockIdx.x < a_blocks)
    mx_dequant_block<BLK>(blockIdx.x, a, as, a_nvec16, k_vec16, a_dst);
  else
    mx_dequant_block<BLK>(blockIdx.x - a_blocks, b, bs, b_nvec16, k_vec16, b_dst);
}

template <int MODE, int BLK>
void front_vpl(int vpl, unsigned grid, const MxRows& p, cudaStream_t s) {
  constexpr unsigned kT = kWarps * 32;
  // at most 64 registers a thread (four blocks of 256 threads per SM): the
  // weight's dequantisation is latency bound and wants the warps; rows
  // longer than 1024 take the two-read form
  if (vpl <= 4)
    mx_front_kernel<MODE, 4, BLK><<<grid, kT, 0, s>>>(p);
  else
    mx_front_kernel<MODE, 0, BLK><<<grid, kT, 0, s>>>(p);
}

inline unsigned dq_blocks_for(int64_t nvec16) {
  const int64_t per_block = 256 * kDqVec;
  return static_cast<unsigned>((nvec16 + per_block - 1) / per_block);
}

}  // namespace

bool mx_block_ok(int64_t block) { return block == 32 || block == 64; }

rnl_status launch_mx_front(const void* x, const void* gamma, int64_t T, int64_t K, float eps,
                           int mode, int64_t block, void* A, uint8_t* q_out, uint8_t* s_out,
                           const uint8_t* w_codes, const uint8_t* w_scale, int64_t N, void* Wb,
                           uint8_t* sfa, uint8_t* sfb, int bn, cudaStream_t s) {
  MxRows p;
  p.x = static_cast<const uint4*>(x);
  p.gamma = static_cast<const uint4*>(gamma);
  p.T = T;
  p.nvec = static_cast<int>(K / 8);
  p.inv_d = static_cast<float>(1.0 / static_cast<double>(K));
  p.eps = eps;
  p.A = static_cast<uint4*>(A);
  p.q_out = reinterpret_cast<uint2*>(q_out);
  p.s_out = s_out;
  p.w = reinterpret_cast<const uint4*>(w_codes);
  p.ws = w_scale;
  p.w_nvec16 = N * K / 16;
  p.k_vec16 = static_cast<int>(K / 16);
  p.Wb = static_cast<uint4*>(Wb);
  p.native = sfa != nullptr;
  p.sfa = reinterpret_cast<uint32_t*>(sfa);
  p.sfb = reinterpret_cast<uint32_t*>(sfb);
  p.T_pad = (T + 255) / 256 * 256;  // whole 256-row tiles of the CTA-pair GEMM
  p.num_kg = static_cast<int>((K + 127) / 128);
  p.N = N;
  p.bn = bn;
  p.b_atoms = (bn + 127) / 128;
  p.sfb_words = p.native ? ((N + bn - 1) / bn) * p.num_kg * p.b_atoms * 128 : 0;
  p.quant_blocks = static_cast<unsigned>(((p.native ? p.T_pad : T) + kWarps - 1) / kWarps);
  p.dq_blocks = p.native ? static_cast<unsigned>((p.sfb_words + 255) / 256) : dq_blocks_for(p.w_nvec16);
  const unsigned grid = p.quant_blocks + p.dq_blocks;
  if (grid == 0) return RNL_OK;
  const int vpl = (p.nvec + 31) / 32;
  trace_before(s);
  if (mode == RNL_NORM_RSQRT) {
    if (block == 64)
      front_vpl<0, 64>(vpl, grid, p, s);
    else
      front_vpl<0, 32>(vpl, grid, p, s);
  } else {
    if (block == 64)
      front_vpl<1, 64>(vpl, grid, p, s);
    else
      front_vpl<1, 32>(vpl, grid, p, s);
  }
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "mxfp8_front");
  return st;
}

rnl_status launch_mx_dequant2(const uint8_t* a_codes, const uint8_t* a_scale, int64_t M,
                              const uint8_t* b_codes, const uint8_t* b_scale, int64_t N, int64_t K,
                              int64_t block, void* A, void* B, cudaStream_t s) {
  const int64_t a16 = M * K / 16, b16 = N * K / 16;
  const unsigned ab = dq_blocks_for(a16), bb = dq_blocks_for(b16);
  if (ab + bb == 0) return RNL_OK;
  const auto* ap = reinterpret_cast<const uint4*>(a_codes);
  const auto* bp = reinterpret_cast<const uint4*>(b_codes);
  const int kv = static_cast<int>(K / 16);
  trace_before(s);
  if (block == 64)
    mx_dequant2_kernel<64><<<ab + bb, 256, 0, s>>>(ap, a_scale, a16, static_cast<uint4*>(A), ab, bp,
                                                   b_scale, b16, static_cast<uint4*>(B), kv);
  else
    mx_dequant2_kernel<32><<<ab + bb, 256, 0, s>>>(ap, a_scale, a16, static_cast<uint4*>(A), ab, bp,
                                                   b_scale, b16, static_cast<uint4*>(B), kv);
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "mxfp8_dequant");
  return st;
}

rnl_status launch_mx_sf_prep(const uint8_t* a_scale, int64_t M, const uint8_t* b_scale, int64_t N,
                             int64_t K, int64_t block, uint8_t* sfa, uint8_t* sfb, int bn,
                             cudaStream_t s) {
  const int num_kg = static_cast<int>((K + 127) / 128);
  const int b_atoms = (bn + 127) / 128;
  const int64_t a_words = ((M + 255) / 256) * 2 * num_kg * 128;  // whole 256-row tiles
  const int64_t b_words = ((N + bn - 1) / bn) * num_kg * b_atoms * 128;
  const int64_t blocks = (a_words + b_words + 255) / 256;
  if (blocks == 0) return RNL_OK;
  auto* wa = reinterpret_cast<uint32_t*>(sfa);
  auto* wb = reinterpret_cast<uint32_t*>(sfb);
  trace_before(s);
  if (block == 64)
    mx_sf_prep_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        a_scale, M, wa, a_words, b_scale, N, wb, b_words, static_cast<int>(K), num_kg, bn, b_atoms);
  else
    mx_sf_prep_kernel<32><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        a_scale, M, wa, a_words, b_scale, N, wb, b_words, static_cast<int>(K), num_kg, bn, b_atoms);
  const rnl_status st = cudaGetLastError() == cudaSuccess ? RNL_OK : RNL_ERR_LAUNCH;
  trace_after(s, "mxfp8_scale_atoms");
  return st;
}

}  // namespace rnl
