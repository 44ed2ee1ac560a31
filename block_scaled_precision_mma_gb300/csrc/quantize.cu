// quantize.cu -- the quantisers that make the GEMMs' operands.
//
// MX ("[gfx1250] Add MXFP4 GEMM support to FlyDSL backend", the MXFP4 test helpers and
// their review: rowwise and columnwise data are quantised separately; BF16 and FP32
// input): per block of 32 values, E8M0 scale 2^e with e = floor(log2 amax) - emax
// (clamped to [-127, 127]; code 127 for an all-zero block) and codes RNE(x * 2^-e)
// saturated to the largest finite value, sign kept.
//
// Groupwise FP8 ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm": quantize_fp8_group
// and the per-group block layout of its scales): FP32 scale s = amax / 448 (1 for an
// all-zero block) per 1x128 activation block or 128x128 weight block, codes
// RNE-saturate(x / s) in E4M3, both divisions in FP32 (s never below 2^-149).
//
// Every kernel streams its input once from HBM with 16-byte loads and writes codes with
// coalesced stores; scales are a small side stream.  Grids are a few CTAs per SM with
// grid-stride loops.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace bsmma {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- element helpers
// 8 consecutive inputs from element index i (16-byte aligned), as FP32 (BF16 widens
// exactly).  Inputs are read once: streaming loads.
template <bool F32>
__device__ __forceinline__ void load8(const void* x, int64_t i, float (&v)[8]) {
  if constexpr (F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + i);
    const float4 a = __ldcs(p), b = __ldcs(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 r = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + i));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

// 4 consecutive inputs from element index i (8- or 16-byte aligned).
template <bool F32>
__device__ __forceinline__ void load4(const void* x, int64_t i, float (&v)[4]) {
  if constexpr (F32) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(x) + i));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  } else {
    const uint2 r = __ldcs(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(x) + i));
    v[0] = __uint_as_float(r.x << 16);
    v[1] = __uint_as_float(r.x & 0xFFFF0000u);
    v[2] = __uint_as_float(r.y << 16);
    v[3] = __uint_as_float(r.y & 0xFFFF0000u);
  }
}

// 2 consecutive inputs from element index i (4- or 8-byte aligned).
template <bool F32>
__device__ __forceinline__ void load2(const void* x, int64_t i, float& a, float& b) {
  if constexpr (F32) {
    const float2 r = __ldcs(reinterpret_cast<const float2*>(static_cast<const float*>(x) + i));
    a = r.x;
    b = r.y;
  } else {
    const uint32_t r = __ldcs(reinterpret_cast<const unsigned int*>(static_cast<const __nv_bfloat16*>(x) + i));
    a = __uint_as_float(r << 16);
    b = __uint_as_float(r & 0xFFFF0000u);
  }
}

// Two FP32 values -> two FP8 codes (RNE, saturated to the largest finite value), lo in
// the low byte.  The conversion keeps the sign bit of the input also when the result
// is zero (-0 and negatives that round to zero), as the quantisers require.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
  uint16_t r;
  if constexpr (FMT == BSMMA_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint32_t>(r);
}

// Two FP32 values -> two E2M1 codes in one byte (lo in the low nibble), RNE, saturated,
// sign kept as above.
__device__ __forceinline__ uint32_t fp4x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// floor(log2 a) of a finite FP32 a > 0, from its bits (subnormals included).
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ef = static_cast<int>((b >> 23) & 0xFFu);
  if (ef != 0) return ef - 127;
  return (31 - __clz(static_cast<int>(b & 0x7FFFFFu))) - 149;
}

// 2^k as FP32 for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float exp2i(int k) {
  return k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23)
                   : __uint_as_float(0x00400000u >> (-127 - k));
}

template <int FMT>
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
  if (!(amax > 0.f)) return 127u;
  constexpr int kEmax = FMT == BSMMA_E4M3 ? 8 : FMT == BSMMA_E5M2 ? 15 : 2;
  int e = floor_log2(amax) - kEmax;
  e = e < -127 ? -127 : (e > 127 ? 127 : e);
  return static_cast<uint32_t>(e + 127);
}

// ---------------------------------------------------------------- MX, rowwise
// Thread v handles inputs [8v, 8v+8) of the row-major tensor; four consecutive threads
// form one 32-value block (cols % 32 == 0, so blocks never straddle rows).
// Thread v handles inputs [8v, 8v+8) of the row-major tensor; four consecutive threads
// form one 32-value block (cols % 32 == 0, so blocks never straddle rows).
template <bool F32, int FMT>
__global__ void __launch_bounds__(kThreads) mx_quant_rows_kernel(const void* x, int64_t vecs,
                                                                  uint8_t* codes, uint8_t* scales) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kThreads + (threadIdx.x & ~31);
       base < vecs; base += stride) {
    const int64_t v = base + lane;
    const bool active = v < vecs;       // whole 4-lane blocks are active or not (vecs % 4 == 0)
    float val[8];
    float amax = 0.f;
    if (active) {
      load8<F32>(x, v * 8, val);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(val[j]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (!active) continue;
    const uint32_t sc = mx_scale_code<FMT>(amax);
    const float inv = exp2i(127 - static_cast<int>(sc));     // 2^-e
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(val[j], inv);
    if constexpr (FMT == BSMMA_E2M1) {
      const uint32_t w = fp4x2(y[0], y[1]) | (fp4x2(y[2], y[3]) << 8) | (fp4x2(y[4], y[5]) << 16) |
                         (fp4x2(y[6], y[7]) << 24);
      __stcs(reinterpret_cast<unsigned int*>(codes + v * 4), w);
    } else {
      const uint32_t w0 = fp8x2<FMT>(y[0], y[1]) | (fp8x2<FMT>(y[2], y[3]) << 16);
      const uint32_t w1 = fp8x2<FMT>(y[4], y[5]) | (fp8x2<FMT>(y[6], y[7]) << 16);
      __stcs(reinterpret_cast<uint2*>(codes + v * 8), make_uint2(w0, w1));
    }
    if ((lane & 3) == 0) scales[v >> 2] = static_cast<uint8_t>(sc);
  }
}

// ---------------------------------------------------------------- MX, columnwise
// A CTA takes a tile of 8 row blocks (256 rows) x 64 columns; warp w owns row block w
// of the tile and each lane two adjacent columns, so every row is read and written by
// a warp with one coalesced access.  The eight scales of a column are staged in shared
// memory and written as one run (scales are [cols][rows/32]).
constexpr int kColTile = 64, kRowBlocksPerTile = 8;

template <bool F32, int FMT>
__global__ void __launch_bounds__(kThreads) mx_quant_cols_kernel(const void* x, int64_t rows,
                                                                  int64_t cols, uint8_t* codes,
                                                                  uint8_t* scales) {
  __shared__ uint8_t sc_tile[kColTile][kRowBlocksPerTile];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rblocks = rows / 32;
  const int64_t col_tiles = (cols + kColTile - 1) / kColTile;
  const int64_t row_tiles = (rblocks + kRowBlocksPerTile - 1) / kRowBlocksPerTile;
  for (int64_t t = blockIdx.x; t < col_tiles * row_tiles; t += gridDim.x) {
    const int64_t rt = t / col_tiles, ct = t - rt * col_tiles;
    const int64_t rb = rt * kRowBlocksPerTile + warp;
    const int64_t c = ct * kColTile + 2 * lane;
    if (rb < rblocks && c < cols) {
      float a[32], b[32];
      float amax_a = 0.f, amax_b = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        load2<F32>(x, (rb * 32 + i) * cols + c, a[i], b[i]);
        amax_a = fmaxf(amax_a, fabsf(a[i]));
        amax_b = fmaxf(amax_b, fabsf(b[i]));
      }
      const uint32_t sa = mx_scale_code<FMT>(amax_a), sb = mx_scale_code<FMT>(amax_b);
      const float ia = exp2i(127 - static_cast<int>(sa)), ib = exp2i(127 - static_cast<int>(sb));
#pragma unroll
      for (int i = 0; i < 32; ++i)
        __stcs(reinterpret_cast<unsigned short*>(codes + (rb * 32 + i) * cols + c),
               static_cast<unsigned short>(fp8x2<FMT>(__fmul_rn(a[i], ia), __fmul_rn(b[i], ib))));
      sc_tile[2 * lane][warp] = static_cast<uint8_t>(sa);
      sc_tile[2 * lane + 1][warp] = static_cast<uint8_t>(sb);
    }
    __syncthreads();
    if (threadIdx.x < kColTile) {
      const int64_t cc = ct * kColTile + threadIdx.x;
      const int64_t rb0 = rt * kRowBlocksPerTile;
      if (cc < cols)
        for (int j = 0; j < kRowBlocksPerTile && rb0 + j < rblocks; ++j)
          scales[cc * rblocks + rb0 + j] = sc_tile[threadIdx.x][j];
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- groupwise FP8
// s = amax / 448 in FP32 (1 for an all-zero block, never below 2^-149); codes
// RNE-saturate(x / s).
__device__ __forceinline__ float group_scale(float amax) {
  if (!(amax > 0.f)) return 1.f;
  return fmaxf(__fdiv_rn(amax, 448.f), __uint_as_float(1u));
}

// E4M3 codes of eight values x / s (correctly rounded FP32 quotients).
__device__ __forceinline__ uint2 e4m3_codes8(const float (&x)[8], float s) {
  const uint32_t w0 = fp8x2<BSMMA_E4M3>(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s)) |
                      (fp8x2<BSMMA_E4M3>(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s)) << 16);
  const uint32_t w1 = fp8x2<BSMMA_E4M3>(__fdiv_rn(x[4], s), __fdiv_rn(x[5], s)) |
                      (fp8x2<BSMMA_E4M3>(__fdiv_rn(x[6], s), __fdiv_rn(x[7], s)) << 16);
  return make_uint2(w0, w1);
}

constexpr int kMaxGroups = 64;

// Activations X[total_M][K] over 1x128 blocks.  A CTA takes 64 rows x one 128-K block:
// sixteen threads share a row (eight consecutive values each, one 16-byte load), and
// every thread owns four rows, all loaded before any is reduced.  Codes go out as
// 8-byte stores; each row's scale to the per-group block layout.
template <bool F32>
__global__ void __launch_bounds__(kThreads) group_quant_kernel(const void* x, int64_t total_M,
                                                                int64_t K, const int64_t* m_sizes,
                                                                int G, uint8_t* codes, float* sx,
                                                                int* status) {
  __shared__ int64_t start[kMaxGroups + 1];
  __shared__ int64_t size[kMaxGroups];
  __shared__ int bad;
  if (threadIdx.x == 0) {
    int64_t row = 0;
    int b = 0;
    for (int g = 0; g < G; ++g) {
      const int64_t m = m_sizes[g];
      if (m < 0 || m > total_M) b = 1;
      start[g] = row;
      size[g] = m;
      if (!b) row += m;
    }
    if (row != total_M) b = 1;
    start[G] = row;
    bad = b;
    if (b && blockIdx.x == 0) report_status(status, kDevBadMSizes);
  }
  __syncthreads();
  if (bad) return;   // uniform: nothing is written
  const int seg = threadIdx.x & 15, rloc = threadIdx.x >> 4;   // rows rloc + 16i, i < 4
  // tile indices fit 32 bits (the entry point bounds total_M and K)
  const int KB = static_cast<int>(K / 128);
  const int row_tiles = static_cast<int>((total_M + 63) / 64);
  for (int t = blockIdx.x; t < row_tiles * KB; t += gridDim.x) {
    const int rt = t / KB, kb = t - rt * KB;
    float v[4][8] = {};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = static_cast<int64_t>(rt) * 64 + rloc + 16 * i;
      if (r < total_M) load8<F32>(x, r * K + kb * 128 + seg * 8, v[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = static_cast<int64_t>(rt) * 64 + rloc + 16 * i;
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (r >= total_M) continue;     // whole half-warps (the row is shared by 16 threads)
      const float s = group_scale(amax);
      __stcs(reinterpret_cast<uint2*>(codes + r * K + kb * 128 + seg * 8), e4m3_codes8(v[i], s));
      // the group owning row r: the last g with start[g] <= r (an empty group shares its
      // start with the next one, so it is never the last), by a binary search every lane
      // runs (no divergent scan)
      int lo = 0, hi = G;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= r) lo = mid;
        else hi = mid;
      }
      if (seg == 0) sx[start[lo] * KB + (r - start[lo]) + static_cast<int64_t>(kb) * size[lo]] = s;
    }
  }
}

// Weights W[G][N][K] over 128x128 blocks.  A CTA of 512 threads takes one block:
// thread t owns eight consecutive values of rows t/16 + 32i (i < 4), so each row
// segment is read and written by 16 threads with 16-byte (8-byte) accesses.
constexpr int kBlockThreads = 512;

template <bool F32>
__global__ void __launch_bounds__(kBlockThreads) block_quant_kernel(const void* w, int64_t G,
                                                                     int64_t N, int64_t K,
                                                                     uint8_t* codes, float* sw) {
  __shared__ float warp_amax[kBlockThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // block indices fit 32 bits (the entry point bounds G * N/128 * K/128)
  const int NB = static_cast<int>(N / 128), KB = static_cast<int>(K / 128);
  const int seg = threadIdx.x & 15, r0 = threadIdx.x >> 4;
  const int blocks = static_cast<int>(G) * NB * KB;
  for (int t = blockIdx.x; t < blocks; t += gridDim.x) {
    const int g = t / (NB * KB), rem = t - g * NB * KB;
    const int nb = rem / KB, kb = rem - nb * KB;
    float v[4][8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = static_cast<int64_t>(nb) * 128 + r0 + 32 * i;
      load8<F32>(w, (g * N + n) * K + kb * 128 + seg * 8, v[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) warp_amax[warp] = amax;
    __syncthreads();
    amax = warp_amax[0];
#pragma unroll
    for (int j = 1; j < kBlockThreads / 32; ++j) amax = fmaxf(amax, warp_amax[j]);
    const float s = group_scale(amax);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = static_cast<int64_t>(nb) * 128 + r0 + 32 * i;
      __stcs(reinterpret_cast<uint2*>(codes + (g * N + n) * K + kb * 128 + seg * 8),
             e4m3_codes8(v[i], s));
    }
    if (threadIdx.x == 0) sw[(static_cast<int64_t>(g) * NB + nb) * KB + kb] = s;
    __syncthreads();   // warp_amax is reused by the next block
  }
}

int grid_for(int64_t work, int per_sm, int sm_count) {
  const int64_t cap = static_cast<int64_t>(sm_count) * per_sm;
  return static_cast<int>(work < cap ? (work > 0 ? work : 1) : cap);
}

}  // namespace

bsmma_status launch_mx_quantize(const void* x, bool f32, int64_t rows, int64_t cols, bsmma_fmt fmt,
                                bool colwise, uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  if (rows == 0 || cols == 0) return BSMMA_OK;
  if (!colwise) {
    const int64_t vecs = rows * (cols / 8);
    const int grid = grid_for((vecs + kThreads - 1) / kThreads, 8, dev->sm_count);
#define BSMMA_ROWS(F, T) mx_quant_rows_kernel<F, T><<<grid, kThreads, 0, stream>>>(x, vecs, codes, scales)
    if (f32) {
      if (fmt == BSMMA_E4M3) BSMMA_ROWS(true, BSMMA_E4M3);
      else if (fmt == BSMMA_E5M2) BSMMA_ROWS(true, BSMMA_E5M2);
      else BSMMA_ROWS(true, BSMMA_E2M1);
    } else {
      if (fmt == BSMMA_E4M3) BSMMA_ROWS(false, BSMMA_E4M3);
      else if (fmt == BSMMA_E5M2) BSMMA_ROWS(false, BSMMA_E5M2);
      else BSMMA_ROWS(false, BSMMA_E2M1);
    }
#undef BSMMA_ROWS
  } else {
    const int64_t tiles = ((cols + kColTile - 1) / kColTile) *
                          ((rows / 32 + kRowBlocksPerTile - 1) / kRowBlocksPerTile);
    const int grid = grid_for(tiles, 8, dev->sm_count);
#define BSMMA_COLS(F, T) mx_quant_cols_kernel<F, T><<<grid, kThreads, 0, stream>>>(x, rows, cols, codes, scales)
    if (f32) {
      if (fmt == BSMMA_E4M3) BSMMA_COLS(true, BSMMA_E4M3);
      else BSMMA_COLS(true, BSMMA_E5M2);
    } else {
      if (fmt == BSMMA_E4M3) BSMMA_COLS(false, BSMMA_E4M3);
      else BSMMA_COLS(false, BSMMA_E5M2);
    }
#undef BSMMA_COLS
  }
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

bsmma_status launch_group_quantize(const void* x, bool f32, int64_t total_M, int64_t K,
                                   const int64_t* m_sizes, int G, uint8_t* codes, float* scales,
                                   cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const int64_t work = ((total_M + 63) / 64) * (K / 128);
  const int grid = grid_for(work, 8, dev->sm_count);
  if (f32)
    group_quant_kernel<true><<<grid, kThreads, 0, stream>>>(x, total_M, K, m_sizes, G, codes, scales, dev->status);
  else
    group_quant_kernel<false><<<grid, kThreads, 0, stream>>>(x, total_M, K, m_sizes, G, codes, scales, dev->status);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

bsmma_status launch_block_quantize(const void* w, bool f32, int64_t G, int64_t N, int64_t K,
                                   uint8_t* codes, float* scales, cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const int64_t work = G * (N / 128) * (K / 128);
  if (work == 0) return BSMMA_OK;
  const int grid = grid_for(work, 4, dev->sm_count);
  if (f32)
    block_quant_kernel<true><<<grid, kBlockThreads, 0, stream>>>(w, G, N, K, codes, scales);
  else
    block_quant_kernel<false><<<grid, kBlockThreads, 0, stream>>>(w, G, N, K, codes, scales);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace bsmma
