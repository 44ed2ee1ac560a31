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
// RNE-saturate(x / s) in E4M3, both divisions in FP32 (s never below 2^-149); the
// per-value quotient comes from an exact FMA sequence on the block's reciprocal.
//
// Every kernel streams its input once from HBM with 16-byte loads and writes codes with
// coalesced stores; scales are a small side stream.  Grids are a few CTAs per SM with
// grid-stride loops.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

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

// The correctly rounded FP32 quotient x / s from y = RN(1 / s) by FMA corrections
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990; the division theorem in Muller et al.,
// "Handbook of Floating-Point Arithmetic", ch. 4): if q is a faithful approximation of
// x / s and y is within half an ulp of 1 / s, then r = x - s q is exact and
// RN(q + r y) = RN(x / s).  q0 = RN(x y) is within 1.5 ulp, so one correction makes it
// faithful and a second makes it exact.  The conditions hold wherever the code depends
// on the quotient: for s in [2^-88, FLT_MAX] every |x / s| >= 2^-11 has a normal x
// (>= 2^-99) and a remainder on a grid of at least 2^-146, so nothing underflows; a
// smaller quotient gives a code of zero either way, whose sign is taken from x.
constexpr float kFastDivMinScale = 0x1p-88f;

__device__ __forceinline__ bool fast_div_ok(float s) {
  return s >= kFastDivMinScale && s <= 3.40282347e38f;   // also false for NaN
}

// The sequence on a pair of values with packed FP32 operations (each lane rounds like
// the scalar operation).  The sign of a zero quotient is restored by the caller.
__device__ __forceinline__ float2 quotient2_rn(float2 x, float2 neg_s, float2 y) {
  const float2 q0 = __fmul2_rn(x, y);
  const float2 q1 = __ffma2_rn(__ffma2_rn(q0, neg_s, x), y, q0);
  return __ffma2_rn(__ffma2_rn(q1, neg_s, x), y, q1);
}

// Sign bits of four FP32 values at bits 7, 15, 23 and 31 (one per code byte).
__device__ __forceinline__ uint32_t sign_bytes4(float a, float b, float c, float d) {
  const uint32_t ab = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0073);
  const uint32_t cd = __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x0073);
  return __byte_perm(ab, cd, 0x5410) & 0x80808080u;
}

// E4M3 codes of eight values x / s, the quotients correctly rounded in FP32: by the FMA
// sequence on pairs when fast_div_ok(s), with y = RN(1 / s), else by IEEE division.  Each
// code's sign bit is then OR-ed in from x, which gives a quotient that vanished (or an
// x of -0) the sign of x; a code of a negative quotient has that bit already.
__device__ __forceinline__ uint2 e4m3_codes8(const float (&x)[8], float s, float y, bool fast) {
  float q[8];
  if (fast) {
    const float2 ns2 = make_float2(-s, -s), y2 = make_float2(y, y);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 r = quotient2_rn(make_float2(x[2 * j], x[2 * j + 1]), ns2, y2);
      q[2 * j] = r.x;
      q[2 * j + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(x[j], s);
  }
  const uint32_t w0 = fp8x2<BSMMA_E4M3>(q[0], q[1]) | (fp8x2<BSMMA_E4M3>(q[2], q[3]) << 16);
  const uint32_t w1 = fp8x2<BSMMA_E4M3>(q[4], q[5]) | (fp8x2<BSMMA_E4M3>(q[6], q[7]) << 16);
  return make_uint2(w0 | sign_bytes4(x[0], x[1], x[2], x[3]),
                    w1 | sign_bytes4(x[4], x[5], x[6], x[7]));
}

constexpr int kMaxGroups = 64;

// Eight consecutive FP32 values from shared memory (BF16 widens exactly).
template <bool F32>
__device__ __forceinline__ void lds8(const uint8_t* p, float (&v)[8]) {
  if constexpr (F32) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 16);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

// Activations X[total_M][K] over 1x128 blocks.  A persistent CTA keeps a ring of
// kXStages tiles of 64 rows x 128 values in shared memory.  Warp 8 produces: one tensor
// copy per tile (rows past total_M arrive as zeros and are not stored), each slot reused
// once its `empty` barrier has one arrival from every consumer warp.  Warps 0-7 consume:
// warp w owns rows 8w .. 8w + 7 of every tile, waits on the tile's `full` barrier itself
// and releases the slot as soon as its rows are in registers, so no CTA-wide barrier is
// taken per tile.  Four threads share a row: thread `seg` of row `row` owns the 8-value
// chunks at columns seg*8 + 32k (k < 4), visited from k = row & 1 on so that a warp's even
// and odd rows read opposite halves of the shared-memory banks.  Per row: the 4-lane amax,
// the scale, its reciprocal and the group lookup, spread over 32 values.  Codes go out as
// 8-byte stores (32 contiguous bytes per row and chunk); each row's scale to the
// per-group block layout.  Every wait is bounded; a timeout raises a CTA-wide abort flag
// that ends the other warps' waits, and the producer waits (bounded) for its copies in
// flight before it exits.
constexpr int kXStages = 4;
constexpr int kXConsumerWarps = 8;
constexpr int kXThreads = (kXConsumerWarps + 1) * 32;

template <bool F32>
struct XRing {
  static constexpr int kRowBytes = 128 * (F32 ? 4 : 2);
  static constexpr int kBytes = 64 * kRowBytes;               // one 64 x 128 tile
  // 1 KB of slack puts the ring on a 1024-byte boundary (tensor copies need 128)
  static constexpr int kSmem = 1024 + kXStages * kBytes + 2 * kXStages * 8;
};

template <bool F32>
__global__ void __launch_bounds__(kXThreads) group_quant_kernel(
    const __grid_constant__ CUtensorMap tmX, int64_t total_M, int64_t K, const int64_t* m_sizes,
    int G, uint8_t* codes, float* sx, int* status, uint64_t limit_ns) {
  using R = XRing<F32>;
  extern __shared__ __align__(16) uint8_t xring_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(xring_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kXStages * R::kBytes);
  uint64_t* empty = full + kXStages;
  __shared__ int64_t start[kMaxGroups + 1];
  __shared__ int64_t size[kMaxGroups];
  __shared__ int bad;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // tile indices fit 32 bits (the entry point bounds total_M and K)
  const int KB = static_cast<int>(K / 128);
  const int tiles = static_cast<int>((total_M + 63) / 64) * KB;
  const int mine = tiles > static_cast<int>(blockIdx.x)
                       ? (tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                       : 0;
  auto tile_of = [&](int it, int& rt, int& kb) {
    const int t = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
    rt = t / KB;
    kb = t - rt * KB;
  };
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
    abort_flag = 0;
    if (b && blockIdx.x == 0) report_status(status, kDevBadMSizes);
    if (!b && mine > 0) {
      for (int st = 0; st < kXStages; ++st) {
        mbar_init(&full[st], 1);
        mbar_init(&empty[st], kXConsumerWarps);
      }
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (bad || mine == 0) return;   // uniform: nothing is written, nothing was issued
  if (warp == kXConsumerWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tmX);
      int issued = 0;
      for (int it = 0; it < mine; ++it) {
        const int slot = it % kXStages;
        if (it >= kXStages &&
            !mbar_wait(&empty[slot], ((it / kXStages) - 1) & 1, limit_ns, &abort_flag, status))
          break;
        int rt, kb;
        tile_of(it, rt, kb);
        mbar_arrive_expect_tx(&full[slot], R::kBytes);
        tma_load_2d(&tmX, &full[slot], ring + slot * R::kBytes, kb * (F32 ? 128 : 64), rt * 64);
        issued = it + 1;
      }
      // copies still in flight must land before the CTA's memory is released
      for (int j = issued > kXStages ? issued - kXStages : 0; j < issued; ++j) {
        volatile int no_abort = 0;
        mbar_wait(&full[j % kXStages], (j / kXStages) & 1, limit_ns / 4 + 1, &no_abort, nullptr);
      }
    }
    return;
  }
  // ------------------------------------------------------------------ consumers
  const int seg = lane & 3, rloc = warp * 8 + (lane >> 2);
  const int rot = rloc & 1;
  for (int it = 0; it < mine; ++it) {
    const int slot = it % kXStages;
    if (!mbar_wait(&full[slot], (it / kXStages) & 1, limit_ns, &abort_flag, status)) break;
    const uint8_t* trow = ring + slot * R::kBytes + rloc * R::kRowBytes;
    float v[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      lds8<F32>(trow + (seg * 8 + 32 * ((k + rot) & 3)) * (F32 ? 4 : 2), v[k]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);   // this warp's rows are in registers
    int rt, kb;
    tile_of(it, rt, kb);
    const int64_t row0 = static_cast<int64_t>(rt) * 64;
    const int64_t r = row0 + rloc;
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[k][j]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (r < total_M) {                    // whole 4-lane row groups
      const float s = group_scale(amax);
      const bool fast = fast_div_ok(s);
      const float y = fast ? __frcp_rn(s) : 0.f;
      uint8_t* out = codes + r * K + kb * 128 + seg * 8;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        __stcs(reinterpret_cast<uint2*>(out + 32 * ((k + rot) & 3)), e4m3_codes8(v[k], s, y, fast));
      // the group owning row r: the last g with start[g] <= r (an empty group shares its
      // start with the next one, so it is never the last); a binary search for the tile's
      // first row, which every lane runs, then a walk past group ends
      int g = 0, hi = G;
      while (hi - g > 1) {
        const int mid = (g + hi) >> 1;
        if (start[mid] <= row0) g = mid;
        else hi = mid;
      }
      while (r >= start[g + 1]) ++g;    // start[G] = total_M > r ends the walk
      if (seg == 0) sx[start[g] * KB + (r - start[g]) + static_cast<int64_t>(kb) * size[g]] = s;
    }
  }
}

// Weights W[G][N][K] over 128x128 blocks.  A persistent CTA of 512 threads keeps a ring
// of kWStages blocks in shared memory, each filled by one tensor copy issued by thread 0,
// and quantises the oldest while the others stream in.
// Thread t owns eight consecutive values of rows t/16 + 32i (i < 4) of a block.  Thread 0
// alone waits on a block's barrier (bounded) and the CTA barrier hands the outcome to
// every thread, so all leave the loop together.
constexpr int kBlockThreads = 512;
constexpr int kWStages = 3;

template <bool F32>
struct WRing {
  static constexpr int kRowBytes = 128 * (F32 ? 4 : 2);
  static constexpr int kBytes = 128 * kRowBytes;              // one 128x128 block
  // the ring starts on a 1024-byte boundary (a tensor copy's shared-memory destination must
  // be 128-byte aligned), so 1 KB of slack in front of it
  static constexpr int kSmem = 1024 + kWStages * kBytes + kWStages * 8;
};

// One 128x128 block of the weights' 3-D tensor map (32-bit words x N rows x G) into
// shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(const void* tmap, uint64_t* bar, void* dst,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

template <bool F32>
__global__ void __launch_bounds__(kBlockThreads) block_quant_kernel(
    const __grid_constant__ CUtensorMap tmW, int64_t G, int64_t N, int64_t K, uint8_t* codes,
    float* sw, int* status, uint64_t limit_ns) {
  using R = WRing<F32>;
  extern __shared__ __align__(16) uint8_t ring_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(ring_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kWStages * R::kBytes);
  __shared__ float warp_amax[2][kBlockThreads / 32];
  __shared__ int landed;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // block indices fit 32 bits (the entry point bounds G * N/128 * K/128)
  const int NB = static_cast<int>(N / 128), KB = static_cast<int>(K / 128);
  const int seg = threadIdx.x & 15, r0 = threadIdx.x >> 4;
  const int blocks = static_cast<int>(G) * NB * KB;
  const int mine = blocks > static_cast<int>(blockIdx.x)
                       ? (blocks - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                       : 0;
  // block (g, nb, kb) of this CTA's iteration `it`
  auto block_of = [&](int it, int& g, int& nb, int& kb) {
    const int t = static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
    g = t / (NB * KB);
    const int rem = t - g * NB * KB;
    nb = rem / KB;
    kb = rem - nb * KB;
    return t;
  };
  // thread 0: the block of iteration `it` into its slot
  auto issue = [&](int it) {
    if (it >= mine) return;
    int g, nb, kb;
    block_of(it, g, nb, kb);
    const int slot = it % kWStages;
    mbar_arrive_expect_tx(&full[slot], R::kBytes);
    tma_load_3d(&tmW, &full[slot], ring + slot * R::kBytes, kb * (F32 ? 128 : 64), nb * 128, g);
  };
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmW);
    for (int st = 0; st < kWStages; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
    for (int it = 0; it < kWStages; ++it) issue(it);
  }
  int it = 0;
  for (; it < mine; ++it) {
    const int slot = it % kWStages;
    if (threadIdx.x == 0) {
      volatile int no_abort = 0;
      landed = mbar_wait(&full[slot], (it / kWStages) & 1, limit_ns, &no_abort, status) ? 1 : 0;
    }
    __syncthreads();                      // the block is visible to every thread
    if (!landed) break;                   // uniform
    const uint8_t* blk = ring + slot * R::kBytes;
    float v[4][8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) lds8<F32>(blk + (r0 + 32 * i) * R::kRowBytes + seg * (F32 ? 32 : 16), v[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) warp_amax[it & 1][warp] = amax;
    __syncthreads();                      // the slot is read out; all warp maxima are in
    if (threadIdx.x == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(it + kWStages);
    }
    amax = warp_amax[it & 1][0];
#pragma unroll
    for (int j = 1; j < kBlockThreads / 32; ++j) amax = fmaxf(amax, warp_amax[it & 1][j]);
    const float s = group_scale(amax);
    const bool fast = fast_div_ok(s);
    const float y = fast ? __frcp_rn(s) : 0.f;
    int g, nb, kb;
    const int t = block_of(it, g, nb, kb);
    const int64_t o = (static_cast<int64_t>(g) * N + static_cast<int64_t>(nb) * 128) * K + kb * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      __stcs(reinterpret_cast<uint2*>(codes + o + static_cast<int64_t>(r0 + 32 * i) * K + seg * 8),
             e4m3_codes8(v[i], s, y, fast));
    if (threadIdx.x == 0) sw[t] = s;
  }
  // after a timeout, copies already issued must land before the CTA's memory is released
  if (threadIdx.x == 0)
    for (int j = it; j < it + kWStages && j < mine; ++j) {
      volatile int no_abort = 0;
      mbar_wait(&full[j % kWStages], (j / kWStages) & 1, limit_ns / 4 + 1, &no_abort, nullptr);
    }
}

// A BF16 / FP32 tensor as a tensor map of 32-bit words (`rank` dimensions, innermost
// first; `strides` in bytes for dimensions 1..rank-1), no swizzle, zero fill outside.
bsmma_status encode_words(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static const Encode encode = []() -> Encode {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<Encode>(fn);
  }();
  if (!encode) return BSMMA_ERR_CUDA;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], e[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    if (i > 0) st[i - 1] = strides[i - 1];
  }
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, static_cast<cuuint32_t>(rank),
                            const_cast<void*>(base), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSMMA_OK : BSMMA_ERR_INVALID_ARG;
}

// Resident CTAs per SM of a ring kernel (its ring takes much of shared memory); sets the
// kernel's dynamic shared-memory limit on first use.  0 on failure.
template <auto Kern>
int ring_ctas_per_sm(int threads, int smem) {
  static int n = -1;   // one per kernel; benign race: every thread computes the same value
  if (n < 0) {
    int k = 0;
    if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, Kern, threads, smem) != cudaSuccess)
      return 0;
    n = k;
  }
  return n;
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
  const int per_sm = f32 ? ring_ctas_per_sm<group_quant_kernel<true>>(kXThreads, XRing<true>::kSmem)
                         : ring_ctas_per_sm<group_quant_kernel<false>>(kXThreads, XRing<false>::kSmem);
  if (per_sm < 1) return BSMMA_ERR_CUDA;
  // X[total_M][K] as 32-bit words: K/2 (BF16) or K (FP32) words x total_M rows, one
  // 64 x 128-value tile per box.  An empty X has no tiles: the kernel only checks m_sizes
  // and never reads the (zeroed) map.
  CUtensorMap tm;
  std::memset(&tm, 0, sizeof(tm));
  if (total_M > 0) {
    const uint64_t row_bytes = static_cast<uint64_t>(K) * (f32 ? 4 : 2);
    const uint64_t dims[2] = {row_bytes / 4, static_cast<uint64_t>(total_M)};
    const uint64_t strides[1] = {row_bytes};
    const uint32_t box[2] = {f32 ? 128u : 64u, 64u};
    st = encode_words(&tm, x, 2, dims, strides, box);
    if (st != BSMMA_OK) return st;
  }
  const int grid = grid_for(work, per_sm, dev->sm_count);
  if (f32)
    group_quant_kernel<true><<<grid, kXThreads, XRing<true>::kSmem, stream>>>(
        tm, total_M, K, m_sizes, G, codes, scales, dev->status, wait_limit_ns());
  else
    group_quant_kernel<false><<<grid, kXThreads, XRing<false>::kSmem, stream>>>(
        tm, total_M, K, m_sizes, G, codes, scales, dev->status, wait_limit_ns());
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
  const int per_sm = f32 ? ring_ctas_per_sm<block_quant_kernel<true>>(kBlockThreads, WRing<true>::kSmem)
                         : ring_ctas_per_sm<block_quant_kernel<false>>(kBlockThreads, WRing<false>::kSmem);
  if (per_sm < 1) return BSMMA_ERR_CUDA;
  // W[G][N][K] as 32-bit words: K/2 (BF16) or K (FP32) words x N rows x G matrices,
  // one 128x128-value block per box
  CUtensorMap tm;
  const uint64_t row_bytes = static_cast<uint64_t>(K) * (f32 ? 4 : 2);
  const uint64_t dims[3] = {row_bytes / 4, static_cast<uint64_t>(N), static_cast<uint64_t>(G)};
  const uint64_t strides[2] = {row_bytes, row_bytes * static_cast<uint64_t>(N)};
  const uint32_t box[3] = {f32 ? 128u : 64u, 128u, 1u};
  st = encode_words(&tm, w, 3, dims, strides, box);
  if (st != BSMMA_OK) return st;
  const int grid = grid_for(work, per_sm, dev->sm_count);
  if (f32)
    block_quant_kernel<true><<<grid, kBlockThreads, WRing<true>::kSmem, stream>>>(
        tm, G, N, K, codes, scales, dev->status, wait_limit_ns());
  else
    block_quant_kernel<false><<<grid, kBlockThreads, WRing<false>::kSmem, stream>>>(
        tm, G, N, K, codes, scales, dev->status, wait_limit_ns());
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace bsmma
