// epilogue.cuh -- the dense GEMMs' output stage: an optional per-column BF16 bias and an
// activation applied to the FP32 accumulator, then BF16 round-to-nearest-even and
// streaming 16-byte stores.  The plain GEMM is the case without either; bias and
// activation are the follow-up named in "[gfx1250] Add MXFP4 GEMM support to FlyDSL
// backend", Description.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace bsmma {

struct Epilogue {
  const __nv_bfloat16* bias;   // [N] or nullptr
  int act;                     // 0 none, 1 ReLU, 2 GELU (erf form), 3 SiLU
};

// GELU in its erf form, x * Phi(x) = x (1 + erf(x / sqrt 2)) / 2.  erf comes from
// Abramowitz & Stegun, "Handbook of Mathematical Functions", formula 7.1.26: for u >= 0,
// erfc(u) = (a1 t + a2 t^2 + ... + a5 t^5) e^(-u^2) + eps with t = 1 / (1 + p u) and
// |eps| <= 1.5e-7.  With q = erfc(|x| / sqrt 2), 1 + erf(x / sqrt 2) is 2 - q for x >= 0
// and q itself for x < 0, so negative inputs lose nothing to cancellation; the error in
// the result stays below about |x| * 5e-7 (reciprocal and exponential by the fast
// intrinsics; 2.8e-7 measured against erf in float32 over [-12, 12]).
__device__ __forceinline__ float gelu_erf(float x) {
  const float u = fabsf(x) * 0.70710678118654752440f;
  const float t = __fdividef(1.f, fmaf(0.3275911f, u, 1.f));
  float poly = 1.061405429f;
  poly = fmaf(poly, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  const float q = poly * t * __expf(-u * u);
  return 0.5f * x * (x >= 0.f ? 2.f - q : q);
}

// gelu_erf on two values at once: the same operations in the same order, with the adds,
// multiplies and FMAs as packed two-lane instructions (each lane rounded as the scalar
// instruction rounds), about 40% fewer instructions; the reciprocal and the exponential
// stay per lane.
__device__ __forceinline__ float2 gelu_erf2(float2 x) {
  const float2 u = __fmul2_rn(make_float2(fabsf(x.x), fabsf(x.y)),
                              make_float2(0.70710678118654752440f, 0.70710678118654752440f));
  const float2 d = __ffma2_rn(make_float2(0.3275911f, 0.3275911f), u, make_float2(1.f, 1.f));
  const float2 t = make_float2(__fdividef(1.f, d.x), __fdividef(1.f, d.y));
  float2 poly = make_float2(1.061405429f, 1.061405429f);
  poly = __ffma2_rn(poly, t, make_float2(-1.453152027f, -1.453152027f));
  poly = __ffma2_rn(poly, t, make_float2(1.421413741f, 1.421413741f));
  poly = __ffma2_rn(poly, t, make_float2(-0.284496736f, -0.284496736f));
  poly = __ffma2_rn(poly, t, make_float2(0.254829592f, 0.254829592f));
  const float2 uu = __fmul2_rn(make_float2(-u.x, -u.y), u);
  const float2 q = __fmul2_rn(__fmul2_rn(poly, t), make_float2(__expf(uu.x), __expf(uu.y)));
  const float2 two_minus_q = __fadd2_rn(make_float2(2.f, 2.f), make_float2(-q.x, -q.y));
  const float2 h = __fmul2_rn(make_float2(0.5f, 0.5f), x);
  return __fmul2_rn(h, make_float2(x.x >= 0.f ? two_minus_q.x : q.x,
                                   x.y >= 0.f ? two_minus_q.y : q.y));
}

// x * sigmoid(x) = x / (1 + e^-x); for x below about -88 the denominator overflows and the
// quotient is 0, the limit.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// Eight accumulator values (FP32 bits) of columns col .. col+7 of one row -> eight BF16
// results packed two per word, with the activation ACT (Epilogue::act) fixed at compile
// time, so that a kernel carries only its own activation's code.  The bias is read with
// one 16-byte load (every lane of a warp reads the same columns, so the load is a
// broadcast).
template <int ACT>
__device__ __forceinline__ void apply8_act(const uint32_t* r, int64_t col,
                                           const __nv_bfloat16* bias, uint32_t (&o)[4]) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
  if (bias) {
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias + col));
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] += __uint_as_float(w[j] << 16);
      v[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
  if constexpr (ACT == 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fmaxf(v[j], 0.f);
  } else if constexpr (ACT == 2) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float2 g = gelu_erf2(make_float2(v[j], v[j + 1]));
      v[j] = g.x;
      v[j + 1] = g.y;
    }
  } else if constexpr (ACT == 3) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = silu(v[j]);
  }
  o[0] = pack_bf16x2(v[0], v[1]);
  o[1] = pack_bf16x2(v[2], v[3]);
  o[2] = pack_bf16x2(v[4], v[5]);
  o[3] = pack_bf16x2(v[6], v[7]);
}

// Same, with the activation chosen at run time.
__device__ __forceinline__ void apply8(const uint32_t* r, int64_t col, const Epilogue& e,
                                       uint32_t (&o)[4]) {
  switch (e.act) {
    case 1: apply8_act<1>(r, col, e.bias, o); break;
    case 2: apply8_act<2>(r, col, e.bias, o); break;
    case 3: apply8_act<3>(r, col, e.bias, o); break;
    default: apply8_act<0>(r, col, e.bias, o); break;
  }
}

// Same, stored to out[0..7] with one streaming 16-byte store.
__device__ __forceinline__ void store8(__nv_bfloat16* out, const uint32_t* r, int64_t col,
                                       const Epilogue& e) {
  uint32_t o[4];
  apply8(r, col, e, o);
  st_global_v4_cs(out, o[0], o[1], o[2], o[3]);
}

}  // namespace bsmma
