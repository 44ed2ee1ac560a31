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

__device__ __forceinline__ float activate(float v, int act) {
  switch (act) {
    case 1: return fmaxf(v, 0.f);
    case 2: return 0.5f * v * (1.f + erff(v * 0.70710678118654752440f));   // x * Phi(x)
    case 3: return __fdiv_rn(v, 1.f + expf(-v));                            // x * sigmoid(x)
    default: return v;
  }
}

// Eight accumulator values (FP32 bits) of columns col .. col+7 of one row -> out[0..7].
// The bias is read with one 16-byte load (every lane of a warp reads the same columns,
// so the load is a broadcast).
__device__ __forceinline__ void store8(__nv_bfloat16* out, const uint32_t* r, int64_t col,
                                       const Epilogue& e) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
  if (e.bias) {
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(e.bias + col));
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] += __uint_as_float(w[j] << 16);
      v[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
  if (e.act) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = activate(v[j], e.act);
  }
  st_global_v4_cs(out, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                  pack_bf16x2(v[6], v[7]));
}

}  // namespace bsmma
