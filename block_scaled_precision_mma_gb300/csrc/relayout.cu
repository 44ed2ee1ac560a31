// relayout.cu -- plain E8M0 scales [rows][kblocks] -> tensor-core block-scale atoms.
//
// The GEMM takes plain scales and rearranges them itself ("[gfx1250] Add MXFP4
// GEMM support to FlyDSL backend", Description: plain scales in, shuffled inside
// the backend).  The target on sm_103a is the layout tcgen05.cp copies into
// tensor memory: 512-byte atoms of 128 rows x 4 K-blocks, atom (rb, kg) at
// (rb*KG + kg)*512, row r / block k at (r%32)*16 + (r/32)*4 + k.  Row blocks are
// padded to an even count, block groups too; padding holds 127 (scale 1.0).
//
// One thread per output 32-bit word (four K-blocks of one row): the writes are
// fully coalesced; each read gathers four bytes of one source row.  One launch
// handles up to two independent scale tensors (sA and sB of one GEMM).
#include <cuda_runtime.h>

#include "internal.h"

namespace bsmma {
namespace {

struct RelayoutJob {
  const uint8_t* src;
  uint8_t* dst;
  int64_t rows, kblocks, kg, words;
};

__device__ __forceinline__ void relayout_word(const RelayoutJob& j, int64_t w) {
  const int64_t atom = w >> 7;           // 128 words per atom
  const int wi = static_cast<int>(w & 127);
  const int64_t rb = atom / j.kg, kg = atom - rb * j.kg;
  const int64_t r = rb * 128 + (wi & 3) * 32 + (wi >> 2);
  uint32_t v = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t kb = kg * 4 + k;
    const uint32_t b = (r < j.rows && kb < j.kblocks) ? j.src[r * j.kblocks + kb] : 127u;
    v |= b << (8 * k);
  }
  reinterpret_cast<uint32_t*>(j.dst)[w] = v;
}

__global__ void __launch_bounds__(256) relayout_kernel(RelayoutJob j0, RelayoutJob j1) {
  const int64_t total = j0.words + j1.words;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (w < j0.words) relayout_word(j0, w);
    else relayout_word(j1, w - j0.words);
  }
}

RelayoutJob make_job(const uint8_t* s, int64_t rows, int64_t kb, uint8_t* out) {
  RelayoutJob j;
  j.src = s;
  j.dst = out;
  j.rows = rows;
  j.kblocks = kb;
  j.kg = 2 * ((kb + 7) / 8);
  j.words = (s && out) ? mx_scale_tiled_bytes(rows, kb) / 4 : 0;
  return j;
}

}  // namespace

bsmma_status launch_relayout(const uint8_t* s0, int64_t rows0, int64_t kb0, uint8_t* out0,
                             const uint8_t* s1, int64_t rows1, int64_t kb1, uint8_t* out1,
                             cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  RelayoutJob j0 = make_job(s0, rows0, kb0, out0), j1 = make_job(s1, rows1, kb1, out1);
  const int64_t total = j0.words + j1.words;
  if (total == 0) return BSMMA_OK;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(dev->sm_count) * 8;
  if (blocks > cap) blocks = cap;
  relayout_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(j0, j1);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace bsmma
