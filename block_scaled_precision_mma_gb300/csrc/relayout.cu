// relayout.cu -- plain E8M0 scales [rows][kblocks] -> tensor-core block-scale atoms.
//
// The GEMM takes plain scales and rearranges them itself ("[gfx1250] Add MXFP4
// GEMM support to FlyDSL backend", Description: plain scales in, shuffled inside
// the backend).  The target on sm_103a is the layout tcgen05.cp copies into
// tensor memory: 512-byte atoms of 128 rows x 4 K-blocks, atom (rb, kg) at
// (rb*KG + kg)*512, row r / block k at (r%32)*16 + (r/32)*4 + k.  Row blocks are
// padded to an even count, block groups too; padding holds 127 (scale 1.0).
//
// One launch handles up to two independent scale tensors (sA and sB of one GEMM).
#include <cuda_runtime.h>

#include "internal.h"

namespace bsmma {
namespace {

// One block turns a 128-row x 32-block tile of plain scales into 8 consecutive
// atoms (4 KB): coalesced reads of the tile into shared memory, then each thread
// writes one 16-byte line of an atom (rows l, l+32, l+64, l+96; four blocks).
constexpr int kTileRows = 128, kTileBlocks = 32, kAtomsPerTile = kTileBlocks / 4;
constexpr int kRowPitch = kTileBlocks + 4;   // bytes; 9 words per row avoids bank conflicts

struct RelayoutJob {
  const uint8_t* src;
  uint8_t* dst;
  int64_t rows, kblocks, kg;   // kg = atoms per 128-row block of the output
  int64_t tiles_k;             // tiles along K
  int64_t tiles;               // total tiles (row blocks x tiles_k)
};

__device__ __forceinline__ void relayout_tile(const RelayoutJob& j, int64_t tile, uint8_t* sm) {
  const int64_t rb = tile / j.tiles_k, tk = tile - rb * j.tiles_k;
  const int t = threadIdx.x;
  {  // read: thread t takes 16 bytes of row t/2
    const int row = t >> 1, half = t & 1;
    const int64_t r = rb * kTileRows + row;
    const int64_t kb0 = tk * kTileBlocks + half * 16;
    uint8_t* d = sm + row * kRowPitch + half * 16;
    if (r < j.rows && kb0 + 16 <= j.kblocks && ((r * j.kblocks + kb0) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(j.src) & 15) == 0) {
      const uint4 v = *reinterpret_cast<const uint4*>(j.src + r * j.kblocks + kb0);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(d + 4 * i) = w[i];
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int64_t kb = kb0 + i;
        d[i] = (r < j.rows && kb < j.kblocks) ? j.src[r * j.kblocks + kb] : uint8_t(127);
      }
    }
  }
  __syncthreads();
  {  // write: thread t writes line t%32 of atom t/32
    const int a = t >> 5, line = t & 31;
    const int64_t kg = tk * kAtomsPerTile + a;
    if (kg < j.kg) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = *reinterpret_cast<const uint32_t*>(sm + (line + 32 * q) * kRowPitch + a * 4);
      *reinterpret_cast<uint4*>(j.dst + (rb * j.kg + kg) * 512 + line * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256) relayout_kernel(RelayoutJob j0, RelayoutJob j1) {
  __shared__ __align__(16) uint8_t sm[kTileRows * kRowPitch];
  const int64_t total = j0.tiles + j1.tiles;
  for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
    if (b < j0.tiles) relayout_tile(j0, b, sm);
    else relayout_tile(j1, b - j0.tiles, sm);
  }
}

RelayoutJob make_job(const uint8_t* s, int64_t rows, int64_t kb, uint8_t* out) {
  RelayoutJob j;
  j.src = s;
  j.dst = out;
  j.rows = rows;
  j.kblocks = kb;
  j.kg = 2 * ((kb + 7) / 8);
  const int64_t rblocks = 2 * ((rows + 255) / 256);
  j.tiles_k = (j.kg + kAtomsPerTile - 1) / kAtomsPerTile;
  j.tiles = (s && out && rows > 0 && kb > 0) ? rblocks * j.tiles_k : 0;
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
  const int64_t total = j0.tiles + j1.tiles;
  if (total == 0) return BSMMA_OK;
  const int64_t cap = static_cast<int64_t>(dev->sm_count) * 8;
  const int64_t blocks = total < cap ? total : cap;
  relayout_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(j0, j1);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace bsmma
