// relayout.cu -- plain E8M0 scales [rows][kblocks] -> the GEMM kernels' tiled layouts.
//
// The GEMM takes plain scales and rearranges them itself ("[gfx1250] Add MXFP4
// GEMM support to FlyDSL backend", Description: plain scales in, shuffled inside
// the backend).  On sm_103a the target is what a 128-lane x 32-byte tcgen05.cp copy
// puts into tensor memory for the block-scaled MMAs.  One launch handles the scales
// of both operands of a GEMM.
#include <cuda_runtime.h>

#include "internal.h"

//
// Row scales (the A side): one 4 KB chunk per 128 rows and 8 K-blocks (two K groups),
// holding for TMEM lane l (row l of the block, lane quarter q = l/32) in column
// c = 4g + q the four scales of row l for K group g of the chunk (other columns are
// padding).  An MMA for K group g names column base + 4g (scale addresses are
// 4-column aligned) and lane quarter q reads its own column base + 4g + q.  Chunk
// (rb, kq) sits at (rb*KQ + kq)*4096 and its bytes are in the order the copy's
// source descriptor walks (8-row groups of 256 bytes, two 16-byte column halves of
// 128 bytes each):
//   byte(l, c, b) = (l/8)*256 + (c/4)*128 + (l%8)*16 + (c%4)*4 + b.
// Column scales (the B side): one 4 KB block per 256 columns and one K group, made
// of four identical 1 KB quarters (every lane quarter of tensor memory needs all
// of them): in each, lane i, column c holds the four scales of column 32c+i.
// Block (nb, kg) sits at (nb*KGp + kg)*4096, bytes ordered like lanes 0-31 above.
// Padding holds 127 (scale 1.0).
namespace bsmma {
namespace {

// One block rearranges one input tile staged in shared memory with coalesced 16-byte
// reads, then writes 16 KB of output with coalesced 16-byte stores:
//   row role: 128 rows x 32 K-blocks -> 4 chunks (each 128 rows x 8 K-blocks);
//   column role: 256 rows x 16 K-blocks -> 4 blocks (each 256 rows x 4 K-blocks).
// Every input tile is 4 KB; rows are padded by 4 bytes in shared memory.
constexpr int kPitchA = 32 + 4;    // bytes per staged row, row role
constexpr int kPitchB = 16 + 4;    // bytes per staged row, column role

struct WideJob {
  const uint8_t* src;
  uint8_t* dst;
  int64_t rows, kblocks;
  int64_t per_block;   // chunks (row role) or blocks (column role) per row block
  int64_t tiles_k;     // input tiles along K per row block
  int64_t tiles;       // input tiles in total
  int role;            // 0 row scales, 1 column scales
};

// Stages rows [r0, r0+nrows) x K-blocks [kb0, kb0+nk) of the plain scales (127 where
// outside the tensor) into sm with the given pitch.
__device__ __forceinline__ void stage_tile(const WideJob& j, uint8_t* sm, int pitch, int64_t r0,
                                           int nrows, int64_t kb0, int nk) {
  const int per_row = nk / 16;                       // 16-byte pieces per row
  for (int t = threadIdx.x; t < nrows * per_row; t += blockDim.x) {
    const int row = t / per_row, piece = t - row * per_row;
    const int64_t r = r0 + row, kb = kb0 + piece * 16;
    uint8_t* d = sm + row * pitch + piece * 16;
    if (r < j.rows && kb + 16 <= j.kblocks && ((r * j.kblocks + kb) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(j.src) & 15) == 0) {
      const uint4 v = *reinterpret_cast<const uint4*>(j.src + r * j.kblocks + kb);
      reinterpret_cast<uint32_t*>(d)[0] = v.x;
      reinterpret_cast<uint32_t*>(d)[1] = v.y;
      reinterpret_cast<uint32_t*>(d)[2] = v.z;
      reinterpret_cast<uint32_t*>(d)[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        d[i] = (r < j.rows && kb + i < j.kblocks) ? j.src[r * j.kblocks + kb + i] : uint8_t(127);
    }
  }
}

__device__ __forceinline__ uint32_t word_at(const uint8_t* sm, int pitch, int row, int byte) {
  return *reinterpret_cast<const uint32_t*>(sm + row * pitch + byte);
}

__device__ void wide_tile(const WideJob& j, int64_t tile, uint8_t* sm) {
  const int64_t rb = tile / j.tiles_k, tk = tile - rb * j.tiles_k;
  if (j.role == 0) {
    stage_tile(j, sm, kPitchA, rb * 128, 128, tk * 32, 32);
    __syncthreads();
    // 4 chunks x 256 vectors of 16 bytes; vector v of a chunk holds lane l's columns
    // 4*ch .. 4*ch+3, of which only column 4*ch + l/32 carries data
    for (int t = threadIdx.x; t < 4 * 256; t += blockDim.x) {
      const int cidx = t >> 8, v = t & 255;
      const int64_t kq = tk * 4 + cidx;
      if (kq >= j.per_block) continue;
      const int lg = v >> 4, ch = (v >> 3) & 1, l8 = v & 7;
      const int l = lg * 8 + l8, q = l >> 5;
      uint32_t w[4] = {0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu};
      w[q] = word_at(sm, kPitchA, l, (cidx * 2 + ch) * 4);
      *reinterpret_cast<uint4*>(j.dst + (rb * j.per_block + kq) * 4096 + v * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    stage_tile(j, sm, kPitchB, rb * 256, 256, tk * 16, 16);
    __syncthreads();
    // 4 blocks x 4 lane-quarter copies x 64 vectors; vector v holds lane i's columns
    // 4*ch .. 4*ch+3, i.e. rows 32c + i
    for (int t = threadIdx.x; t < 4 * 256; t += blockDim.x) {
      const int bidx = t >> 8, v = t & 63, copy = (t >> 6) & 3;
      const int64_t kg = tk * 4 + bidx;
      if (kg >= j.per_block) continue;
      const int lg = v >> 4, ch = (v >> 3) & 1, l8 = v & 7;
      const int i = lg * 8 + l8;
      uint32_t w[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) w[c4] = word_at(sm, kPitchB, 32 * (ch * 4 + c4) + i, bidx * 4);
      *reinterpret_cast<uint4*>(j.dst + (rb * j.per_block + kg) * 4096 + copy * 1024 + v * 16) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256) wide_relayout_kernel(WideJob j0, WideJob j1) {
  __shared__ __align__(16) uint8_t sm[256 * kPitchB > 128 * kPitchA ? 256 * kPitchB : 128 * kPitchA];
  const int64_t total = j0.tiles + j1.tiles;
  for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
    if (b < j0.tiles) wide_tile(j0, b, sm);
    else wide_tile(j1, b - j0.tiles, sm);
  }
}

WideJob make_wide(const uint8_t* s, int64_t rows, int64_t kb, uint8_t* out, int role) {
  WideJob j;
  j.src = s;
  j.dst = out;
  j.rows = rows;
  j.kblocks = kb;
  j.role = role;
  j.per_block = role == 0 ? (kb + 7) / 8 : 2 * ((kb + 7) / 8);
  const int64_t row_blocks = role == 0 ? 2 * ((rows + 255) / 256) : (rows + 255) / 256;
  j.tiles_k = (j.per_block + 3) / 4;
  j.tiles = (s && out && rows > 0 && kb > 0) ? row_blocks * j.tiles_k : 0;
  return j;
}

}  // namespace

int64_t wide_scale_bytes(int64_t rows, int64_t kblocks, int role) {
  if (rows <= 0 || kblocks <= 0) return 0;
  if (role == 0) return 2 * ((rows + 255) / 256) * ((kblocks + 7) / 8) * 4096;
  return ((rows + 255) / 256) * 2 * ((kblocks + 7) / 8) * 4096;
}

bsmma_status launch_wide_relayout(const uint8_t* sa, int64_t rows_a, uint8_t* out_a,
                                  const uint8_t* sb, int64_t rows_b, uint8_t* out_b,
                                  int64_t kblocks, cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  WideJob j0 = make_wide(sa, rows_a, kblocks, out_a, 0), j1 = make_wide(sb, rows_b, kblocks, out_b, 1);
  const int64_t total = j0.tiles + j1.tiles;
  if (total == 0) return BSMMA_OK;
  const int64_t cap = static_cast<int64_t>(dev->sm_count) * 8;
  const int64_t blocks = total < cap ? total : cap;
  wide_relayout_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(j0, j1);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace bsmma
