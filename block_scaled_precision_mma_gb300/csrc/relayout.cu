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

// ---------------------------------------------------------------------------
// Wide scale layouts for the SM-pair kernel, read by tcgen05.cp 128x256b copies.
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
// Column scales (the B side): one 1 KB block per 256 columns and one K-group,
// 32 lanes x 8 columns: lane i, column c holds the four scales of column 32c+i.
// Block (nb, kg) sits at (nb*KGp + kg)*1024, bytes ordered like lanes 0-31 above.
// Padding holds 127 (scale 1.0).
namespace bsmma {
namespace {

__device__ __forceinline__ uint32_t gather4(const uint8_t* s, int64_t rows, int64_t kblocks,
                                            int64_t r, int64_t kb0) {
  uint32_t v = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int64_t kb = kb0 + b;
    const uint32_t x = (r < rows && kb < kblocks) ? s[r * kblocks + kb] : 127u;
    v |= x << (8 * b);
  }
  return v;
}

struct WideJob {
  const uint8_t* src;
  uint8_t* dst;
  int64_t rows, kblocks;
  int64_t per_block;   // chunks (row role: KQ) or blocks (column role: KGp) per row block
  int64_t words;       // output words
  int role;            // 0 row scales, 1 column scales
};

__device__ __forceinline__ void wide_word(const WideJob& j, int64_t w) {
  uint32_t v;
  if (j.role == 0) {
    const int64_t chunk = w >> 10;                 // 1024 words per 4 KB chunk
    const int wi = static_cast<int>(w & 1023);
    const int64_t rb = chunk / j.per_block, kq = chunk - rb * j.per_block;
    const int byte = wi * 4;
    const int lg = byte >> 8, ch = (byte >> 7) & 1, l8 = (byte >> 4) & 7, c4 = (byte >> 2) & 3;
    const int l = lg * 8 + l8, c = ch * 4 + c4, q = l >> 5;
    v = (c4 == q) ? gather4(j.src, j.rows, j.kblocks, rb * 128 + l, (kq * 2 + ch) * 4)
                  : 0x7f7f7f7fu;
  } else {
    const int64_t blk = w >> 8;                    // 256 words per 1 KB block
    const int wi = static_cast<int>(w & 255);
    const int64_t nb = blk / j.per_block, kg = blk - nb * j.per_block;
    const int byte = wi * 4;
    const int lg = byte >> 8, ch = (byte >> 7) & 1, l8 = (byte >> 4) & 7, c4 = (byte >> 2) & 3;
    const int i = lg * 8 + l8, c = ch * 4 + c4;
    v = gather4(j.src, j.rows, j.kblocks, nb * 256 + 32 * c + i, kg * 4);
  }
  reinterpret_cast<uint32_t*>(j.dst)[w] = v;
}

__global__ void __launch_bounds__(256) wide_relayout_kernel(WideJob j0, WideJob j1) {
  const int64_t total = j0.words + j1.words;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (w < j0.words) wide_word(j0, w);
    else wide_word(j1, w - j0.words);
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
  j.words = (s && out && rows > 0 && kb > 0) ? wide_scale_bytes(rows, kb, role) / 4 : 0;
  return j;
}

}  // namespace

int64_t wide_scale_bytes(int64_t rows, int64_t kblocks, int role) {
  if (rows <= 0 || kblocks <= 0) return 0;
  if (role == 0) return 2 * ((rows + 255) / 256) * ((kblocks + 7) / 8) * 4096;
  return ((rows + 255) / 256) * 2 * ((kblocks + 7) / 8) * 1024;
}

bsmma_status launch_wide_relayout(const uint8_t* sa, int64_t rows_a, uint8_t* out_a,
                                  const uint8_t* sb, int64_t rows_b, uint8_t* out_b,
                                  int64_t kblocks, cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  WideJob j0 = make_wide(sa, rows_a, kblocks, out_a, 0), j1 = make_wide(sb, rows_b, kblocks, out_b, 1);
  const int64_t total = j0.words + j1.words;
  if (total == 0) return BSMMA_OK;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(dev->sm_count) * 8;
  if (blocks > cap) blocks = cap;
  wide_relayout_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(j0, j1);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace bsmma
