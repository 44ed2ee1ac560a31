// grouped_gemm.cu -- grouped groupwise FP8 GEMM for sm_103a.
//
// X [total_M][K] E4M3 with one FP32 scale per row per 128-K block (per-group block
// layout), W [G][N][K] E4M3 with one FP32 scale per 128x128 block, groups of uneven
// or zero size, BF16 output ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm":
// introduction; the commit that replaced the host tile map by in-kernel group
// resolution; the commit that fixed the activation-scale layout; Architecture
// support: FP32 scales applied in software per scale block).
//
// One persistent, warp-specialised launch, grid = #SMs at most:
//   every CTA reads m_sizes (int64, device memory), checks it (no negative entry,
//   sum == total_M; otherwise nothing is written and a status is latched) and
//   prefix-sums it into shared memory; a flat tile id -> (group, 128-row block of
//   that group, column block), in bands of row blocks walked along N.  Empty groups
//   own no tiles; no tile spans two groups; rows past a group's end are computed but
//   never stored.
//   warp 0      TMA producer: 128x128 X and W tiles into a 6-stage ring;
//   warp 1      lane 0 issues kind::f8f6f4 MMAs: each 128-K block goes into a fresh
//               FP32 partial in tensor memory (two partial slots, so the MMA of block
//               kb+1 overlaps the fold of block kb);
//   warps 2-3   idle (with warps 0-1 they form warpgroup 0, whose registers go to the fold)
//   warps 4-11  fold: acc += sX(row,kb) * sW(g,nblk,kb) * partial in FP32 registers
//               (packed two-lane FMAs; scales copied four blocks ahead into shared memory),
//               then BF16 round-to-nearest-even and masked 32-byte stores (16-byte ones
//               when D is only 16-byte aligned).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "grouped_sched.cuh"
#include "ptx.cuh"

namespace bsmma {
namespace {

using grouped::find_group;
using grouped::GroupTable;
using grouped::kBM;
using grouped::tile_coords;
constexpr int kBK = 128;
constexpr int kATileBytes = kBM * kBK;

// Tile 128 x BN; each of the 8 fold warps owns one 32-lane quarter x BN/2 columns.
template <int BN>
struct GCfg {
  static constexpr int kEpiWarps = 8;
  static constexpr int kFoldWarp0 = 4;        // warpgroup 0: producer, MMA issuer, two idle warps
  static constexpr int kCols = BN / 2;        // accumulator columns per fold warp
  static constexpr int kThreads = (kFoldWarp0 + kEpiWarps) * 32;
  // Registers: 384 threads launch with 168 each; warpgroup 0 then gives back down to 40
  // and the two fold warpgroups grow to 232 (128 x 40 + 256 x 232 = 384 x 168).
  static constexpr int kLaunchRegs = 168, kCtrlRegs = 40, kFoldRegs = 232;
  static constexpr int kBTileBytes = BN * kBK;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes;
  static constexpr int kStages = BN == 128 ? 6 : 4;
  static constexpr int kSlots = 512 / BN;         // partial slots in tensor memory (4 or 2)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kScaleAhead = 4;           // 128-K blocks of scales in flight per fold thread
  static constexpr int kScaleSlots = kScaleAhead + 1;
  static constexpr int kScaleRingBytes = kScaleSlots * 2 * kEpiWarps * 32 * 4;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 2048 + kScaleRingBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(128 * kCtrlRegs + 256 * kFoldRegs <= kThreads * kLaunchRegs, "register split");
};

struct GroupedParams {
  const float* sX;
  const float* sW;
  const uint8_t* Wp;    // packed weights (grouped_fp8_pack_weights layout), or null
  __nv_bfloat16* D;
  const int64_t* m_sizes;
  int64_t total_M, N;
  int G, num_n_tiles, num_kb;
  int d_align32;        // D is 32-byte aligned: rows are stored in 32-byte pieces
  uint32_t idesc;
  int* status;
  uint64_t limit_ns;
};

// 12 warps (three warpgroups) share an SM's four register-file quarters (16384
// registers each) three to a quarter, so a thread launches with at most
// 16384 / (3 * 32) = 170 registers (168 allocated); the warpgroups then rebalance.
// PACKED: W comes from the packed layout, one contiguous bulk copy per stage (the
// weight tile is stored exactly as the 128-byte-swizzled shared-memory image the MMA
// reads); otherwise a 2-D tensor copy from W [G*N][K].
template <int BN, bool PACKED>
__global__ void __launch_bounds__(384, 1)
    grouped_fp8_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const GroupedParams p) {
  using C = GCfg<BN>;
  constexpr int kStages = C::kStages, kStageBytes = C::kStageBytes, kEpiWarps = C::kEpiWarps;
  constexpr uint32_t kTmemCols = C::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  constexpr int kSlots = C::kSlots;
  uint64_t* p_full = empty + kStages;      // [kSlots]
  uint64_t* p_empty = p_full + kSlots;     // [kSlots]
  uint64_t* drain = p_empty + kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  GroupTable& gt = *reinterpret_cast<GroupTable*>(
      reinterpret_cast<uint8_t*>(full) + 512);
  // fold scales: [kScaleSlots][sX, sW][fold thread], filled by each fold thread's own
  // asynchronous copies
  float* scale_ring = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 2048);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  grouped::build_group_table(gt, p.m_sizes, G, p.total_M, p.status, [&] {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&p_full[s], 1);
      mbar_init(&p_empty[s], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  });
  if (gt.bad) return;   // uniform across the block; nothing allocated, nothing written

  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int NT = p.num_n_tiles, KB = p.num_kb;
  const int total_tiles = gt.tile_start[G] * NT;

  if (warp < C::kFoldWarp0) {
    setmaxnreg_dec<C::kCtrlRegs>();
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0, armed = 0, armed_parity = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
          int mt, nt;
          tile_coords(t, NT, gt.tile_start[G], mt, nt);
          const int g = find_group(gt, G, mt);
          const int row0 = static_cast<int>(gt.start[g] + static_cast<int64_t>(mt - gt.tile_start[g]) * kBM);
          const int wrow0 = static_cast<int>(static_cast<int64_t>(g) * p.N + static_cast<int64_t>(nt) * BN);
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, p.limit_ns, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            uint8_t* dst = ring + stage * kStageBytes;
            tma_load_2d(&tmX, &full[stage], dst, kb * kBK, row0);
            if constexpr (PACKED)
              bulk_load(dst + kATileBytes,
                        p.Wp + ((static_cast<int64_t>(g) * KB + kb) * (p.N / 128) + nt * (BN / 128)) *
                                   (128 * kBK),
                        C::kBTileBytes, &full[stage]);
            else
              tma_load_2d(&tmW, &full[stage], dst + kATileBytes, kb * kBK, wrow0);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        for (int s = 0; s < kStages; ++s)
          if (armed & (1u << s)) {
            volatile int no_abort = 0;
            mbar_wait(&full[s], (armed_parity >> s) & 1u, p.limit_ns / 4 + 1, &no_abort, nullptr);
          }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0, pcount = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
          for (int kb = 0; kb < KB; ++kb) {
            const uint32_t slot = pcount % kSlots;
            if (!mbar_wait(&full[stage], phase, p.limit_ns, abort_flag, p.status) ||
                !mbar_wait(&p_empty[slot], ((pcount / kSlots) & 1) ^ 1, p.limit_ns, abort_flag,
                           p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(ring + stage * kStageBytes);
            const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mma_f8f6f4(tmem + slot * BN, make_sdesc(a_base + j * 32, 16, 1024, kSwizzle128B),
                         make_sdesc(b_base + j * 32, 16, 1024, kSwizzle128B), p.idesc, j != 0);
            tc_commit(&empty[stage]);
            tc_commit(&p_full[slot]);
            ++pcount;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        tc_commit(drain);
        volatile int no_abort = 0;
        mbar_wait(drain, 0, p.limit_ns, &no_abort, nullptr);
      }
    }
    // both warpgroups meet once every MMA and tensor-memory read has been issued and fenced
    named_barrier_sync(1, C::kThreads);
    if (warp == 1) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }
  setmaxnreg_inc<C::kFoldRegs>();
  {
    // -------------------------------------------------------------- fold + epilogue
    constexpr int kCols = C::kCols;
    const int q = warp & 3;           // tensor-memory lane quarter
    const int h = (warp - C::kFoldWarp0) >> 2;    // which half of the tile's columns
    uint32_t pcount = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
      int mt, nt;
      tile_coords(t, NT, gt.tile_start[G], mt, nt);
      const int g = find_group(gt, G, mt);
      const int64_t m_g = gt.size[g];
      const int64_t l = static_cast<int64_t>(mt - gt.tile_start[g]) * kBM + q * 32 + lane;
      const bool valid = l < m_g;
      // a warp whose 32 rows all lie past the group's end folds nothing (it still
      // takes part in the partial-slot handshake)
      const bool warp_rows = static_cast<int64_t>(mt - gt.tile_start[g]) * kBM + q * 32 < m_g;
      const float* sx = p.sX + gt.start[g] * KB + l;   // + kb * m_g
      // weight scale of the 128-column block of this warp's columns
      static_assert(kCols <= 128, "a fold warp's columns lie in one 128-column scale block");
      const float* sw = p.sW + (static_cast<int64_t>(g) * (p.N / 128) +
                                static_cast<int64_t>(nt) * (BN / 128) + (h * kCols) / 128) * KB;
      // FP32 accumulators in pairs: one packed two-lane FMA (fma.rn.f32x2) per pair,
      // rounding each lane exactly as a scalar fmaf would
      float2 acc[kCols / 2];
#pragma unroll
      for (int i = 0; i < kCols / 2; ++i) acc[i] = make_float2(0.f, 0.f);
      // The scales of block kb are copied kScaleAhead blocks ahead of their use, one
      // commit group per block (empty past the last block), so that with all but the
      // newest kScaleAhead - 1 groups complete block kb has landed.  Block kb+kScaleAhead
      // goes to the slot read in the previous iteration, never the one being read.
      constexpr int kFoldThreads = kEpiWarps * 32;
      float* ring = scale_ring + (threadIdx.x - C::kFoldWarp0 * 32);
      // streaming source pointers: row scale of block kb at sx + kb*m_g (not read for rows
      // past the group's end), weight scale at sw + kb
      const float* sx_next = valid ? sx : p.sX;
      const int64_t sx_step = valid ? m_g : 0;
      const float* sw_next = sw;
      int fetched = 0;
      auto fetch = [&]() {
        if (fetched < KB) {
          float* dst = ring + (fetched % C::kScaleSlots) * 2 * kFoldThreads;
          cp_async_4(dst, sx_next, valid ? 4u : 0u);
          cp_async_4(dst + kFoldThreads, sw_next, 4u);
          sx_next += sx_step;
          ++sw_next;
        }
        ++fetched;
        cp_async_commit();
      };
#pragma unroll
      for (int d = 0; d < C::kScaleAhead; ++d) fetch();
      int rd = 0;   // ring slot of block kb
      for (int kb = 0; kb < KB; ++kb) {
        cp_async_wait<C::kScaleAhead - 1>();
        const float* cur = ring + rd * 2 * kFoldThreads;
        rd = rd + 1 == C::kScaleSlots ? 0 : rd + 1;
        const float s = cur[0] * cur[kFoldThreads];
        fetch();
        const uint32_t slot = pcount % kSlots;
        if (!mbar_wait(&p_full[slot], (pcount / kSlots) & 1, p.limit_ns, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem + (static_cast<uint32_t>(q * 32) << 16) + slot * BN + h * kCols;
        if (!warp_rows) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_empty[slot]);
          ++pcount;
          continue;
        }
        const float2 s2 = make_float2(s, s);
        if constexpr (kCols == 64) {
          // the whole 64-column slice in one round trip; the slot is released before the FMAs
          uint32_t r0[32], r1[32];
          tmem_ld32(taddr, r0);
          tmem_ld32(taddr + 32, r1);
          tmem_ld_wait(r0);
          reg_fence(r1);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_empty[slot]);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[i] = __ffma2_rn(s2, make_float2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1])), acc[i]);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[16 + i] = __ffma2_rn(s2, make_float2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1])),
                                     acc[16 + i]);
        } else {
          // 128 columns in 32-column pieces, software-pipelined: the load of piece c+1
          // is in flight while piece c is folded
          uint32_t ra[32], rb[32];
          tmem_ld32(taddr, ra);
          tmem_ld_wait(ra);
#pragma unroll
          for (int c = 0; c < kCols / 32; c += 2) {
            tmem_ld32(taddr + (c + 1) * 32, rb);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              acc[c * 16 + i] = __ffma2_rn(s2, make_float2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])),
                                           acc[c * 16 + i]);
            tmem_ld_wait(rb);
            if (c + 2 < kCols / 32) tmem_ld32(taddr + (c + 2) * 32, ra);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              acc[(c + 1) * 16 + i] = __ffma2_rn(s2, make_float2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1])),
                                                 acc[(c + 1) * 16 + i]);
            if (c + 2 < kCols / 32) tmem_ld_wait(ra);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_empty[slot]);
        }
        ++pcount;
      }
      if (!ok) break;
      if (valid) {
        // the fold warps' stores hold up the next tile's fold (and, two partial slots on, the
        // MMAs), so they go out in as few instructions as the alignment allows: a full
        // 32-byte sector per lane (rows are N*2 bytes, a multiple of 256)
        const int64_t row = gt.start[g] + l;
        __nv_bfloat16* out = p.D + row * p.N + static_cast<int64_t>(nt) * BN + h * kCols;
        if (p.d_align32) {
#pragma unroll
          for (int v = 0; v < kCols / 16; ++v)
            st_global_v8_cs(out + v * 16, pack_bf16x2(acc[v * 8 + 0].x, acc[v * 8 + 0].y),
                            pack_bf16x2(acc[v * 8 + 1].x, acc[v * 8 + 1].y),
                            pack_bf16x2(acc[v * 8 + 2].x, acc[v * 8 + 2].y),
                            pack_bf16x2(acc[v * 8 + 3].x, acc[v * 8 + 3].y),
                            pack_bf16x2(acc[v * 8 + 4].x, acc[v * 8 + 4].y),
                            pack_bf16x2(acc[v * 8 + 5].x, acc[v * 8 + 5].y),
                            pack_bf16x2(acc[v * 8 + 6].x, acc[v * 8 + 6].y),
                            pack_bf16x2(acc[v * 8 + 7].x, acc[v * 8 + 7].y));
        } else {
#pragma unroll
          for (int v = 0; v < kCols / 8; ++v)
            st_global_v4_cs(out + v * 8, pack_bf16x2(acc[v * 4 + 0].x, acc[v * 4 + 0].y),
                            pack_bf16x2(acc[v * 4 + 1].x, acc[v * 4 + 1].y),
                            pack_bf16x2(acc[v * 4 + 2].x, acc[v * 4 + 2].y),
                            pack_bf16x2(acc[v * 4 + 3].x, acc[v * 4 + 3].y));
        }
      }
    }
    cp_async_wait_all();   // no scale copy may land after the block has finished
  }
  tc_fence_before();
  named_barrier_sync(1, C::kThreads);
}

template <int BN, bool PACKED>
bsmma_status launch_grouped_bn(const CUtensorMap& tx, const CUtensorMap& tw, GroupedParams p,
                               int64_t total_M, int G, int sm_count, cudaStream_t stream) {
  using C = GCfg<BN>;
  p.num_n_tiles = static_cast<int>(p.N / BN);
  p.idesc = idesc_f8f6f4(0, 0, 0, 0, kBM, BN);
  const int64_t bound = ((total_M + kBM - 1) / kBM + G) * p.num_n_tiles;
  int64_t grid = bound < sm_count ? bound : sm_count;
  if (grid < 1) grid = 1;
  static bool attr_set = false;   // benign race: setting the attribute twice is harmless
  if (!attr_set) {
    if (cudaFuncSetAttribute(grouped_fp8_kernel<BN, PACKED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return BSMMA_ERR_CUDA;
    attr_set = true;
  }
  grouped_fp8_kernel<BN, PACKED><<<static_cast<int>(grid), C::kThreads, C::kSmemBytes, stream>>>(tx, tw, p);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace

namespace {
bsmma_status launch_grouped_width(const uint8_t* X, const float* sX, const uint8_t* W,
                                  const float* sW, void* D, const int64_t* m_sizes, int64_t total_M,
                                  int G, int64_t N, int64_t K, int bn, bool packed,
                                  const DeviceInfo* dev, cudaStream_t stream);

// Packed weight layout: for group g, 128-K block kb and 128-row block nb of W, one
// 16 KB block at ((g*KB + kb)*NB + nb) * 16384 holding rows nb*128 .. nb*128+127, 128
// bytes of K each, with the 16-byte pieces of row r stored in the order that the
// 128-byte swizzle of a shared-memory tile uses (piece c at position c ^ (r % 8)).  Two
// neighbouring 128-row blocks of one K block are contiguous, so a 128- or 256-row tile
// is one contiguous copy whose bytes land in shared memory exactly as the MMA reads them.
__global__ void pack_weights_kernel(const uint4* __restrict__ W, uint4* __restrict__ Wp, int64_t G,
                                    int64_t N, int64_t K) {
  const int64_t pieces_per_row = K / 16;
  const int64_t total = G * N * pieces_per_row;
  const int64_t KB = K / 128, NB = N / 128;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / pieces_per_row;          // g*N + n
    const int64_t piece = i - row * pieces_per_row;  // 16-byte piece of the row
    const int64_t g = row / N, n = row - g * N;
    const int64_t kb = piece / 8, c = piece % 8;
    const int64_t nb = n / 128, r = n % 128;
    const int64_t dst = ((g * KB + kb) * NB + nb) * 1024 + r * 8 + (c ^ (r % 8));
    Wp[dst] = W[i];
  }
}
}  // namespace

bsmma_status launch_pack_weights(const uint8_t* W, int64_t G, int64_t N, int64_t K, uint8_t* Wp,
                                 cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  pack_weights_kernel<<<dev->sm_count * 8, 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(W), reinterpret_cast<uint4*>(Wp), G, N, K);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

bsmma_status launch_grouped(const uint8_t* X, const float* sX, const uint8_t* W, const float* sW,
                            void* D, const int64_t* m_sizes, int64_t total_M, int G, int64_t N,
                            int64_t K, cudaStream_t stream, bool packed) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  static_assert(sizeof(GroupTable) + 512 <= 2048, "group table fits its shared-memory slot");
  // A 128x128 MMA takes as long as a 128x256 one, so wide tiles do the same work in half
  // the MMA time and read W half as often per flop; they lose only when so few tiles
  // remain that too few SMs stream W.  The row-block count is estimated from total_M
  // (the sizes are on the device): each group adds on average half a partial block.
  const int64_t row_blocks_est = (total_M + kBM - 1) / kBM + G / 2;
  const bool wide = (N % 256 == 0) &&
                    row_blocks_est * (N / 256) * 2 >= static_cast<int64_t>(dev->sm_count) &&
                    grouped_tile_width() != 128;
  const bool force_wide = grouped_tile_width() == 256 && N % 256 == 0;
  int bn = (wide || force_wide) ? 256 : 128;
  if (grouped_tile_width() == 0 && N % 256 == 0) {
    // opt-in autotuning per (nextPow2(total_M), N, K, G)
    const std::string key = std::string(packed ? "grouped_packed " : "grouped ") +
                            std::to_string(next_pow2(total_M)) + " " + std::to_string(N) + " " +
                            std::to_string(K) + " " + std::to_string(G);
    bn = autotune_pick(key, {256, 128}, bn, stream, [&](int c) {
      return launch_grouped_width(X, sX, W, sW, D, m_sizes, total_M, G, N, K, c, packed, dev,
                                  stream);
    });
  }
  return launch_grouped_width(X, sX, W, sW, D, m_sizes, total_M, G, N, K, bn, packed, dev, stream);
}

namespace {
bsmma_status launch_grouped_width(const uint8_t* X, const float* sX, const uint8_t* W,
                                  const float* sW, void* D, const int64_t* m_sizes, int64_t total_M,
                                  int G, int64_t N, int64_t K, int bn, bool packed,
                                  const DeviceInfo* dev, cudaStream_t stream) {
  bsmma_status st;
  CUtensorMap tx, tw;
  // With no rows there is no X tile to load; W's address stands in for the map.
  st = encode_tmap_u8(&tx, total_M > 0 ? static_cast<const void*>(X) : W, K,
                      total_M > 0 ? total_M : 1, K, 128, 128);
  if (st != BSMMA_OK) return st;
  st = encode_tmap_u8(&tw, W, K, static_cast<uint64_t>(G) * N, K, 128, bn);
  if (st != BSMMA_OK) return st;
  GroupedParams p;
  p.sX = sX;
  p.sW = sW;
  p.Wp = packed ? W : nullptr;
  p.D = static_cast<__nv_bfloat16*>(D);
  p.d_align32 = (reinterpret_cast<uintptr_t>(D) & 31u) == 0;
  p.m_sizes = m_sizes;
  p.total_M = total_M;
  p.N = N;
  p.G = G;
  p.num_kb = static_cast<int>(K / kBK);
  p.status = dev->status;
  p.limit_ns = wait_limit_ns();
  if (packed) {
    if (bn == 256) return launch_grouped_bn<256, true>(tx, tw, p, total_M, G, dev->sm_count, stream);
    return launch_grouped_bn<128, true>(tx, tw, p, total_M, G, dev->sm_count, stream);
  }
  if (bn == 256) return launch_grouped_bn<256, false>(tx, tw, p, total_M, G, dev->sm_count, stream);
  return launch_grouped_bn<128, false>(tx, tw, p, total_M, G, dev->sm_count, stream);
}
}  // namespace

}  // namespace bsmma
