// grouped_bf16.cu -- grouped BF16 GEMM for sm_103a.
//
// X [total_M][K] BF16, W [G][N][K] BF16, groups of uneven or zero size (m_sizes on the
// device), BF16 output D[r] = X[r] . W[g(r)]^T with FP32 accumulation ("PyTorch on AMD
// GPUs gains a FlyDSL backend", Interpretation: grouped GEMM over uneven and empty
// expert groups, the BF16 grouped-GEMM cases).  No scales: the tensor core accumulates
// the whole of K in tensor memory.
//
// One persistent, warp-specialised launch, grid = #SMs at most, tiles of 128 rows x BN
// columns in the grouped tile order (grouped_sched.cuh):
//   warp 0      TMA producer: 128 x 64 X and BN x 64 W tiles (128-byte rows, 128-byte
//               swizzle) into a ring of stages;
//   warp 1      lane 0 issues kind::f16 MMAs (M=128, N=BN, K=16; four per stage) into
//               one of two FP32 accumulators in tensor memory, so that a tile's output
//               stage overlaps the next tile's main loop;
//   warps 2-9   output stage: two warps per 32-lane quarter, each reading half of the
//               tile's columns with tcgen05.ld, rounding to BF16 (nearest-even) and
//               storing 16 bytes per lane, only rows of the tile's group and columns
//               below N.
// Groups of many rows go instead to grouped_bf16_pair_kernel: the same roles on 256 x 256
// tiles spread over the two CTAs of a cluster (an SM pair), whose M = 256 MMAs read a third
// less shared memory per flop.
// K need only be a multiple of 8 (16-byte rows): the last stage's columns past K are
// filled with zeros by the tensor copy.  N need only be a multiple of 8: columns of the
// last column block past N are computed from whatever rows the copy returns (the next
// group's weights, or zeros past the tensor) and never stored.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "grouped_sched.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace bsmma {
namespace {

using grouped::find_group;
using grouped::GroupTable;
using grouped::kBM;
using grouped::tile_coords;
constexpr int kBKBytes = 128;                 // one 128-byte swizzle row: 64 BF16 of K
constexpr int kATileBytes = kBM * kBKBytes;   // 16 KB

// Instruction descriptor of kind::f16: FP32 accumulator, BF16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D(tmem) (+)= A(smem) x B(smem), BF16 operands, FP32 accumulation.
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// The same over an SM pair: M = 256 (128 rows of A in each CTA's shared memory at the same
// offset), N split in two halves of B likewise, each CTA's tensor memory receiving its
// 128 rows x N.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

template <int BN>
struct BCfg {
  static constexpr int kOutWarps = 8;
  static constexpr int kOutWarp0 = 2;
  static constexpr int kThreads = (kOutWarp0 + kOutWarps) * 32;
  static constexpr int kCols = BN / 2;             // accumulator columns per output warp
  static constexpr int kBTileBytes = BN * kBKBytes;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes;
  static constexpr int kStages = BN == 128 ? 6 : 4;
  static constexpr uint32_t kTmemCols = 2 * BN;    // two accumulators
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 2048;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Bf16Params {
  __nv_bfloat16* D;
  const int64_t* m_sizes;
  int64_t total_M, N;
  int G, num_n_tiles, num_kb;
  int d_align32;        // D 32-byte aligned and N % 16 == 0: rows stored in 32-byte pieces
  uint32_t idesc;
  int* status;
  uint64_t limit_ns;
};

// 32 columns of this lane's row (x: 32 FP32 values from tcgen05.ld), rounded to BF16 and
// stored with streaming stores, columns at or past N skipped: 32-byte pieces (a full sector
// per lane) when D is 32-byte aligned and N % 16 == 0, else 16-byte pieces.
__device__ __forceinline__ void store32(__nv_bfloat16* out, int64_t col0, int c, const uint32_t* x,
                                        const Bf16Params& p) {
  auto pk = [&](int i) {
    return pack_bf16x2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
  };
  if (p.d_align32) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (col0 + c * 32 + e * 16 < p.N)
        st_global_v8_cs(out + c * 32 + e * 16, pk(8 * e), pk(8 * e + 1), pk(8 * e + 2), pk(8 * e + 3),
                        pk(8 * e + 4), pk(8 * e + 5), pk(8 * e + 6), pk(8 * e + 7));
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (col0 + c * 32 + e * 8 < p.N)
        st_global_v4_cs(out + c * 32 + e * 8, pk(4 * e), pk(4 * e + 1), pk(4 * e + 2), pk(4 * e + 3));
  }
}

template <int BN>
__global__ void __launch_bounds__(BCfg<BN>::kThreads, 1)
    grouped_bf16_kernel(const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW, const Bf16Params p) {
  using C = BCfg<BN>;
  constexpr int kStages = C::kStages, kStageBytes = C::kStageBytes, kOutWarps = C::kOutWarps;
  constexpr uint32_t kTmemCols = C::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;    // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  GroupTable& gt = *reinterpret_cast<GroupTable*>(reinterpret_cast<uint8_t*>(full) + 512);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  grouped::build_group_table(gt, p.m_sizes, G, p.total_M, p.status, [&] {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kOutWarps);
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

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------------- producer
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
          tma_load_2d(&tmX, &full[stage], dst, kb * kBKBytes, row0);
          tma_load_2d(&tmW, &full[stage], dst + kATileBytes, kb * kBKBytes, wrow0);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // no copy may land after the block has finished
      for (int s = 0; s < kStages; ++s)
        if (armed & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait(&full[s], (armed_parity >> s) & 1u, p.limit_ns / 4 + 1, &no_abort, nullptr);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0, tcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, ++tcount) {
        const uint32_t buf = tcount & 1;
        if (!mbar_wait(&acc_empty[buf], ((tcount >> 1) & 1) ^ 1, p.limit_ns, abort_flag,
                       p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(ring + stage * kStageBytes);
          const uint32_t b_base = a_base + kATileBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_bf16(d, make_sdesc(a_base + j * 32, 16, 1024, kSwizzle128B),
                     make_sdesc(b_base + j * 32, 16, 1024, kSwizzle128B), p.idesc,
                     (kb | j) != 0);
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, p.limit_ns, &no_abort, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- output stage
    constexpr int kCols = C::kCols, kPieces = kCols / 32;
    const int q = warp & 3;                            // tensor-memory lane quarter
    const int h = (warp - C::kOutWarp0) >> 2;          // which half of the tile's columns
    uint32_t tcount = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++tcount) {
      int mt, nt;
      tile_coords(t, NT, gt.tile_start[G], mt, nt);
      const int g = find_group(gt, G, mt);
      const int64_t l = static_cast<int64_t>(mt - gt.tile_start[g]) * kBM + q * 32 + lane;
      const bool valid = l < gt.size[g];
      const uint32_t buf = tcount & 1;
      if (!mbar_wait(&acc_full[buf], (tcount >> 1) & 1, p.limit_ns, abort_flag, p.status)) break;
      tc_fence_after();
      // 32-column pieces of 32 lanes x 32 values (tcgen05.ld.32x32b), two in flight; the
      // accumulator is released after the warp's last load
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + h * kCols;
      const int64_t col0 = static_cast<int64_t>(nt) * BN + h * kCols;
      __nv_bfloat16* out = p.D + (gt.start[g] + l) * p.N + col0;
      auto store_piece = [&](int c, const uint32_t* x) { store32(out, col0, c, x, p); };
#pragma unroll
      for (int c = 0; c < kPieces; c += 2) {
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c * 32, ra);
        tmem_ld32(taddr + (c + 1) * 32, rb);
        tmem_ld_wait(ra);
        reg_fence(rb);
        if (c + 2 == kPieces) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (valid) {
          store_piece(c, ra);
          store_piece(c + 1, rb);
        }
      }
    }
  }
  // every MMA and tensor-memory read has been issued and fenced
  tc_fence_before();
  named_barrier_sync(1, C::kThreads);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// SM-pair tiles of 256 rows x 256 columns: a 2-CTA cluster, CTA r loading rows r*128 ..
// r*128+127 of the tile's X rows and of its W columns, the leader issuing M = 256 MMAs
// that read both CTAs' shared memory.  Per SM a stage moves 32 KB (16 KB of X, 16 KB of W)
// and the MMAs read 8 KB per K = 16 step from each CTA, against 48 KB and 12 KB for a
// one-CTA 128 x 256 tile: shared memory, the limit of the one-CTA tile at large M, carries
// a third less per flop.  Row blocks are 256 rows of one group.
struct PCfg {
  static constexpr int kOutWarps = 8;
  static constexpr int kOutWarp0 = 2;
  static constexpr int kThreads = (kOutWarp0 + kOutWarps) * 32;
  static constexpr int kHalfBytes = 128 * kBKBytes;        // 128 rows x 64 BF16 of K
  static constexpr int kStageBytes = 2 * kHalfBytes;       // this CTA's X half and W half
  static constexpr int kStages = 6;
  static constexpr uint32_t kTmemCols = 512;               // two 256-column accumulators
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 2048;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert((2 * kStages + 5) * 8 + 8 <= 512, "barriers fit below the group table");
};

__global__ void __launch_bounds__(PCfg::kThreads, 1)
    grouped_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmX,
                             const __grid_constant__ CUtensorMap tmW, const Bf16Params p) {
  using C = PCfg;
  constexpr int kStages = C::kStages, kStageBytes = C::kStageBytes, kOutWarps = C::kOutWarps;
  constexpr int BN = 256;
  constexpr uint16_t kPairMask = 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;    // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2], used in the leader
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  GroupTable& gt = *reinterpret_cast<GroupTable*>(reinterpret_cast<uint8_t*>(full) + 512);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int G = p.G;
  grouped::build_group_table<256>(gt, p.m_sizes, G, p.total_M, p.status, [&] {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);     // used in the leader: its producer's arrive + both CTAs' bytes
      mbar_init(&empty[s], 1);    // released by the leader's commit in both CTAs
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 2 * kOutWarps);   // output warps of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  });
  // both CTAs read the same m_sizes, so a bad table stops the whole cluster here, before
  // anything is allocated or waited for
  if (gt.bad) return;

  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int NT = p.num_n_tiles, KB = p.num_kb;
  const int total_tiles = gt.tile_start[G] * NT;
  const int cluster_id = static_cast<int>(blockIdx.x >> 1);
  const int clusters = static_cast<int>(gridDim.x >> 1);

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------------- producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int t = cluster_id; ok && t < total_tiles; t += clusters) {
        int mt, nt;
        tile_coords(t, NT, gt.tile_start[G], mt, nt);
        const int g = find_group(gt, G, mt);
        const int row0 = static_cast<int>(gt.start[g] + static_cast<int64_t>(mt - gt.tile_start[g]) * 256 +
                                          128 * static_cast<int>(rank));
        const int wrow0 = static_cast<int>(static_cast<int64_t>(g) * p.N + static_cast<int64_t>(nt) * BN +
                                           128 * static_cast<int>(rank));
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t bar = map_to_cta(smem_u32(&full[stage]), 0);
          if (leader) {
            mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          uint8_t* dst = ring + stage * kStageBytes;
          tma_load_2d_pair(&tmX, bar, dst, kb * kBKBytes, row0);
          tma_load_2d_pair(&tmW, bar, dst + C::kHalfBytes, kb * kBKBytes, wrow0);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // no copy may land after the block has finished (both CTAs' copies complete on the
      // leader's barriers)
      for (int s = 0; s < kStages; ++s)
        if (armed & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait(&full[s], (armed_parity >> s) & 1u, p.limit_ns / 4 + 1, &no_abort, nullptr);
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // -------------------------------------------------------------- MMA issuer (leader)
      int stage = 0;
      uint32_t phase = 0, tcount = 0;
      bool ok = true;
      for (int t = cluster_id; ok && t < total_tiles; t += clusters, ++tcount) {
        const uint32_t buf = tcount & 1;
        if (!mbar_wait(&acc_empty[buf], ((tcount >> 1) & 1) ^ 1, p.limit_ns, abort_flag,
                       p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(ring + stage * kStageBytes);
          const uint32_t b_base = a_base + C::kHalfBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_bf16_pair(d, make_sdesc(a_base + j * 32, 16, 1024, kSwizzle128B),
                          make_sdesc(b_base + j * 32, 16, 1024, kSwizzle128B), p.idesc,
                          (kb | j) != 0);
          tc_commit_pair(&empty[stage], kPairMask);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair(&acc_full[buf], kPairMask);
      }
      // every MMA must be finished before tensor memory is freed
      tc_commit_pair(drain, 1);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, p.limit_ns, &no_abort, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- output stage (both CTAs)
    constexpr int kCols = BN / 2, kPieces = kCols / 32;
    const int q = warp & 3;                            // tensor-memory lane quarter
    const int h = (warp - C::kOutWarp0) >> 2;          // which half of the tile's columns
    const uint32_t acc_empty_leader = map_to_cta(smem_u32(acc_empty), 0);
    uint32_t tcount = 0;
    for (int t = cluster_id; t < total_tiles; t += clusters, ++tcount) {
      int mt, nt;
      tile_coords(t, NT, gt.tile_start[G], mt, nt);
      const int g = find_group(gt, G, mt);
      const int64_t l = static_cast<int64_t>(mt - gt.tile_start[g]) * 256 + 128 * static_cast<int>(rank) +
                        q * 32 + lane;
      const bool valid = l < gt.size[g];
      const uint32_t buf = tcount & 1;
      if (!mbar_wait(&acc_full[buf], (tcount >> 1) & 1, p.limit_ns, abort_flag, p.status)) break;
      tc_fence_after();
      // 32-column pieces of 32 lanes x 32 values (tcgen05.ld.32x32b), two in flight; the
      // leader's accumulator barrier is told after the warp's last load
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + h * kCols;
      const int64_t col0 = static_cast<int64_t>(nt) * BN + h * kCols;
      __nv_bfloat16* out = p.D + (gt.start[g] + l) * p.N + col0;
      auto store_piece = [&](int c, const uint32_t* x) { store32(out, col0, c, x, p); };
#pragma unroll
      for (int c = 0; c < kPieces; c += 2) {
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c * 32, ra);
        tmem_ld32(taddr + (c + 1) * 32, rb);
        tmem_ld_wait(ra);
        reg_fence(rb);
        if (c + 2 == kPieces) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_leader + buf * 8);
        }
        if (valid) {
          store_piece(c, ra);
          store_piece(c + 1, rb);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs are done with tensor memory and with each other's barriers
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
  cluster_sync();
}

bsmma_status launch_bf16_pair(const CUtensorMap& tx, const CUtensorMap& tw, Bf16Params p,
                              int64_t total_M, int G, cudaStream_t stream) {
  using C = PCfg;
  p.num_n_tiles = static_cast<int>((p.N + 255) / 256);
  p.idesc = idesc_bf16(256, 256);
  static int max_clusters = -1;   // benign race: every thread computes the same value
  if (max_clusters < 0) {
    if (cudaFuncSetAttribute(grouped_bf16_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return BSMMA_ERR_CUDA;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * sms, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_bf16_pair_kernel, &cfg) != cudaSuccess || n < 1)
      return BSMMA_ERR_CUDA;
    max_clusters = n;
  }
  const int64_t bound = ((total_M + 255) / 256 + G) * p.num_n_tiles;
  int64_t clusters = bound < max_clusters ? bound : max_clusters;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_bf16_pair_kernel, tx, tw, p);
  count_launches(1);
  return cuda_ok(e == cudaSuccess ? cudaGetLastError() : e);
}

template <int BN>
bsmma_status launch_bf16_bn(const CUtensorMap& tx, const CUtensorMap& tw, Bf16Params p,
                            int64_t total_M, int G, int sm_count, cudaStream_t stream) {
  using C = BCfg<BN>;
  p.num_n_tiles = static_cast<int>((p.N + BN - 1) / BN);
  p.idesc = idesc_bf16(kBM, BN);
  const int64_t bound = ((total_M + kBM - 1) / kBM + G) * p.num_n_tiles;
  int64_t grid = bound < sm_count ? bound : sm_count;
  if (grid < 1) grid = 1;
  static bool attr_set = false;   // benign race: setting the attribute twice is harmless
  if (!attr_set) {
    if (cudaFuncSetAttribute(grouped_bf16_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return BSMMA_ERR_CUDA;
    attr_set = true;
  }
  grouped_bf16_kernel<BN><<<static_cast<int>(grid), C::kThreads, C::kSmemBytes, stream>>>(tx, tw, p);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

// Tile choice: 128 or 256 columns on one CTA, or kPairTile (256 x 256 on an SM pair).
constexpr int kPairTile = 2;

bsmma_status launch_bf16_width(const void* X, const void* W, void* D, const int64_t* m_sizes,
                               int64_t total_M, int G, int64_t N, int64_t K, int bn,
                               const DeviceInfo* dev, cudaStream_t stream) {
  CUtensorMap tx, tw;
  // BF16 rows as bytes: a 128-byte box is 64 BF16 of K, the same shared-memory image.
  // With no rows there is no X tile to load; W's address stands in for the map.
  bsmma_status st = encode_tmap_u8(&tx, total_M > 0 ? X : W, K * 2, total_M > 0 ? total_M : 1,
                                   K * 2, kBKBytes, kBM);
  if (st != BSMMA_OK) return st;
  // a CTA of a pair loads 128 of the tile's 256 weight rows
  st = encode_tmap_u8(&tw, W, K * 2, static_cast<uint64_t>(G) * N, K * 2, kBKBytes,
                      bn == kPairTile ? 128 : bn);
  if (st != BSMMA_OK) return st;
  Bf16Params p;
  p.D = static_cast<__nv_bfloat16*>(D);
  p.d_align32 = (reinterpret_cast<uintptr_t>(D) & 31u) == 0 && N % 16 == 0;
  p.m_sizes = m_sizes;
  p.total_M = total_M;
  p.N = N;
  p.G = G;
  p.num_kb = static_cast<int>((K + 63) / 64);
  p.status = dev->status;
  p.limit_ns = wait_limit_ns();
  if (bn == kPairTile) return launch_bf16_pair(tx, tw, p, total_M, G, stream);
  if (bn == 256) return launch_bf16_bn<256>(tx, tw, p, total_M, G, dev->sm_count, stream);
  return launch_bf16_bn<128>(tx, tw, p, total_M, G, dev->sm_count, stream);
}

}  // namespace

bsmma_status launch_grouped_bf16(const void* X, const void* W, void* D, const int64_t* m_sizes,
                                 int64_t total_M, int G, int64_t N, int64_t K,
                                 cudaStream_t stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  static_assert(sizeof(GroupTable) + 512 <= 2048, "group table fits its shared-memory slot");
  // Wide tiles halve the MMA issue count and the reads of X per flop; they lose only when
  // too few tiles remain to keep every SM streaming W (row blocks estimated from total_M:
  // each group adds on average half a partial block).  SM-pair tiles (256 x 256) when the
  // groups average at least 128 rows: they carry a third less shared-memory traffic per
  // flop, which bounds the one-CTA tiles when the MMAs are busy (groups of a few dozen
  // rows stream W faster on one-CTA tiles).
  const int64_t row_blocks_est = (total_M + kBM - 1) / kBM + G / 2;
  const int forced = grouped_tile_width();
  const int variant = grouped_variant();
  int bn = (N > 128 && row_blocks_est * ((N + 255) / 256) * 2 >= dev->sm_count) ? 256 : 128;
  if (forced == 128 || forced == 256) bn = forced;
  const bool pair = variant == 3 ||
                    (variant == 0 && forced == 0 && N > 128 && total_M >= 128 * static_cast<int64_t>(G));
  if (pair) bn = kPairTile;
  if (forced == 0 && variant == 0 && N > 128) {
    // opt-in autotuning per (nextPow2(total_M), N, K, G)
    const std::string key = "grouped_bf16 " + std::to_string(next_pow2(total_M)) + " " +
                            std::to_string(N) + " " + std::to_string(K) + " " + std::to_string(G);
    bn = autotune_pick(key, {kPairTile, 256, 128}, bn, stream, [&](int c) {
      return launch_bf16_width(X, W, D, m_sizes, total_M, G, N, K, c, dev, stream);
    });
  }
  return launch_bf16_width(X, W, D, m_sizes, total_M, G, N, K, bn, dev, stream);
}

}  // namespace bsmma
