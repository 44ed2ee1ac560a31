// mx_gemm_2sm.cu -- dense block-scaled GEMM on SM pairs (tcgen05 cta_group::2).
//
// Same operation as mx_gemm.cu (D = op(A) . op(B)^T with E8M0 block scales; "PyTorch
// on AMD GPUs gains a FlyDSL backend", Interpretation), computed by 2-CTA clusters:
// one MMA instruction covers a 256 x 256 output tile spread over the two SMs of a
// pair.  Each CTA holds its own 128 rows of A and its own 128 rows of B in shared
// memory, so per SM the operand bytes per flop are two thirds of the single-CTA
// 128 x 256 tile, and six stages fit where four did.
//
//   both CTAs, warp 0   TMA producer: its A half, its B half and the scale atoms of
//                       its A rows and of all 256 B rows, completing bytes on the
//                       leader CTA's stage barrier;
//   leader,    warp 1   lane 0 copies the scales into both CTAs' tensor memory and
//                       issues the pair MMAs; commits release the stage in both CTAs;
// Work split: whole 256 x 256 units go round robin over the clusters; when the last wave
// would leave clusters idle, the k-stages of its leftover units are shared out in equal
// contiguous ranges instead (stream-K), and a unit whose stages fall to several clusters
// is finished by the last of them to arrive: each writes its FP32 partial sums to a
// workspace slot and counts itself in, and the last one adds the slots in stage order
// (the same order whoever arrives last) before its output stage.
//   both CTAs, warps 2-9  epilogue of the CTA's 128 accumulator rows: tensor memory ->
//                       registers, an arrive on the leader's accumulator barrier (the next
//                       unit's MMAs may start), then BF16 pieces of 32 rows x 32 columns
//                       through a 2 KB shared-memory buffer per warp to TMA tensor
//                       stores.
// Every wait is bounded; on a timeout each role unwinds to the common teardown.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"
#include "store_stage.cuh"
#include "stream_k.cuh"

namespace bsmma {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaCol = 256;   // 2 slots x 8 columns: row-scale chunks
constexpr uint32_t kSfbCol = 288;   // 4 slots x 8 columns: column-scale blocks
constexpr int kSmemLimit = 232448;
constexpr int kBandUnits = 8;       // unit rows (256 output rows each) per raster band

template <bool FP4>
struct Cfg2 {
  static constexpr int kSfbRepl = 4;                      // one column-scale copy per lane quarter
  static constexpr int kKgPerStage = FP4 ? 2 : 1;        // 4-block K groups per 128-byte stage
  static constexpr int kStagesPerChunk = 2 / kKgPerStage; // a row-scale chunk spans 2 K groups
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = 128 * 128;
  static constexpr int kSfbBytes = kKgPerStage * kSfbRepl * 1024;
  static constexpr int kChunkBytes = 4096;                // row-scale chunk, in the stage that loads it
  static constexpr int kStageBytes = kABytes + kBBytes + kSfbBytes + kChunkBytes;
  static constexpr int kOutBytes = 8 * 2048;               // output staging: 2 KB per epilogue warp
  static constexpr int kStages0 = (kSmemLimit - 2048 - kOutBytes) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kOutBytes + 512;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
};

struct Pair2Params {
  __nv_bfloat16* D;
  float* part;          // split-unit partial sums [clusters][2][2 CTAs][128 x 256], or null
  int* arrivals;        // [leftover units][2 CTAs][8 epilogue warps] arrivals (zero between launches)
  Epilogue epi;         // optional bias and activation
  int64_t M, N;
  int sfa_kq;           // row-scale chunks per 128-row block
  int sfb_kg;           // column-scale blocks per 256-column block
  int num_m_tiles;      // 128-row tiles of D
  int num_unit_rows;    // 256-row pair units
  int num_n_tiles;      // 256-column tiles
  int num_k_stages;
  uint32_t idesc;
  int* status;
  uint64_t limit_ns;
};

// 128 lanes x 32 bytes of shared memory into 8 tensor-memory columns, in both CTAs.
__device__ __forceinline__ void tc_cp_wide_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
__device__ __forceinline__ void mma_mxf8f6f4_pair(uint32_t d, uint64_t a, uint64_t b,
                                                  uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                                  uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void mma_mxf4_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

// A range shorter than this many stage granules is not worth splitting a unit for.
constexpr int kMinGranules = 8;
// The extra time of a split range (pipeline start, partial sums written and added), in
// k-stages of the unit's own MMA time.
constexpr int kSplitCostStages = 40;

// Unit u -> (256-row unit row ur, 256-column tile nt), banded along N for L2 reuse.
__device__ __forceinline__ void unit_tile2(const Pair2Params& p, int u, int& ur, int& nt) {
  const int per_band = kBandUnits * p.num_n_tiles;
  const int b = u / per_band;
  const int r0 = b * kBandUnits;
  const int h = p.num_unit_rows - r0 < kBandUnits ? p.num_unit_rows - r0 : kBandUnits;
  const int v = u - b * per_band;
  ur = r0 + v % h;
  nt = v / h;
}

// 10 warps share an SM's four register-file quarters (16384 registers each) as
// 3+3+2+2 warps, so a thread may hold at most 16384 / (3 * 32) = 170 registers.
// EPI: 0 for the plain output stage; else the stage adds the bias (when given) and
// applies activation EPI - 1 (Epilogue::act).  Each is an instantiation of its own, so
// the plain GEMM's registers and code are unchanged and an activated kernel carries only
// its own activation's code (with every activation behind a run-time switch, even a
// bias alone cost 4% at 8192^3: the epilogue's unrolled code grew about tenfold).
template <bool FP4, bool A_MN, bool B_MN, int EPI>
__global__ void __maxnreg__(168)
    mx_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmSFA,
                       const __grid_constant__ CUtensorMap tmSFB,
                       const __grid_constant__ CUtensorMap tmD, const Pair2Params p) {
  using C = Cfg2<FP4>;
  constexpr int kSfbRepl = C::kSfbRepl;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::kStages * C::kABytes;
  uint8_t* sSFB = sB + C::kStages * C::kBBytes;
  uint8_t* sSFA = sSFB + C::kStages * C::kSfbBytes;        // one chunk slot per stage
  uint8_t* sOut = sSFA + C::kStages * C::kChunkBytes;       // output staging
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + C::kOutBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  DSched& sched = *reinterpret_cast<DSched*>(const_cast<int*>(abort_flag + 2));   // + 1 unused
  volatile int* work_state = abort_flag + 2 + (sizeof(DSched) + 3) / 4;   // [10 warps][4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  constexpr uint16_t kPairMask = 3;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);     // used in the leader: its producer's arrive + both CTAs' bytes
      mbar_init(&empty[s], 1);    // released by the leader's commit in both CTAs
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * kEpiWarps);   // used in the leader: epilogues of both CTAs
    mbar_init(drain, 1);
    *abort_flag = 0;
    // the split cost as measured (8192^3 FP8, KS 64, 36 leftover units of 76: 2.5% slower
    // with splits; 4096x4096x14336, KS 112, 28 of 76: 3.3% faster; FP4 8192^3, KS 32:
    // 4.9% slower)
    sched = make_dsched(p.num_unit_rows * p.num_n_tiles, p.num_k_stages, C::kStagesPerChunk,
                        static_cast<int>(gridDim.x >> 1), p.part != nullptr, kSplitCostStages,
                        kMinGranules);
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
    prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int cluster_id = static_cast<int>(blockIdx.x >> 1);
  const int clusters = static_cast<int>(gridDim.x >> 1);
  volatile int* wst = work_state + warp * 4;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      dwork_init(sched, wst, cluster_id);
      int u, ks0, ks1;
      while (ok && dwork_next(sched, wst, clusters, u, ks0, ks1)) {
        int ur, nt;
        unit_tile2(p, u, ur, nt);
        const int mt = ur * 2 + static_cast<int>(rank);          // this CTA's 128 rows of A
        const int nb = nt * 2 + static_cast<int>(rank);          // this CTA's 128 rows of B
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t bar = map_to_cta(smem_u32(&full[stage]), 0);
          const int kq = ks / C::kStagesPerChunk;
          const bool chunk_start = (ks % C::kStagesPerChunk) == 0;
          if (leader) {
            mbar_arrive_expect_tx(&full[stage], 2 * (C::kStageBytes - C::kChunkBytes +
                                                     (chunk_start ? C::kChunkBytes : 0)));
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          uint8_t* a_dst = sA + stage * C::kABytes;
          uint8_t* b_dst = sB + stage * C::kBBytes;
          if (A_MN) tma_load_2d_pair(&tmA, bar, a_dst, mt * 128, ks * 128);
          else      tma_load_2d_pair(&tmA, bar, a_dst, ks * 128, mt * 128);
          if (B_MN) tma_load_2d_pair(&tmB, bar, b_dst, nb * 128, ks * 128);
          else      tma_load_2d_pair(&tmB, bar, b_dst, ks * 128, nb * 128);
          // column scales of all 256 B rows (blocks already hold one copy per lane quarter)
          tma_load_2d_pair(&tmSFB, bar, sSFB + stage * C::kSfbBytes, 0,
                           (nt * p.sfb_kg + ks * C::kKgPerStage) * kSfbRepl);
          // row scales of this CTA's 128 A rows, one chunk per 4 K groups
          if (chunk_start)
            tma_load_2d_pair(&tmSFA, bar, sSFA + stage * C::kChunkBytes, 0,
                             (mt * p.sfa_kq + kq) * 4);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait(&full[s], (armed_parity >> s) & 1u, p.limit_ns / 4 + 1, &no_abort, nullptr);
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer (leader)
      int stage = 0;
      uint32_t phase = 0, kiter = 0, chunk = 0;
      bool ok = true;
      int local = 0;
      dwork_init(sched, wst, cluster_id);
      int u, ks0, ks1;
      for (; ok && dwork_next(sched, wst, clusters, u, ks0, ks1); ++local) {
        if (!mbar_wait(acc_empty, (local & 1) ^ 1, p.limit_ns, abort_flag, p.status)) break;
        tc_fence_after();
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!mbar_wait(&full[stage], phase, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int sub = ks % C::kStagesPerChunk;                  // stage within the chunk
          const uint32_t sfa_t = tmem + kSfaCol + (chunk & 1) * 8;
          if (sub == 0)
            tc_cp_wide_pair(sfa_t, make_sdesc(smem_u32(sSFA + stage * C::kChunkBytes), 128, 256, 0));
          uint32_t sfb_t[C::kKgPerStage];
#pragma unroll
          for (int g = 0; g < C::kKgPerStage; ++g) {
            sfb_t[g] = tmem + kSfbCol + ((kiter * C::kKgPerStage + g) & 3) * 8;
            tc_cp_wide_pair(sfb_t[g], make_sdesc(smem_u32(sSFB + stage * C::kSfbBytes +
                                                           g * kSfbRepl * 1024),
                                                 128, 256, 0));
          }
          const uint32_t a_base = smem_u32(sA + stage * C::kABytes);
          const uint32_t b_base = smem_u32(sB + stage * C::kBBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = A_MN ? make_sdesc(a_base + j * 4096, 16384, 1024, kSwizzle128B)
                                     : make_sdesc(a_base + j * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = B_MN ? make_sdesc(b_base + j * 4096, 16384, 1024, kSwizzle128B)
                                     : make_sdesc(b_base + j * 32, 16, 1024, kSwizzle128B);
            const uint32_t acc = ks != ks0 || j != 0;
            if (FP4) {
              const int g = j >> 1;                                   // K group within the stage
              const uint32_t sfid = (j & 1) * 2;
              mma_mxf4_pair(tmem, ad, bd, p.idesc | idesc_sf_id(sfid, sfid),
                            sfa_t + 4 * (sub * C::kKgPerStage + g), sfb_t[g], acc);
            } else {
              mma_mxf8f6f4_pair(tmem, ad, bd, p.idesc | idesc_sf_id(j, j), sfa_t + 4 * sub,
                                sfb_t[0], acc);
            }
          }
          tc_commit_pair(&empty[stage], kPairMask);
          ++kiter;
          if (sub == C::kStagesPerChunk - 1 || ks == ks1 - 1) ++chunk;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit_pair(acc_full, kPairMask);
      }
      // every MMA and scale copy must be finished before tensor memory is freed
      tc_commit_pair(drain, 1);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, p.limit_ns, &no_abort, nullptr);
    }
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs)
    constexpr int kCols = 128;             // columns per epilogue warp
    constexpr int kChunks = kCols / 32;
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t acc_empty_leader = map_to_cta(smem_u32(acc_empty), 0);
    int local = 0;
    dwork_init(sched, wst, cluster_id);
    int u, ks0, ks1;
    for (; dwork_next(sched, wst, clusters, u, ks0, ks1); ++local) {
      int ur, nt;
      unit_tile2(p, u, ur, nt);
      const int mt = ur * 2 + static_cast<int>(rank);
      if (!mbar_wait(acc_full, local & 1, p.limit_ns, abort_flag, p.status)) break;
      tc_fence_after();
      uint32_t r[kChunks][32];
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * kCols;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) tmem_ld32(tbase + c * 32, r[c]);
      tmem_ld_wait(r[0]);
#pragma unroll
      for (int c = 1; c < kChunks; ++c) reg_fence(r[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
      const int64_t row0 = static_cast<int64_t>(mt) * 128 + q * 32;
      const int64_t col0 = static_cast<int64_t>(nt) * 256 + h * kCols;
      uint8_t* stg = sOut + (warp - 2) * 2048;
      // Output of the 32-column piece c of this warp's 32 rows x 128 columns (vals: 32
      // FP32 values of this lane's row): BF16 through the warp's buffer to a TMA tensor
      // store -- lane = row, the 16-byte group v of 8 columns at position
      // v ^ ((r / 2) % 4), the tensor map's 64-byte swizzle, so the lanes hit distinct
      // banks.
      auto store_piece = [&](int c, const uint32_t* vals) {
        if (row0 >= p.M || col0 + c * 32 >= p.N) return;   // warp-uniform
        uint32_t o[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int64_t col = col0 + c * 32 + g * 8;
          if constexpr (EPI != 0) {
            if (col < p.N) {
              apply8_act<EPI - 1>(vals + g * 8, col, p.epi.bias, o[g]);
              continue;
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            o[g][j] = pack_bf16x2(__uint_as_float(vals[g * 8 + 2 * j]),
                                  __uint_as_float(vals[g * 8 + 2 * j + 1]));
        }
        if (lane == 0) bulk_wait_group_read<0>();   // the previous piece has been read
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t a = smem_u32(stg + lane * 64 + ((g ^ ((lane >> 1) & 3)) * 16));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(o[g][0]),
                       "r"(o[g][1]), "r"(o[g][2]), "r"(o[g][3])
                       : "memory");
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmD, stg, static_cast<int32_t>(col0 + c * 32), static_cast<int32_t>(row0));
          bulk_commit_group();
        }
      };
      if (ks0 == 0 && ks1 == p.num_k_stages) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) store_piece(c, r[c]);
        continue;
      }
      // A split unit.  Slot layout, chosen so that a warp's 32 lanes write and read 512
      // contiguous bytes: [warp (quarter, half)][32-column piece][4-column group][lane];
      // the slot of cluster c for this unit is (c, its first or last unit, this CTA's half).
      const int v = u - sched.t_dp;
      float4* const part = reinterpret_cast<float4*>(p.part) + (q * 2 + h) * (kChunks * 8 * 32) + lane;
      auto slot_of = [&](int c) -> float4* {
        return part + static_cast<uint32_t>((c * 2 + dsk_slot(sched, c, v)) * 2 + static_cast<int>(rank)) *
                          (128 * 256 / 4);
      };
      float4* mine = slot_of(cluster_id);
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          __stcg(mine + (c * 8 + j) * 32,
                 make_float4(__uint_as_float(r[c][4 * j]), __uint_as_float(r[c][4 * j + 1]),
                             __uint_as_float(r[c][4 * j + 2]), __uint_as_float(r[c][4 * j + 3])));
      // each epilogue warp counts itself in on the unit's counter for its own rows and
      // columns, and the warp that arrives last for that part adds the slots: no barrier
      // between warps, so a warp that gives up on a wait blocks no other
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        int* ctr = p.arrivals + (v * 2 + static_cast<int>(rank)) * kEpiWarps + (warp - 2);
        const int nseg = dsk_last_worker(sched, v) - dsk_first_worker(sched, v) + 1;
        last = atomicAdd(ctr, 1) + 1 == nseg;
        if (last) *ctr = 0;   // every contributor has counted itself in
      }
      if (!__shfl_sync(0xffffffffu, last, 0)) continue;
      __threadfence();
      // the last to arrive: every contributor's slot summed in stage order, a 32-column
      // piece at a time, and stored.  Two contributors' loads are in flight together (the
      // sum sits at the end of the launch, and each round trip to L2 is on its path); the
      // additions keep contributor order, so the bits do not change.
      const int c_lo = dsk_first_worker(sched, v), c_hi = dsk_last_worker(sched, v);
      auto add4 = [](uint32_t* acc, const float4& x) {
        acc[0] = __float_as_uint(__uint_as_float(acc[0]) + x.x);
        acc[1] = __float_as_uint(__uint_as_float(acc[1]) + x.y);
        acc[2] = __float_as_uint(__uint_as_float(acc[2]) + x.z);
        acc[3] = __float_as_uint(__uint_as_float(acc[3]) + x.w);
      };
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        uint32_t sum[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) sum[i] = 0u;
        for (int cc = c_lo; cc <= c_hi; cc += 2) {
          const bool two = cc < c_hi;
          const float4* src0 = slot_of(cc) + c * 8 * 32;
          const float4* src1 = slot_of(two ? cc + 1 : cc) + c * 8 * 32;   // a repeat if alone
          float4 x0[8], x1[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            x0[j] = __ldcg(src0 + j * 32);
            x1[j] = __ldcg(src1 + j * 32);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) add4(sum + 4 * j, x0[j]);
          if (two) {
#pragma unroll
            for (int j = 0; j < 8; ++j) add4(sum + 4 * j, x1[j]);
          }
        }
        store_piece(c, sum);
      }
    }
    // every tensor store of this warp has finished reading and writing before the
    // buffers (and the block) go away
    if (lane == 0) bulk_wait_group<0>();
  }
  __syncthreads();
  cluster_sync();   // both CTAs are done with tensor memory and with each other's barriers
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  cluster_sync();
}

template <bool FP4, bool A_MN, bool B_MN, int EPI>
bsmma_status launch_2sm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                        const CUtensorMap& tsb, const CUtensorMap& td, const Pair2Params& p,
                        cudaStream_t stream) {
  using C = Cfg2<FP4>;
  auto kern = mx_gemm_2sm_kernel<FP4, A_MN, B_MN, EPI>;
  static int max_clusters = -1;   // benign race: every thread computes the same value
  if (max_clusters < 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
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
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
      return BSMMA_ERR_CUDA;
    max_clusters = n;
  }
  const int64_t units = static_cast<int64_t>(p.num_unit_rows) * p.num_n_tiles;
  const int grid = static_cast<int>(2 * (units < max_clusters ? units : max_clusters));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, td, p);
  count_launches(1);
  return cuda_ok(e == cudaSuccess ? cudaGetLastError() : e);
}

}  // namespace

bsmma_status launch_mx_gemm_2sm(const void* A, const uint8_t* sfa, const void* B,
                                const uint8_t* sfb, void* D, int64_t M, int64_t N, int64_t K,
                                bsmma_layout layout, bsmma_fmt a_fmt, bsmma_fmt b_fmt,
                                cudaStream_t stream, const void* bias, int act, bool may_split) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const bool fp4 = (a_fmt == BSMMA_E2M1);
  const uint64_t kbytes = fp4 ? static_cast<uint64_t>(K / 2) : static_cast<uint64_t>(K);
  const int64_t kblocks = K / 32;
  const int64_t kq = (kblocks + 7) / 8;                   // row-scale chunks per 128 rows
  const int64_t kgp = 2 * ((kblocks + 7) / 8);            // column-scale blocks per 256 columns
  CUtensorMap ta, tb, tsa, tsb, td;
  st = encode_tmap_bf16_out(&td, D, static_cast<uint64_t>(N), static_cast<uint64_t>(M), 32, 32);
  if (st != BSMMA_OK) return st;
  if (layout == BSMMA_TN) st = encode_tmap_u8(&ta, A, M, K, M, 128, 128);
  else st = encode_tmap_u8(&ta, A, kbytes, M, kbytes, 128, 128);
  if (st != BSMMA_OK) return st;
  if (layout == BSMMA_NT) st = encode_tmap_u8(&tb, B, kbytes, N, kbytes, 128, 128);
  else st = encode_tmap_u8(&tb, B, N, K, N, 128, 128);
  if (st != BSMMA_OK) return st;
  // both scale layouts viewed as rows of 1 KB ([*][256 words]): a row-scale chunk is 4
  // rows, a column-scale block 4 rows (its lane-quarter copies)
  st = encode_tmap_words(&tsa, sfa, 256, static_cast<uint64_t>(2 * ((M + 255) / 256) * kq * 4), 256, 4);
  if (st != BSMMA_OK) return st;
  st = encode_tmap_words(&tsb, sfb, 256, static_cast<uint64_t>(((N + 255) / 256) * kgp * 4), 256,
                         fp4 ? 8 : 4);
  if (st != BSMMA_OK) return st;
  Pair2Params p;
  p.part = nullptr;
  p.arrivals = nullptr;
  if (may_split) {
    st = split_workspace(stream, &p.part, &p.arrivals);
    if (st == BSMMA_ERR_WORKSPACE) {   // captured on a stream without one: no unit is split
      p.part = nullptr;
      p.arrivals = nullptr;
    } else if (st != BSMMA_OK) {
      return st;
    }
  }
  p.D = static_cast<__nv_bfloat16*>(D);
  p.epi.bias = static_cast<const __nv_bfloat16*>(bias);
  p.epi.act = act;
  p.M = M;
  p.N = N;
  p.sfa_kq = static_cast<int>(kq);
  p.sfb_kg = static_cast<int>(kgp);
  p.num_m_tiles = static_cast<int>((M + 127) / 128);
  p.num_unit_rows = static_cast<int>((M + 255) / 256);
  p.num_n_tiles = static_cast<int>((N + 255) / 256);
  p.num_k_stages = static_cast<int>((static_cast<int64_t>(kbytes) + 127) / 128);
  const uint32_t af = fp4 ? 1u : static_cast<uint32_t>(a_fmt);
  const uint32_t bf = fp4 ? 1u : static_cast<uint32_t>(b_fmt);
  p.idesc = idesc_block_scaled(af, bf, layout == BSMMA_TN, layout != BSMMA_NT, 256, 256);
  p.status = dev->status;
  p.limit_ns = wait_limit_ns();
  // output stage: 0 plain, else 1 + the activation (bias applied when given)
  const int epi = bias == nullptr && act == 0 ? 0 : 1 + act;
#define BSMMA_2SM(F, A, B)                                                       \
  (epi == 0   ? launch_2sm<F, A, B, 0>(ta, tb, tsa, tsb, td, p, stream)          \
   : epi == 1 ? launch_2sm<F, A, B, 1>(ta, tb, tsa, tsb, td, p, stream)          \
   : epi == 2 ? launch_2sm<F, A, B, 2>(ta, tb, tsa, tsb, td, p, stream)          \
   : epi == 3 ? launch_2sm<F, A, B, 3>(ta, tb, tsa, tsb, td, p, stream)          \
              : launch_2sm<F, A, B, 4>(ta, tb, tsa, tsb, td, p, stream))
  if (fp4) return BSMMA_2SM(true, false, false);
  switch (layout) {
    case BSMMA_NT: return BSMMA_2SM(false, false, false);
    case BSMMA_NN: return BSMMA_2SM(false, false, true);
    default:       return BSMMA_2SM(false, true, true);
  }
#undef BSMMA_2SM
}

}  // namespace bsmma
