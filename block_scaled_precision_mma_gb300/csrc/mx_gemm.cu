// mx_gemm.cu -- dense block-scaled GEMM (MXFP8 / MXFP4) for sm_103a, one CTA per MMA.
//
// D[M][N] (BF16) = op(A) . op(B)^T with one E8M0 scale per 32 values along K
// ("PyTorch on AMD GPUs gains a FlyDSL backend", Interpretation; "Experimental
// FlyDSL GEMM backend for TE PyTorch", Supported Data Types / Validation).
//
// One persistent, warp-specialised kernel per (format, layout):
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) into a 4-stage ring; the
//               wide scale layouts into two small rings of their own (row-scale
//               chunks of 2 K groups, column-scale blocks of 1 or 2 K groups);
//   warp 1      allocates tensor memory; lane 0 copies scales into tensor memory with
//               128-lane x 32-byte tcgen05.cp copies and issues the block-scaled MMAs
//               (kind::mxf8f6f4 scale_vec::1X for FP8, kind::mxf4 scale_vec::2X for
//               packed FP4) into an FP32 accumulator in tensor memory;
//   warps 2-9   epilogue: tcgen05.ld of the accumulator, release of tensor memory to
//               the next tile, BF16 round-to-nearest-even, streaming 16-byte stores.
// Tile 128 x 256, 128 bytes of K per stage (128 FP8 / 256 FP4 values), four MMAs per
// stage.  Every wait is bounded; a timed-out wait latches a status and every role
// unwinds to the common teardown, which frees tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace bsmma {
namespace {

constexpr int kBM = 128, kBN = 256;
constexpr int kThreads = 320;       // 10 warps
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaCol = 256;   // 2 slots x 8 columns: row-scale chunks
constexpr uint32_t kSfbCol = 288;   // 4 slots x 8 columns: column-scale blocks
constexpr int kSmemLimit = 232448;  // 227 KB of dynamic shared memory per block

template <bool FP4>
struct Cfg {
  static constexpr int kKgPerStage = FP4 ? 2 : 1;         // 4-block K groups per stage
  static constexpr int kStagesPerChunk = 2 / kKgPerStage;  // a row-scale chunk spans 2 K groups
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = kBN * 128;
  static constexpr int kStages = 4;
  static constexpr int kSfaSlots = 2, kSfaSlotBytes = 4096;
  static constexpr int kSfbSlots = 3, kSfbSlotBytes = kKgPerStage * 4096;
  static constexpr int kSmemBytes = 1024 + kStages * (kABytes + kBBytes) +
                                    kSfaSlots * kSfaSlotBytes + kSfbSlots * kSfbSlotBytes + 256;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
};

struct DenseParams {
  __nv_bfloat16* D;
  Epilogue epi;         // optional bias and activation
  int64_t M, N;
  int sfa_kq;               // row-scale chunks per 128-row block
  int sfb_kg;               // column-scale blocks per 256-column block
  int num_m_tiles, num_n_tiles, num_k_stages;
  uint32_t idesc;
  int* status;
  uint64_t limit_ns;
};

// Scheduling unit u -> output tile (mt, nt).  Units walk the output in bands of
// kBandRows tile rows, along N inside a band, so that the CTAs running at the same
// time touch a compact block of A and B that stays in L2.
constexpr int kBandRows = 16;

__device__ __forceinline__ void unit_tile(const DenseParams& p, int u, int& mt, int& nt) {
  const int per_band = kBandRows * p.num_n_tiles;
  const int b = u / per_band;
  const int r0 = b * kBandRows;
  const int h = p.num_m_tiles - r0 < kBandRows ? p.num_m_tiles - r0 : kBandRows;
  const int v = u - b * per_band;
  mt = r0 + v % h;
  nt = v / h;
}

// A ring position: slot index and the parity of its current phase.
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance(int slots) {
    if (++slot == slots) {
      slot = 0;
      phase ^= 1;
    }
  }
};

// Copies 128 lanes x 32 bytes of shared memory into 8 tensor-memory columns.
__device__ __forceinline__ void tc_cp_wide(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 10 warps share an SM's four register-file quarters (16384 registers each) as
// 3+3+2+2 warps, so a thread may hold at most 16384 / (3 * 32) = 170 registers.
// EPI: the output stage adds a bias and / or applies an activation (a separate
// instantiation, so the plain GEMM's registers and code are unchanged).
template <bool FP4, bool A_MN, bool B_MN, bool EPI>
__global__ void __maxnreg__(168)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSFA,
                   const __grid_constant__ CUtensorMap tmSFB, const DenseParams p) {
  using C = Cfg<FP4>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::kStages * C::kABytes;
  uint8_t* sSFA = sB + C::kStages * C::kBBytes;
  uint8_t* sSFB = sSFA + C::kSfaSlots * C::kSfaSlotBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + C::kSfbSlots * C::kSfbSlotBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* sfa_full = empty + C::kStages;
  uint64_t* sfa_empty = sfa_full + C::kSfaSlots;
  uint64_t* sfb_full = sfa_empty + C::kSfaSlots;
  uint64_t* sfb_empty = sfb_full + C::kSfbSlots;
  uint64_t* acc_full = sfb_empty + C::kSfbSlots;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::kSfaSlots; ++s) {
      mbar_init(&sfa_full[s], 1);
      mbar_init(&sfa_empty[s], 1);
    }
    for (int s = 0; s < C::kSfbSlots; ++s) {
      mbar_init(&sfb_full[s], 1);
      mbar_init(&sfb_empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total_units = p.num_m_tiles * p.num_n_tiles;
  const int first_unit = static_cast<int>(blockIdx.x);
  const int unit_stride = static_cast<int>(gridDim.x);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      Ring st, sa, sb;
      uint32_t armed = 0, armed_parity = 0;   // data stages armed, for the drain at exit
      bool ok = true;
      for (int u = first_unit; ok && u < total_units; u += unit_stride) {
        int mt, nt;
        unit_tile(p, u, mt, nt);
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          if (!mbar_wait(&empty[st.slot], st.phase ^ 1, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st.slot], C::kABytes + C::kBBytes);
          armed |= 1u << st.slot;
          armed_parity = (armed_parity & ~(1u << st.slot)) | (st.phase << st.slot);
          uint8_t* a_dst = sA + st.slot * C::kABytes;
          uint8_t* b_dst = sB + st.slot * C::kBBytes;
          if (A_MN) tma_load_2d(&tmA, &full[st.slot], a_dst, mt * kBM, ks * 128);
          else      tma_load_2d(&tmA, &full[st.slot], a_dst, ks * 128, mt * kBM);
          if (B_MN) {
            tma_load_2d(&tmB, &full[st.slot], b_dst, nt * kBN, ks * 128);
            tma_load_2d(&tmB, &full[st.slot], b_dst + 16384, nt * kBN + 128, ks * 128);
          } else {
            tma_load_2d(&tmB, &full[st.slot], b_dst, ks * 128, nt * kBN);
          }
          st.advance(C::kStages);
          // column scales of the stage's K groups (each block: one copy per lane quarter)
          if (!mbar_wait(&sfb_empty[sb.slot], sb.phase ^ 1, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sfb_full[sb.slot], C::kSfbSlotBytes);
          tma_load_2d(&tmSFB, &sfb_full[sb.slot], sSFB + sb.slot * C::kSfbSlotBytes, 0,
                      (nt * p.sfb_kg + ks * C::kKgPerStage) * 4);
          sb.advance(C::kSfbSlots);
          // row scales of this CTA's 128 A rows, one chunk per two K groups
          if (ks % C::kStagesPerChunk == 0) {
            if (!mbar_wait(&sfa_empty[sa.slot], sa.phase ^ 1, p.limit_ns, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sfa_full[sa.slot], C::kSfaSlotBytes);
            tma_load_2d(&tmSFA, &sfa_full[sa.slot], sSFA + sa.slot * C::kSfaSlotBytes, 0,
                        (mt * p.sfa_kq + ks / C::kStagesPerChunk) * 4);
            sa.advance(C::kSfaSlots);
          }
        }
      }
      // Make sure no copy into shared memory is still in flight at exit.
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait(&full[s], (armed_parity >> s) & 1u, p.limit_ns / 4 + 1, &no_abort, nullptr);
        }
      if (!ok) {   // scale copies may still be landing after an abort: give them time
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      Ring st, sa, sb;
      uint32_t chunk = 0, kgs = 0;   // row-scale chunks and column-scale K groups consumed
      bool ok = true;
      int local = 0;
      for (int u = first_unit; ok && u < total_units; u += unit_stride, ++local) {
        if (!mbar_wait(acc_empty, (local & 1) ^ 1, p.limit_ns, abort_flag, p.status)) break;
        tc_fence_after();
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          const int sub = ks % C::kStagesPerChunk;
          const uint32_t sfa_t = tmem + kSfaCol + (chunk & 1) * 8;
          if (sub == 0) {
            if (!mbar_wait(&sfa_full[sa.slot], sa.phase, p.limit_ns, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            tc_cp_wide(sfa_t, make_sdesc(smem_u32(sSFA + sa.slot * C::kSfaSlotBytes), 128, 256, 0));
            tc_commit(&sfa_empty[sa.slot]);
            sa.advance(C::kSfaSlots);
          }
          if (!mbar_wait(&sfb_full[sb.slot], sb.phase, p.limit_ns, abort_flag, p.status) ||
              !mbar_wait(&full[st.slot], st.phase, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sfb_t[C::kKgPerStage];
#pragma unroll
          for (int g = 0; g < C::kKgPerStage; ++g) {
            sfb_t[g] = tmem + kSfbCol + ((kgs + g) & 3) * 8;
            tc_cp_wide(sfb_t[g], make_sdesc(smem_u32(sSFB + sb.slot * C::kSfbSlotBytes + g * 4096),
                                            128, 256, 0));
          }
          tc_commit(&sfb_empty[sb.slot]);
          sb.advance(C::kSfbSlots);
          kgs += C::kKgPerStage;
          const uint32_t a_base = smem_u32(sA + st.slot * C::kABytes);
          const uint32_t b_base = smem_u32(sB + st.slot * C::kBBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = A_MN ? make_sdesc(a_base + j * 4096, 16384, 1024, kSwizzle128B)
                                     : make_sdesc(a_base + j * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = B_MN ? make_sdesc(b_base + j * 4096, 16384, 1024, kSwizzle128B)
                                     : make_sdesc(b_base + j * 32, 16, 1024, kSwizzle128B);
            const uint32_t acc = (ks | j) != 0;
            if (FP4) {
              const int g = j >> 1;                      // K group within the stage
              const uint32_t sfid = (j & 1) * 2;
              mma_mxf4(tmem, ad, bd, p.idesc | idesc_sf_id(sfid, sfid),
                       sfa_t + 4 * (sub * C::kKgPerStage + g), sfb_t[g], acc);
            } else {
              mma_mxf8f6f4(tmem, ad, bd, p.idesc | idesc_sf_id(j, j), sfa_t + 4 * sub, sfb_t[0], acc);
            }
          }
          tc_commit(&empty[st.slot]);
          st.advance(C::kStages);
          if (sub == C::kStagesPerChunk - 1 || ks == p.num_k_stages - 1) ++chunk;
        }
        if (ok) tc_commit(acc_full);
      }
      // Every MMA and scale copy must be finished before tensor memory is freed.
      tc_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, p.limit_ns, &no_abort, nullptr);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    constexpr int kCols = kBN / 2;         // columns per epilogue warp
    constexpr int kChunks = kCols / 32;
    const int q = warp & 3;                // tensor-memory lane quarter of this warp
    const int h = (warp - 2) >> 2;         // which half of the tile's columns
    int local = 0;
    for (int u = first_unit; u < total_units; u += unit_stride, ++local) {
      int mt, nt;
      unit_tile(p, u, mt, nt);
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
      if (lane == 0) mbar_arrive(acc_empty);
      const int64_t row = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
      const int64_t col0 = static_cast<int64_t>(nt) * kBN + h * kCols;
      if (row < p.M) {
        __nv_bfloat16* out = p.D + row * p.N + col0;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int o = c * 32 + v * 8;
            if (col0 + o < p.N) {
              if constexpr (EPI)
                store8(out + o, &r[c][v * 8], col0 + o, p.epi);
              else
                st_global_v4_cs(out + o,
                                pack_bf16x2(__uint_as_float(r[c][v * 8 + 0]), __uint_as_float(r[c][v * 8 + 1])),
                                pack_bf16x2(__uint_as_float(r[c][v * 8 + 2]), __uint_as_float(r[c][v * 8 + 3])),
                                pack_bf16x2(__uint_as_float(r[c][v * 8 + 4]), __uint_as_float(r[c][v * 8 + 5])),
                                pack_bf16x2(__uint_as_float(r[c][v * 8 + 6]), __uint_as_float(r[c][v * 8 + 7])));
            }
          }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool FP4, bool A_MN, bool B_MN, bool EPI>
bsmma_status launch_dense(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                          const CUtensorMap& tsb, const DenseParams& p, int sm_count,
                          cudaStream_t stream) {
  using C = Cfg<FP4>;
  auto kern = mx_gemm_kernel<FP4, A_MN, B_MN, EPI>;
  static bool attr_set = false;   // benign race: setting the attribute twice is harmless
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
      return BSMMA_ERR_CUDA;
    attr_set = true;
  }
  const int64_t units = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
  const int grid = static_cast<int>(units < sm_count ? units : sm_count);
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(ta, tb, tsa, tsb, p);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace

namespace {
bsmma_status launch_mx_gemm_variant(const void* A, const uint8_t* sfa, const void* B,
                                    const uint8_t* sfb, void* D, int64_t M, int64_t N, int64_t K,
                                    bsmma_layout layout, bsmma_fmt a_fmt, bsmma_fmt b_fmt,
                                    cudaStream_t stream, const void* bias, int act, int variant,
                                    bool may_split);
}  // namespace

bsmma_status launch_mx_gemm(const void* A, const uint8_t* sfa, const void* B, const uint8_t* sfb,
                            void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                            bsmma_fmt a_fmt, bsmma_fmt b_fmt, cudaStream_t stream,
                            const void* bias, int act, bool may_allocate) {
  // SM-pair MMAs unless the one-CTA variant is asked for, or (opt-in) tuning per
  // (nextPow2(M), N, K, layout, formats) picks it
  int variant = dense_variant();
  if (variant == 0) {
    const std::string key = "dense " + std::to_string(next_pow2(M)) + " " + std::to_string(N) +
                            " " + std::to_string(K) + " " + std::to_string(static_cast<int>(layout)) +
                            " " + std::to_string(static_cast<int>(a_fmt)) + " " +
                            std::to_string(static_cast<int>(b_fmt));
    if (may_allocate) {
      variant = autotune_pick(key, {3, 1}, 3, stream, [&](int v) {
        return launch_mx_gemm_variant(A, sfa, B, sfb, D, M, N, K, layout, a_fmt, b_fmt, stream,
                                      bias, act, v, true);
      });
    } else {
      const int cached = autotune_cached(key);
      variant = cached == 1 || cached == 3 ? cached : 3;
    }
  }
  return launch_mx_gemm_variant(A, sfa, B, sfb, D, M, N, K, layout, a_fmt, b_fmt, stream, bias,
                                act, variant, may_allocate);
}

namespace {
bsmma_status launch_mx_gemm_variant(const void* A, const uint8_t* sfa, const void* B,
                                    const uint8_t* sfb, void* D, int64_t M, int64_t N, int64_t K,
                                    bsmma_layout layout, bsmma_fmt a_fmt, bsmma_fmt b_fmt,
                                    cudaStream_t stream, const void* bias, int act, int variant,
                                    bool may_split) {
  if (variant == 3)
    return launch_mx_gemm_2sm(A, sfa, B, sfb, D, M, N, K, layout, a_fmt, b_fmt, stream, bias, act,
                              may_split);
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  const bool fp4 = (a_fmt == BSMMA_E2M1);
  const uint64_t kbytes = fp4 ? static_cast<uint64_t>(K / 2) : static_cast<uint64_t>(K);
  const int64_t kblocks = K / 32;
  const int64_t kq = (kblocks + 7) / 8;          // row-scale chunks per 128 rows
  const int64_t kgp = 2 * ((kblocks + 7) / 8);   // column-scale blocks per 256 columns
  const int num_m_tiles = static_cast<int>((M + kBM - 1) / kBM);
  CUtensorMap ta, tb, tsa, tsb;
  if (layout == BSMMA_TN) st = encode_tmap_u8(&ta, A, M, K, M, 128, 128);
  else st = encode_tmap_u8(&ta, A, kbytes, M, kbytes, 128, 128);
  if (st != BSMMA_OK) return st;
  if (layout == BSMMA_NT) st = encode_tmap_u8(&tb, B, kbytes, N, kbytes, 128, kBN);
  else st = encode_tmap_u8(&tb, B, N, K, N, 128, 128);
  if (st != BSMMA_OK) return st;
  // both scale layouts viewed as rows of 1 KB ([*][256 words]): a row-scale chunk is 4
  // rows, a column-scale block 4 rows (its lane-quarter copies)
  st = encode_tmap_words(&tsa, sfa, 256, static_cast<uint64_t>(2 * ((M + 255) / 256) * kq * 4), 256, 4);
  if (st != BSMMA_OK) return st;
  st = encode_tmap_words(&tsb, sfb, 256, static_cast<uint64_t>(((N + 255) / 256) * kgp * 4), 256,
                         fp4 ? 8 : 4);
  if (st != BSMMA_OK) return st;

  DenseParams p;
  p.D = static_cast<__nv_bfloat16*>(D);
  p.epi.bias = static_cast<const __nv_bfloat16*>(bias);
  p.epi.act = act;
  p.M = M;
  p.N = N;
  p.sfa_kq = static_cast<int>(kq);
  p.sfb_kg = static_cast<int>(kgp);
  p.num_m_tiles = num_m_tiles;
  p.num_n_tiles = static_cast<int>((N + kBN - 1) / kBN);
  p.num_k_stages = static_cast<int>((static_cast<int64_t>(kbytes) + 127) / 128);
  const uint32_t af = fp4 ? 1u : static_cast<uint32_t>(a_fmt);   // kind::mxf4 codes E2M1 as 1
  const uint32_t bf = fp4 ? 1u : static_cast<uint32_t>(b_fmt);
  p.idesc = idesc_block_scaled(af, bf, layout == BSMMA_TN, layout != BSMMA_NT, kBM, kBN);
  p.status = dev->status;
  p.limit_ns = wait_limit_ns();
  const int sms = dev->sm_count;
  const bool epi = bias != nullptr || act != 0;
#define BSMMA_DENSE(F, A, B)                                                     \
  (epi ? launch_dense<F, A, B, true>(ta, tb, tsa, tsb, p, sms, stream)           \
       : launch_dense<F, A, B, false>(ta, tb, tsa, tsb, p, sms, stream))
  if (fp4) return BSMMA_DENSE(true, false, false);
  switch (layout) {
    case BSMMA_NT: return BSMMA_DENSE(false, false, false);
    case BSMMA_NN: return BSMMA_DENSE(false, false, true);
    default:       return BSMMA_DENSE(false, true, true);
  }
#undef BSMMA_DENSE
}
}  // namespace

}  // namespace bsmma
