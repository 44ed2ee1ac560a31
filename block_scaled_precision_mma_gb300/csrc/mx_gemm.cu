// mx_gemm.cu -- dense block-scaled GEMM (MXFP8 / MXFP4) for sm_103a.
//
// D[M][N] (BF16) = op(A) . op(B)^T with one E8M0 scale per 32 values along K
// ("PyTorch on AMD GPUs gains a FlyDSL backend", Interpretation; "Experimental
// FlyDSL GEMM backend for TE PyTorch", Supported Data Types / Validation).
//
// One persistent, warp-specialised kernel per (format, layout):
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and the tile's scale
//               atoms (bulk copies) into a multi-stage shared-memory ring;
//   warp 1      allocates tensor memory; lane 0 copies the stage's scale atoms into
//               tensor memory (tcgen05.cp) and issues the block-scaled MMAs
//               (kind::mxf8f6f4 scale_vec::1X for FP8, kind::mxf4 scale_vec::2X for
//               packed FP4) into an FP32 accumulator in tensor memory;
//   warps 2-9   epilogue: tcgen05.ld of the accumulator, release of tensor memory to
//               the next tile, BF16 round-to-nearest-even, 16-byte global stores.
// Tile 128 x BN, 128 bytes of K per stage (128 FP8 / 256 FP4 values), four MMAs
// per stage.  Every wait is bounded; a timed-out wait latches a status and every
// role unwinds to the common teardown, which frees tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace bsmma {
namespace {

constexpr int kBM = 128;
constexpr int kThreads = 320;       // 10 warps
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaCol = 256;   // 4 slots x 8 columns
constexpr uint32_t kSfbCol = 288;   // 4 slots x 16 columns
constexpr uint32_t kSfSlots = 4;
constexpr int kSmemLimit = 232448;  // 227 KB of dynamic shared memory per block
constexpr bool kPairDefault = true;

template <int BN, bool FP4>
struct Cfg {
  static constexpr int kAP = FP4 ? 2 : 1;                  // scale atoms per stage per 128 rows
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kSfaBytes = kAP * 512;
  static constexpr int kSfbBytes = (BN / 128) * kAP * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStages0 = (kSmemLimit - 2048) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
  static_assert(BN == 128 || BN == 256, "tile width");
};

struct DenseParams {
  const uint8_t* sfa;   // tiled scales of op(A)
  const uint8_t* sfb;   // tiled scales of op(B)
  __nv_bfloat16* D;
  int64_t M, N;
  int64_t sfa_kg, sfb_kg;   // 512-byte atoms per 128-row block of each scale buffer
  int num_m_tiles, num_n_tiles, num_k_stages;
  uint32_t idesc;
  int* status;
  uint64_t limit_ns;
};

// Scheduling unit u -> output tile (mt, nt).  Single CTAs take one tile per unit;
// a CTA pair (2-CTA cluster) takes two vertically adjacent tiles that share their
// B tile, which each CTA loads half of and multicasts to both.  Units walk the
// output in bands of kBandRows tile rows, along N inside a band, so that the CTAs
// running at the same time touch a compact block of A and B that stays in L2.
constexpr int kBandRows = 16;

template <bool PAIR>
__device__ __forceinline__ void unit_tile(const DenseParams& p, int u, uint32_t rank, int& mt,
                                          int& nt) {
  const int rows = PAIR ? (p.num_m_tiles + 1) >> 1 : p.num_m_tiles;   // unit rows
  const int band = PAIR ? kBandRows / 2 : kBandRows;
  const int per_band = band * p.num_n_tiles;
  const int b = u / per_band;
  const int r0 = b * band;
  const int h = rows - r0 < band ? rows - r0 : band;
  const int v = u - b * per_band;
  const int ur = r0 + v % h;
  nt = v / h;
  mt = PAIR ? ur * 2 + static_cast<int>(rank) : ur;
}

// 10 warps share an SM's four register-file quarters (16384 registers each) as
// 3+3+2+2 warps, so a thread may hold at most 16384 / (3 * 32) = 170 registers.
template <int BN, bool FP4, bool A_MN, bool B_MN, bool PAIR>
__global__ void __maxnreg__(168)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const DenseParams p) {
  using C = Cfg<BN, FP4>;
  static_assert(!PAIR || BN == 256, "a CTA pair splits a 256-wide B tile");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::kStages * C::kABytes;
  uint8_t* sSFA = sB + C::kStages * C::kBBytes;
  uint8_t* sSFB = sSFA + C::kStages * C::kSfaBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + C::kStages * C::kSfbBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  constexpr uint16_t kPairMask = 3;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PAIR ? 2 : 1);   // a pair frees a stage only when both MMAs are done
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();   // the peer's barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total_units = PAIR ? ((p.num_m_tiles + 1) >> 1) * p.num_n_tiles
                               : p.num_m_tiles * p.num_n_tiles;
  const int first_unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_stride = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int u = first_unit; ok && u < total_units; u += unit_stride) {
        int mt, nt;
        unit_tile<PAIR>(p, u, rank, mt, nt);
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          uint8_t* a_dst = sA + stage * C::kABytes;
          uint8_t* b_dst = sB + stage * C::kBBytes;
          if (A_MN) tma_load_2d(&tmA, &full[stage], a_dst, mt * kBM, ks * 128);
          else      tma_load_2d(&tmA, &full[stage], a_dst, ks * 128, mt * kBM);
          bulk_load(sSFA + stage * C::kSfaBytes,
                    p.sfa + (static_cast<int64_t>(mt) * p.sfa_kg + ks * C::kAP) * 512,
                    C::kSfaBytes, &full[stage]);
          if (PAIR) {
            // this CTA's 128-row half of the B tile and of its scales, to both CTAs
            const int r = static_cast<int>(rank);
            if (B_MN)
              tma_load_2d_mc(&tmB, &full[stage], b_dst + r * 16384, nt * BN + r * 128, ks * 128,
                             kPairMask);
            else
              tma_load_2d_mc(&tmB, &full[stage], b_dst + r * 16384, ks * 128, nt * BN + r * 128,
                             kPairMask);
            bulk_load_mc(sSFB + stage * C::kSfbBytes + r * C::kAP * 512,
                         p.sfb + ((static_cast<int64_t>(nt) * 2 + r) * p.sfb_kg + ks * C::kAP) * 512,
                         C::kAP * 512, &full[stage], kPairMask);
          } else {
            if (B_MN) {
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tma_load_2d(&tmB, &full[stage], b_dst + j * 16384, nt * BN + j * 128, ks * 128);
            } else {
              tma_load_2d(&tmB, &full[stage], b_dst, ks * 128, nt * BN);
            }
#pragma unroll
            for (int rb = 0; rb < BN / 128; ++rb)
              bulk_load(sSFB + stage * C::kSfbBytes + rb * C::kAP * 512,
                        p.sfb + ((static_cast<int64_t>(nt) * (BN / 128) + rb) * p.sfb_kg +
                                 ks * C::kAP) * 512,
                        C::kAP * 512, &full[stage]);
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Make sure no copy into shared memory is still in flight at exit.
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait(&full[s], (armed_parity >> s) & 1u, p.limit_ns / 4 + 1, &no_abort, nullptr);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0, kiter = 0;
      bool ok = true;
      int local = 0;
      for (int u = first_unit; ok && u < total_units; u += unit_stride, ++local) {
        if (!mbar_wait(acc_empty, (local & 1) ^ 1, p.limit_ns, abort_flag, p.status)) break;
        tc_fence_after();
        for (int ks = 0; ks < p.num_k_stages; ++ks) {
          if (!mbar_wait(&full[stage], phase, p.limit_ns, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t slot = kiter % kSfSlots;
          const uint32_t sfa_t = tmem + kSfaCol + slot * 8;
          const uint32_t sfb_t = tmem + kSfbCol + slot * 16;
          const uint32_t sfa_s = smem_u32(sSFA + stage * C::kSfaBytes);
          const uint32_t sfb_s = smem_u32(sSFB + stage * C::kSfbBytes);
#pragma unroll
          for (int a = 0; a < C::kAP; ++a) tc_cp_sf(sfa_t + a * 4, make_sdesc(sfa_s + a * 512, 0, 128, 0));
#pragma unroll
          for (int rb = 0; rb < BN / 128; ++rb)
#pragma unroll
            for (int a = 0; a < C::kAP; ++a)
              tc_cp_sf(sfb_t + a * 8 + rb * 4,
                       make_sdesc(sfb_s + (rb * C::kAP + a) * 512, 0, 128, 0));
          const uint32_t a_base = smem_u32(sA + stage * C::kABytes);
          const uint32_t b_base = smem_u32(sB + stage * C::kBBytes);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = A_MN ? make_sdesc(a_base + j * 4096, 16384, 1024, kSwizzle128B)
                                     : make_sdesc(a_base + j * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = B_MN ? make_sdesc(b_base + j * 4096, 16384, 1024, kSwizzle128B)
                                     : make_sdesc(b_base + j * 32, 16, 1024, kSwizzle128B);
            const uint32_t acc = (ks | j) != 0;
            if (FP4) {
              const uint32_t atom = j >> 1, sfid = (j & 1) * 2;
              mma_mxf4(tmem, ad, bd, p.idesc | idesc_sf_id(sfid, sfid), sfa_t + atom * 4,
                       sfb_t + atom * 8, acc);
            } else {
              mma_mxf8f6f4(tmem, ad, bd, p.idesc | idesc_sf_id(j, j), sfa_t, sfb_t, acc);
            }
          }
          if (PAIR) tc_commit_mc(&empty[stage], kPairMask);
          else tc_commit(&empty[stage]);
          ++kiter;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
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
    constexpr int kCols = BN / 2;          // columns per epilogue warp
    constexpr int kChunks = kCols / 32;
    const int q = warp & 3;                // tensor-memory lane quarter of this warp
    const int h = (warp - 2) >> 2;         // which half of the tile's columns
    int local = 0;
    for (int u = first_unit; u < total_units; u += unit_stride, ++local) {
      int mt, nt;
      unit_tile<PAIR>(p, u, rank, mt, nt);
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
      const int64_t col0 = static_cast<int64_t>(nt) * BN + h * kCols;
      if (row < p.M) {
        __nv_bfloat16* out = p.D + row * p.N + col0;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int o = c * 32 + v * 8;
            if (col0 + o < p.N)
              st_global_v4_cs(out + o,
                           pack_bf16x2(__uint_as_float(r[c][v * 8 + 0]), __uint_as_float(r[c][v * 8 + 1])),
                           pack_bf16x2(__uint_as_float(r[c][v * 8 + 2]), __uint_as_float(r[c][v * 8 + 3])),
                           pack_bf16x2(__uint_as_float(r[c][v * 8 + 4]), __uint_as_float(r[c][v * 8 + 5])),
                           pack_bf16x2(__uint_as_float(r[c][v * 8 + 6]), __uint_as_float(r[c][v * 8 + 7])));
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
  // neither CTA of a pair leaves while its peer may still signal its barriers
  if (PAIR) cluster_sync();
}

template <int BN, bool FP4, bool A_MN, bool B_MN, bool PAIR>
bsmma_status launch_dense(const CUtensorMap& ta, const CUtensorMap& tb, const DenseParams& p,
                          int sm_count, cudaStream_t stream) {
  using C = Cfg<BN, FP4>;
  auto kern = mx_gemm_kernel<BN, FP4, A_MN, B_MN, PAIR>;
  static int max_clusters = -1;   // benign race: every thread computes the same value
  if (max_clusters < 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
      return BSMMA_ERR_CUDA;
    int n = sm_count;
    if (PAIR) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) !=
          cudaSuccess)
        return BSMMA_ERR_CUDA;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * sm_count, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = C::kSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
        return BSMMA_ERR_CUDA;
    }
    max_clusters = n;
  }
  const int64_t units = PAIR ? static_cast<int64_t>((p.num_m_tiles + 1) / 2) * p.num_n_tiles
                             : static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
  const int64_t slots = PAIR ? max_clusters : sm_count;   // co-resident CTAs (pairs)
  const int grid = static_cast<int>((units < slots ? units : slots) * (PAIR ? 2 : 1));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, p);
  count_launches(1);
  return cuda_ok(e == cudaSuccess ? cudaGetLastError() : e);
}

// Which dense variant runs (see bsmma_set_dense_variant): CTA pairs or single CTAs.
bool use_pair(int num_m_tiles) {
  const int v = dense_variant();
  if (v == 1) return false;
  if (v == 2) return num_m_tiles >= 1;
  return kPairDefault && num_m_tiles >= 2;
}

}  // namespace

bsmma_status launch_mx_gemm(const void* A, const uint8_t* sfa, const void* B, const uint8_t* sfb,
                            void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                            bsmma_fmt a_fmt, bsmma_fmt b_fmt, cudaStream_t stream) {
  if (dense_variant() >= 3) return BSMMA_ERR_UNSUPPORTED;   // takes the wide scale layouts
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  constexpr int BN = 256;
  const bool fp4 = (a_fmt == BSMMA_E2M1);
  const uint64_t kbytes = fp4 ? static_cast<uint64_t>(K / 2) : static_cast<uint64_t>(K);
  CUtensorMap ta, tb;
  if (layout == BSMMA_TN)
    st = encode_tmap_u8(&ta, A, M, K, M, 128, 128);
  else
    st = encode_tmap_u8(&ta, A, kbytes, M, kbytes, 128, 128);
  if (st != BSMMA_OK) return st;
  const int num_m_tiles = static_cast<int>((M + kBM - 1) / kBM);
  const bool pair = use_pair(num_m_tiles);
  if (layout == BSMMA_NT)
    st = encode_tmap_u8(&tb, B, kbytes, N, kbytes, 128, pair ? 128 : BN);
  else
    st = encode_tmap_u8(&tb, B, N, K, N, 128, 128);
  if (st != BSMMA_OK) return st;

  DenseParams p;
  p.sfa = sfa;
  p.sfb = sfb;
  p.D = static_cast<__nv_bfloat16*>(D);
  p.M = M;
  p.N = N;
  p.sfa_kg = 2 * ((K / 32 + 7) / 8);   // block groups per row block of the tiled layout
  p.sfb_kg = p.sfa_kg;
  p.num_m_tiles = num_m_tiles;
  p.num_n_tiles = static_cast<int>((N + BN - 1) / BN);
  p.num_k_stages = static_cast<int>((static_cast<int64_t>(kbytes) + 127) / 128);
  const uint32_t af = fp4 ? 1u : static_cast<uint32_t>(a_fmt);   // kind::mxf4 codes E2M1 as 1
  const uint32_t bf = fp4 ? 1u : static_cast<uint32_t>(b_fmt);
  p.idesc = idesc_block_scaled(af, bf, layout == BSMMA_TN, layout != BSMMA_NT, kBM, BN);
  p.status = dev->status;
  p.limit_ns = wait_limit_ns();
  const int sms = dev->sm_count;
  if (pair) {
    if (fp4) return launch_dense<BN, true, false, false, true>(ta, tb, p, sms, stream);
    switch (layout) {
      case BSMMA_NT: return launch_dense<BN, false, false, false, true>(ta, tb, p, sms, stream);
      case BSMMA_NN: return launch_dense<BN, false, false, true, true>(ta, tb, p, sms, stream);
      default:       return launch_dense<BN, false, true, true, true>(ta, tb, p, sms, stream);
    }
  }
  if (fp4) return launch_dense<BN, true, false, false, false>(ta, tb, p, sms, stream);
  switch (layout) {
    case BSMMA_NT: return launch_dense<BN, false, false, false, false>(ta, tb, p, sms, stream);
    case BSMMA_NN: return launch_dense<BN, false, false, true, false>(ta, tb, p, sms, stream);
    default:       return launch_dense<BN, false, true, true, false>(ta, tb, p, sms, stream);
  }
}

}  // namespace bsmma
