// probe_mma_rate.cu -- standalone throughput probe of the tcgen05 instructions the
// GEMM kernels use: back-to-back MMAs (block-scaled and plain, one CTA and SM
// pairs) on data resident in shared memory, with and without scale-factor copies
// into tensor memory.  No TMA, no epilogue: it measures the ceiling a kernel built
// from these instructions can reach.  One CTA per SM; every access stays inside the
// CTA's shared memory and a 512-column tensor-memory allocation, and every wait is
// bounded.  Not part of libbsmma; build with
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -I block_scaled_precision_mma_gb300/csrc -o probe_mma_rate \
//        block_scaled_precision_mma_gb300/csrc/probe_mma_rate.cu
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx.cuh"
using namespace bsmma;

// mode: 0 mxf8f6f4 N256 ; 1 mxf8f6f4 N256 + 3 cp per 4 MMAs ; 2 f8f6f4 N256 ; 3 mxf4 N256 ;
//       4 mxf4 N256 + 6 cp per 4 MMAs ; 5 mxf8f6f4 N128 ; 6 mxf8f6f4 N256 + 1 cp per 4 MMAs ;
//       7, 8 mxf8f6f4 N256 + 128x256b copies ; 9 f8f6f4 N128
__global__ void __launch_bounds__(128, 1) probe(int mode, int iters, int* status, unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;              // 16 KB
  uint8_t* sB = smem + 16384;      // 32 KB
  uint8_t* sSF = smem + 49152;     // 4 KB of scale atoms
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  for (int i = threadIdx.x; i < (49152 + 4096) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem)[i] = (i * 4 >= 49152) ? 0x7f7f7f7fu : 0x38383838u;
  if (threadIdx.x == 0) { mbar_init(&bar, 1); abort_flag = 0; fence_mbar_init(); }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x < 32) { tmem_alloc(&tslot, 512); tmem_relinquish(); }
  tc_fence_before(); __syncthreads(); tc_fence_after();
  const uint32_t tmem = tslot;
  if (threadIdx.x == 0) {
    const int n = (mode == 5 || mode == 9) ? 128 : 256;
    const bool fp4 = (mode == 3 || mode == 4);
    uint32_t idesc = (mode == 2 || mode == 9) ? idesc_f8f6f4(0, 0, 0, 0, 128, n)
                   : idesc_block_scaled(fp4 ? 1 : 0, fp4 ? 1 : 0, 0, 0, 128, n);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB), s0 = smem_u32(sSF);
    const int ncp = (mode == 1) ? 3 : (mode == 4) ? 6 : (mode == 6) ? 1 : 0;
    unsigned long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      for (int c = 0; c < ncp; ++c) tc_cp_sf(tmem + 256 + (it & 3) * 16 + c * 4, make_sdesc(s0 + c * 512, 0, 128, 0));
      if (mode == 7 && (it & 3) == 0)
        for (int c = 0; c < 3; ++c)
          asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(tmem + 320 + c * 8), "l"(make_sdesc(s0, 128, 256, 0)) : "memory");
      if (mode == 8)
        asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(tmem + 320), "l"(make_sdesc(s0, 128, 256, 0)) : "memory");
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t ad = make_sdesc(a0 + j * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = make_sdesc(b0 + j * 32, 16, 1024, kSwizzle128B);
        if (mode == 2 || mode == 9) mma_f8f6f4(tmem, ad, bd, idesc, 1);
        else if (fp4) mma_mxf4(tmem, ad, bd, idesc | idesc_sf_id((j & 1) * 2, (j & 1) * 2), tmem + 256, tmem + 288, 1);
        else mma_mxf8f6f4(tmem, ad, bd, idesc | idesc_sf_id(j, j), tmem + 256, tmem + 288, 1);
      }
    }
    tc_commit(&bar);
    mbar_wait(&bar, 0, 2000000000ull, &abort_flag, status);
    unsigned long long t1 = clock64();
    if (blockIdx.x == 0) *cycles = t1 - t0;
  }
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

// Pair probe: cta_group::2 MMAs over a 2-CTA cluster (256-row A split across the pair).
// mode: 0 mxf8f6f4 256x256x32 ; 1 + 3 cp.cta_group::2 per 4 MMAs ; 2 f8f6f4 256x256x32 ; 3 mxf4 256x256x64 ;
//       4 mxf8f6f4 with the dense kernel's scale addresses and copies (one 128x256b copy of
//         column scales per 4 MMAs, one of row scales per 8) ; 5 the same addresses, no copies ;
//       6 mxf4 with the dense kernel's copies (two column-scale copies and one row-scale copy per 4 MMAs) ;
//       7 f8f6f4 256x128x32 ; 8 mode 0 again (drift check) ; 9 mode 4 over three rotating stage
//       buffers ; 10 mode 9 with random operand codes and scales ; 11 f8f6f4 256x256x32 over three
//       rotating buffers ; 12, 13 mode 9 over five and two buffers ; 14 mode 12 with a commit per
//       iteration ; 15 mode 12 while three warps per CTA write shared memory ; 16 both
__global__ void __launch_bounds__(128, 1) probe2(int mode, int iters, int* status, unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;              // 16 KB
  uint8_t* sB = smem + 16384;      // 16 KB (half of B)
  uint8_t* sSF = smem + 49152;     // moved to 96 KB in modes 9-10
  __shared__ uint64_t bar;
  __shared__ uint64_t stage_bar;            // per-iteration commits of modes 14 and 16
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  __shared__ volatile int stop_writers;     // ends the shared-memory writers of modes 15 and 16
  // modes 9-13 rotate over 32 KB stage buffers (A then B) with the scale source after them;
  // mode 10 fills them with hashed random E4M3 codes and E8M0 scales in [120, 133]
  const bool rot = mode >= 9;
  const int nbuf = (mode == 12 || mode >= 14) ? 5 : mode == 13 ? 2 : 3;   // stage buffers of the rotating modes
  if (rot) sSF = smem + nbuf * 32768;
  const int fill_words = rot ? (nbuf * 32768 + 4096) / 4 : (49152 + 4096) / 4;
  const int sf_word0 = rot ? nbuf * 32768 / 4 : 49152 / 4;
  for (int i = threadIdx.x; i < fill_words; i += blockDim.x) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u;
    h ^= h >> 15; h *= 2246822519u; h ^= h >> 13;
    uint32_t v;
    if (i >= sf_word0) v = (mode == 10) ? 0x78787878u + (h % 14u) * 0x01010101u : 0x7f7f7f7fu;
    else v = (mode == 10) ? (h & 0x77777777u) : 0x38383838u;
    reinterpret_cast<uint32_t*>(smem)[i] = v;
  }
  uint32_t rank; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  if (threadIdx.x == 0) { mbar_init(&bar, 1); mbar_init(&stage_bar, 1); abort_flag = 0; stop_writers = 0; fence_mbar_init(); }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tslot)), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before(); __syncthreads(); cluster_sync(); tc_fence_after();
  const uint32_t tmem = tslot;
  if (threadIdx.x == 0 && rank == 0) {
    const bool fp4 = mode == 3 || mode == 6;
    uint32_t idesc = (mode == 2 || mode == 11) ? idesc_f8f6f4(0, 0, 0, 0, 256, 256)
                   : (mode == 7) ? idesc_f8f6f4(0, 0, 0, 0, 256, 128)
                   : idesc_block_scaled(fp4 ? 1 : 0, fp4 ? 1 : 0, 0, 0, 256, 256);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB), s0 = smem_u32(sSF);
    unsigned long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      if (mode == 1)
        for (int c = 0; c < 3; ++c)
          asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(tmem + 256 + (it & 3) * 16 + c * 4), "l"(make_sdesc(s0 + c * 512, 0, 128, 0)) : "memory");
      // the dense kernel's layout: row-scale chunks in columns 256-271 (two slots of 8),
      // column-scale blocks in columns 288-319 (four slots of 8)
      const int kgs = (mode == 6) ? 2 : 1;                 // column-scale blocks per 4 MMAs
      const int spc = (mode == 6) ? 1 : 2;                 // iterations per row-scale chunk
      const uint32_t sfa_t = tmem + 256 + ((it / spc) & 1) * 8;
      const int sub = it % spc;
      const bool kcp = mode == 4 || mode == 6 || (mode >= 9 && mode != 11);
      if (kcp && sub == 0)
        asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(sfa_t), "l"(make_sdesc(s0, 128, 256, 0)) : "memory");
      uint32_t sfb_t[2];
      for (int g = 0; g < kgs; ++g) {
        sfb_t[g] = tmem + 288 + ((it * kgs + g) & 3) * 8;
        if (kcp)
          asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(sfb_t[g]), "l"(make_sdesc(s0, 128, 256, 0)) : "memory");
      }
      const uint32_t ab = rot ? smem_u32(smem) + (it % nbuf) * 32768 : a0;
      const uint32_t bb = rot ? ab + 16384 : b0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t ad = make_sdesc(ab + j * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = make_sdesc(bb + j * 32, 16, 1024, kSwizzle128B);
        if (mode == 2 || mode == 7 || mode == 11)
          asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(1) : "memory");
        else if (mode == 6)
          asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc | idesc_sf_id((j & 1) * 2, (j & 1) * 2)), "r"(1), "r"(sfa_t + 4 * (j >> 1)), "r"(sfb_t[j >> 1]) : "memory");
        else if (mode == 4 || mode == 5 || (mode >= 9 && mode != 11))
          asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc | idesc_sf_id(j, j)), "r"(1), "r"(sfa_t + 4 * sub), "r"(sfb_t[0]) : "memory");
        else if (fp4)
          asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc | idesc_sf_id((j & 1) * 2, (j & 1) * 2)), "r"(1), "r"(tmem + 256), "r"(tmem + 288) : "memory");
        else
          asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc | idesc_sf_id(j, j)), "r"(1), "r"(tmem + 256), "r"(tmem + 288) : "memory");
      }
      if (mode == 14 || mode == 16)   // a commit per stage, as the GEMM kernel makes
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(smem_u32(&stage_bar)), "h"((uint16_t)3) : "memory");
    }
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(smem_u32(&bar)), "h"((uint16_t)1) : "memory");
    mbar_wait(&bar, 0, 2000000000ull, &abort_flag, status);
    unsigned long long t1 = clock64();
    if (blockIdx.x == 0) *cycles = t1 - t0;
    stop_writers = 1;
    uint32_t peer_flag;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 1;" : "=r"(peer_flag) : "r"(smem_u32((const void*)&stop_writers)));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_flag), "r"(1) : "memory");
  }
  if ((mode == 15 || mode == 16) && threadIdx.x >= 32) {
    // warps 1-3 of both CTAs write 16-byte vectors into a 32 KB region of their own shared
    // memory (after the stage buffers and scales) until the MMA thread is done, standing in
    // for the operand traffic TMA writes in the GEMM kernel; bounded by an iteration limit
    uint4* region = reinterpret_cast<uint4*>(smem + nbuf * 32768 + 4096);
    const uint4 v = make_uint4(threadIdx.x, 1, 2, 3);
    for (int i = 0; i < (1 << 22); ++i) {
      region[(i * 96 + threadIdx.x - 32) & 2047] = v;
      if ((i & 63) == 0 && stop_writers) break;
    }
  }
  __syncthreads();
  cluster_sync();
  if (threadIdx.x < 32) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
  cluster_sync();
}

int main() {
  int* status; unsigned long long* cyc;
  cudaMalloc(&status, 4); cudaMemset(status, 0, 4); cudaMalloc(&cyc, 8);
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int smem = 1024 + 49152 + 4096 + 70000;   // one CTA per SM
  cudaFuncSetAttribute(probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const char* names[] = {"mxf8f6f4 128x256x32", "mxf8f6f4 128x256x32 + 3 cp/4 MMA", "f8f6f4 128x256x32",
                         "mxf4 128x256x64", "mxf4 128x256x64 + 6 cp/4 MMA", "mxf8f6f4 128x128x32",
                         "mxf8f6f4 128x256x32 + 1 cp/4 MMA", "mxf8f6f4 + 3 cp.128x256b/16 MMA",
                         "mxf8f6f4 + 1 cp.128x256b/4 MMA", "f8f6f4 128x128x32"};
  for (int mode = 0; mode < 10; ++mode) {
    const int iters = 4096;
    probe<<<sms, 128, smem>>>(mode, 64, status, cyc);   // warm-up
    cudaDeviceSynchronize();
    cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
    cudaEventRecord(e0);
    probe<<<sms, 128, smem>>>(mode, iters, status, cyc);
    cudaEventRecord(e1); cudaError_t err = cudaDeviceSynchronize();
    float ms; cudaEventElapsedTime(&ms, e0, e1);
    unsigned long long c; cudaMemcpy(&c, cyc, 8, cudaMemcpyDeviceToHost);
    int st; cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost);
    const double n = (mode == 5 || mode == 9) ? 128 : 256, k = (mode == 3 || mode == 4) ? 64 : 32;
    const double macs = 128.0 * n * k * 4 * iters;
    printf("%-36s err=%d status=%d  %.1f cycles/MMA  %.0f MAC/clk/SM  %.1f TFLOPS (all SMs, event)\n",
           names[mode], (int)err, st, (double)c / (4.0 * iters), macs / (double)c, 2 * macs * sms / (ms * 1e-3) / 1e12);
  }
  const char* names2[] = {"pair mxf8f6f4 256x256x32", "pair mxf8f6f4 + 3 cp.cta_group::2/4 MMA",
                          "pair f8f6f4 256x256x32", "pair mxf4 256x256x64",
                          "pair mxf8f6f4 + kernel's 128x256b copies", "pair mxf8f6f4 kernel addresses",
                          "pair mxf4 + kernel's 128x256b copies", "pair f8f6f4 256x128x32",
                          "pair mxf8f6f4 256x256x32 (again)", "pair kernel pattern, 3 stage buffers",
                          "pair kernel pattern, 3 buffers, random data", "pair f8f6f4, 3 stage buffers",
                          "pair kernel pattern, 5 stage buffers", "pair kernel pattern, 2 stage buffers",
                          "pair 5 buffers + commit per stage", "pair 5 buffers + smem writers",
                          "pair 5 buffers + commits + writers"};
  const int smem2 = 1024 + 5 * 32768 + 4096 + 32768;   // one CTA per SM: five stage buffers + writer region
  cudaFuncSetAttribute(probe2, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
  for (int mode0 = 0; mode0 < 17; ++mode0) {
    const int mode = mode0 == 8 ? 0 : mode0;
    const int iters = 4096;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2; attr[0].val.clusterDim.y = 1; attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(sms / 2 * 2, 1, 1); cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = smem2; cfg.attrs = attr; cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, probe2, mode, 64, status, cyc);
    cudaDeviceSynchronize();
    cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
    cudaEventRecord(e0);
    cudaLaunchKernelEx(&cfg, probe2, mode, iters, status, cyc);
    cudaEventRecord(e1); cudaError_t err = cudaDeviceSynchronize();
    float ms; cudaEventElapsedTime(&ms, e0, e1);
    unsigned long long c; cudaMemcpy(&c, cyc, 8, cudaMemcpyDeviceToHost);
    int st; cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost);
    const double k = (mode == 3 || mode == 6) ? 64 : 32;
    const double macs = 256.0 * (mode == 7 ? 128 : 256) * k * 4 * iters;   // per pair
    printf("%-40s err=%d status=%d  %.1f cycles/MMA  %.0f MAC/clk/SM  %.1f TFLOPS (all SMs, event)\n",
           names2[mode0], (int)err, st, (double)c / (4.0 * iters), macs / 2 / (double)c,
           2 * macs * (sms / 2) / (ms * 1e-3) / 1e12);
  }
  return 0;
}
