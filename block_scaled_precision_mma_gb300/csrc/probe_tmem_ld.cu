// probe_tmem_ld.cu -- standalone throughput probe of tensor-memory reads
// (tcgen05.ld.sync.aligned.32x32b.xN): the rate at which warps move FP32 accumulator
// columns from tensor memory into registers, which bounds any epilogue or software
// fold that reads whole accumulators.  One CTA per SM with W warps; warp w reads lane
// quarter w % 4 and its share of a 512-column allocation, L loads of N columns in
// flight before each wait.  Every access stays inside the CTA's allocation.  Not part
// of libbsmma; build with
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -I block_scaled_precision_mma_gb300/csrc -o probe_tmem_ld \
//        block_scaled_precision_mma_gb300/csrc/probe_tmem_ld.cu
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx.cuh"
using namespace bsmma;

__device__ __forceinline__ void ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, "
      "%45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, "
      "%62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}

// Orders the use of a loaded register after the wait (volatile asm statements keep their order).
__device__ __forceinline__ void after_wait(uint32_t& x) { asm volatile("" : "+r"(x)); }

// Each warp: iters x [L loads of N columns, one wait, fold the values into a checksum].
template <int N, int L>
__global__ void tmem_read(int iters, int warps, unsigned long long* cycles, uint32_t* sink) {
  __shared__ uint32_t tslot;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    tmem_alloc(&tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tslot;
  const int q = warp & 3;
  const int per_quarter = warps / 4;                 // warps sharing a lane quarter
  const int slice = 512 / per_quarter;               // columns of this warp
  const uint32_t base = tmem + (static_cast<uint32_t>(q * 32) << 16) + (warp >> 2) * slice;
  uint32_t acc = 0;
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    const uint32_t off = static_cast<uint32_t>((it * N * L) % slice);
    uint32_t r[L][N];
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const uint32_t a = base + (off + l * N) % slice;
      if constexpr (N == 64) ld_x64(a, r[l]);
      else if constexpr (N == 32) tmem_ld32(a, r[l]);
      else tmem_ld16(a, r[l]);
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int l = 0; l < L; ++l)
#pragma unroll
      for (int i = 0; i < N; ++i) {
        after_wait(r[l][i]);
        acc += r[l][i];
      }
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  if (threadIdx.x == 0 && blockIdx.x == 0) *cycles = t1 - t0;
  sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int N, int L>
void run(int warps, int sms, unsigned long long* cyc, uint32_t* sink) {
  const int iters = 4096;
  auto k = tmem_read<N, L>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 150000);
  k<<<sms, warps * 32, 150000>>>(64, warps, cyc, sink);   // warm-up; 150 KB keeps one CTA per SM
  cudaDeviceSynchronize();
  k<<<sms, warps * 32, 150000>>>(iters, warps, cyc, sink);
  cudaError_t err = cudaDeviceSynchronize();
  unsigned long long c = 0;
  cudaMemcpy(&c, cyc, 8, cudaMemcpyDeviceToHost);
  const double bytes = static_cast<double>(iters) * L * N * 4 * 32 * warps;   // per SM
  printf("warps %2d  32x32b.x%-3d x %d in flight  err=%d  %8.1f bytes/clk/SM  (%.1f cycles per wait)\n",
         warps, N, L, static_cast<int>(err), bytes / static_cast<double>(c),
         static_cast<double>(c) / iters);
}

int main() {
  int sms;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* cyc;
  uint32_t* sink;
  cudaMalloc(&cyc, 8);
  cudaMalloc(&sink, static_cast<size_t>(sms) * 512 * 4);
  for (int warps : {4, 8, 16}) {
    run<16, 1>(warps, sms, cyc, sink);
    run<16, 2>(warps, sms, cyc, sink);
    run<32, 1>(warps, sms, cyc, sink);
    run<32, 2>(warps, sms, cyc, sink);
    run<32, 4>(warps, sms, cyc, sink);
    run<64, 1>(warps, sms, cyc, sink);
    run<64, 2>(warps, sms, cyc, sink);
  }
  return 0;
}
