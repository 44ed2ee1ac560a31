// noalloc.cu -- mx_gemm for callers that cannot allocate device memory.
//
// mx_gemm rearranges the E8M0 scales into a workspace that the library allocates
// with cudaMalloc the first time a stream needs it.  Some callers cannot allow
// that: code running while a CUDA graph is being captured, code that runs under
// a framework's own memory pool or a fixed memory budget, and code that must not
// synchronise (cudaMalloc/cudaFree can).  mx_gemm_noalloc does the same work with
// the scales placed in a fixed array in device memory that belongs to the
// library module, so it never allocates.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace bsmma {
namespace {

constexpr int64_t kNoAllocScratchBytes = BSMMA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Scratch shared by every mx_gemm_noalloc call on a device; it lives as long as
// the library is loaded, on every device that loads it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
uint8_t* g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device.  The array's name
// in host code is only a host-side stand-in, so the address is asked of the
// runtime once per device, with that device current.
bsmma_status noalloc_scratch(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSMMA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return BSMMA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return BSMMA_OK;
}

}  // namespace
}  // namespace bsmma

using namespace bsmma;

extern "C" {

bsmma_status mx_gemm_noalloc(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                             void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                             bsmma_fmt a_fmt, bsmma_fmt b_fmt, bsmma_stream stream) {
  bsmma_status st = validate_dense(A, sA, B, sB, D, M, N, K, layout, a_fmt, b_fmt);
  if (st != BSMMA_OK || M == 0 || N == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_ok(cudaMemsetAsync(D, 0, static_cast<size_t>(M * N * 2), s));
  const int64_t bytes_a = (wide_scale_bytes(M, K / 32, 0) + 255) / 256 * 256;
  const int64_t bytes_b = wide_scale_bytes(N, K / 32, 1);
  if (bytes_a + bytes_b > kNoAllocScratchBytes) return BSMMA_ERR_SCRATCH_LIMIT;
  uint8_t* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != BSMMA_OK) return st;
  // every byte of both tiled buffers (padding included) is rewritten here, so the
  // previous call's contents never leak into this one
  st = launch_wide_relayout(sA, M, scratch, sB, N, scratch + bytes_a, K / 32, s);
  if (st != BSMMA_OK) return st;
  // no tuning runs (they would create events and synchronise the stream) and no split
  // units (their workspace is allocated on first use)
  return launch_mx_gemm(A, scratch, B, scratch + bytes_a, D, M, N, K, layout, a_fmt, b_fmt, s,
                        nullptr, 0, /*may_allocate=*/false);
}

}  // extern "C"
