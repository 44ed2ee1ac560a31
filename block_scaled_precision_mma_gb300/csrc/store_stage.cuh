// store_stage.cuh -- the staged output stage of the dense SM-pair kernel: BF16 pieces
// written to shared memory leave through TMA tensor stores, tracked by the issuing
// thread's bulk async-groups.  Device helpers plus the host encoder of D's tensor map.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "bsmma.h"
#include "ptx.cuh"

namespace bsmma {

// Encodes a 2-D BF16 tensor map for stores with 64-byte swizzle: `cols` contiguous BF16
// values per row (a multiple of 8), `rows` rows, box of box_cols x box_rows.
bsmma_status encode_tmap_bf16_out(CUtensorMap* map, const void* base, uint64_t cols,
                                  uint64_t rows, uint32_t box_cols, uint32_t box_rows);

// 2-D tiled tensor store from shared memory (this CTA's), tracked by the thread's bulk
// async-group; coordinates past the tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* src, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(c0), "r"(c1), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of the thread's bulk async-groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N of the thread's bulk async-groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the async proxy
// (tensor copies that read them).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace bsmma
