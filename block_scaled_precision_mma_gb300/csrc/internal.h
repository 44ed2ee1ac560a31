// internal.h -- host-side interfaces shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <functional>
#include <string>
#include <vector>

#include "bsmma.h"

namespace bsmma {

// Per-device facts the launchers need.
struct DeviceInfo {
  int device;
  int sm_count;
  int* status;   // device address of the latched device-status word
};

// Info for the current device (initialised on first use).  Returns nullptr and
// sets *err on failure.
const DeviceInfo* current_device(bsmma_status* err);

uint64_t wait_limit_ns();
int dense_variant();   // 0 automatic, 1 single CTAs, 3 SM-pair MMAs
int grouped_tile_width();   // 0 automatic, 128 or 256
int grouped_variant();      // grouped BF16: 0 automatic, 1 one CTA per tile, 3 SM-pair tiles
void count_launches(int n);

// Encodes a 2-D uint8 tensor map with 128-byte swizzle: `inner` contiguous bytes per
// row, `outer` rows `row_stride` bytes apart, box of box_inner x box_outer.
bsmma_status encode_tmap_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride, uint32_t box_inner, uint32_t box_outer);

// Host-side argument checks shared by the dense entry points.
bsmma_status validate_dense(const void* A, const void* sA, const void* B, const void* sB,
                            const void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                            bsmma_fmt a_fmt, bsmma_fmt b_fmt);

// Encodes a 2-D tensor map of 32-bit words without swizzle: `inner` words per row,
// `outer` rows, box of box_inner x box_outer words.
bsmma_status encode_tmap_words(CUtensorMap* map, const void* base, uint64_t inner,
                               uint64_t outer, uint32_t box_inner, uint32_t box_outer);

// Tiled scale layouts (role 0 scales of op(A) rows, role 1 scales of op(B) rows); a
// null source or destination skips that operand.
int64_t wide_scale_bytes(int64_t rows, int64_t kblocks, int role);
bsmma_status launch_wide_relayout(const uint8_t* sa, int64_t rows_a, uint8_t* out_a,
                                  const uint8_t* sb, int64_t rows_b, uint8_t* out_b,
                                  int64_t kblocks, cudaStream_t stream);

// The dense SM-pair kernel's split workspace for (current device, stream): arrival
// counters [#SMs][8 epilogue warps] (zero between launches) and partial-sum slots
// [2 * #SMs][128 x 256 FP32].
// Allocated, its counters zeroed, by the first call on a stream outside a capture
// (inside one it returns BSMMA_ERR_WORKSPACE, and the caller runs without splits); a
// fixed size per device.
bsmma_status split_workspace(cudaStream_t stream, float** part, int** arrivals);

// Launchers (arguments already validated by the entry points).
// bias: BF16 [N] or nullptr; act: bsmma_activation (0 = none).  may_allocate: false keeps
// the dense GEMM off the autotuner's timing runs (it then takes a stored choice, else the
// SM-pair kernel) and off the split workspace (units are not split).
bsmma_status launch_mx_gemm(const void* A, const uint8_t* sfa, const void* B, const uint8_t* sfb,
                            void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                            bsmma_fmt a_fmt, bsmma_fmt b_fmt, cudaStream_t stream,
                            const void* bias = nullptr, int act = 0, bool may_allocate = true);
bsmma_status launch_mx_gemm_2sm(const void* A, const uint8_t* sfa, const void* B,
                                const uint8_t* sfb, void* D, int64_t M, int64_t N, int64_t K,
                                bsmma_layout layout, bsmma_fmt a_fmt, bsmma_fmt b_fmt,
                                cudaStream_t stream, const void* bias = nullptr, int act = 0,
                                bool may_split = true);
// packed: W is in the grouped_fp8_pack_weights layout.
bsmma_status launch_grouped(const uint8_t* X, const float* sX, const uint8_t* W, const float* sW,
                            void* D, const int64_t* m_sizes, int64_t total_M, int G, int64_t N,
                            int64_t K, cudaStream_t stream, bool packed = false);
bsmma_status launch_grouped_bf16(const void* X, const void* W, void* D, const int64_t* m_sizes,
                                 int64_t total_M, int G, int64_t N, int64_t K,
                                 cudaStream_t stream);
bsmma_status launch_pack_weights(const uint8_t* W, int64_t G, int64_t N, int64_t K, uint8_t* Wp,
                                 cudaStream_t stream);

// Quantisers (arguments already validated by the entry points).
bsmma_status launch_mx_quantize(const void* x, bool f32, int64_t rows, int64_t cols, bsmma_fmt fmt,
                                bool colwise, uint8_t* codes, uint8_t* scales, cudaStream_t stream);
bsmma_status launch_group_quantize(const void* x, bool f32, int64_t total_M, int64_t K,
                                   const int64_t* m_sizes, int G, uint8_t* codes, float* scales,
                                   cudaStream_t stream);
bsmma_status launch_block_quantize(const void* w, bool f32, int64_t G, int64_t N, int64_t K,
                                   uint8_t* codes, float* scales, cudaStream_t stream);

// Autotuning (opt-in): the cached choice for `key`, else -- when tuning is enabled and the
// stream is not capturing -- the fastest of `candidates` timed with `launch`, else
// `fallback`.
int64_t next_pow2(int64_t v);
// The stored choice for `key` when tuning is enabled, else -1; never times anything.
int autotune_cached(const std::string& key);
int autotune_pick(const std::string& key, const std::vector<int>& candidates, int fallback,
                  cudaStream_t stream, const std::function<bsmma_status(int)>& launch);

inline bsmma_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? BSMMA_OK : BSMMA_ERR_CUDA; }

}  // namespace bsmma
