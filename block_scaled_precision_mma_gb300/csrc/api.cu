// api.cu -- the C ABI: argument validation, per-device state, the scale workspace,
// the device-status word, tensor-map encoding and the wait-timeout probe.
//
// Validation follows the source pages' preconditions: 64-bit extents everywhere
// (launch arguments that overflowed 32 bits: "Experimental FlyDSL GEMM backend for
// TE PyTorch", BF16 skipped shapes; "Add FlyDSL grouped groupwise FP8 GEMM for
// ROCm", the commit passing operands with their natural shape), N and K multiples
// of 128 and m_sizes of length G for the grouped GEMM (same page, introduction and
// the format/rank check commit), OCP FP8 formats only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "store_stage.cuh"

namespace bsmma {

// Latched device-side status, one per device that loads the library.
__device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];
std::atomic<int64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_dense_variant{0};
std::atomic<int> g_grouped_width{0};
std::atomic<int> g_grouped_variant{0};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

struct Workspace {
  int device;
  cudaStream_t stream;
  void* ptr;
  int64_t bytes;
  bool captured;   // handed to a kernel launch recorded into a CUDA graph
};
std::vector<Workspace> g_ws;
// The dense kernel's split workspace of one (device, stream): a fixed size per device, its
// arrival counters zero between launches.
struct SplitWorkspace {
  int device;
  cudaStream_t stream;
  void* ptr;
  int64_t counter_bytes;
};
std::vector<SplitWorkspace> g_sws;
// Buffers replaced by a larger one after a graph capture used them: a replay of that
// graph still reads and writes them, so they stay allocated until the process exits.
std::vector<void*> g_ws_kept;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

const DeviceInfo* current_device(bsmma_status* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = BSMMA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev_ready[dev]) {
    DeviceInfo d;
    d.device = dev;
    void* status = nullptr;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaGetSymbolAddress(&status, g_device_status) != cudaSuccess) {
      *err = BSMMA_ERR_CUDA;
      return nullptr;
    }
    d.status = static_cast<int*>(status);
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
  }
  return &g_dev[dev];
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }
int dense_variant() { return g_dense_variant.load(); }
int grouped_tile_width() { return g_grouped_width.load(); }
int grouped_variant() { return g_grouped_variant.load(); }
void count_launches(int n) { g_launches += n; }

bsmma_status encode_tmap_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride, uint32_t box_inner, uint32_t box_outer) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return BSMMA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSMMA_OK : BSMMA_ERR_INVALID_ARG;
}

bsmma_status encode_tmap_words(CUtensorMap* map, const void* base, uint64_t inner,
                               uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return BSMMA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSMMA_OK : BSMMA_ERR_INVALID_ARG;
}

bsmma_status encode_tmap_bf16_out(CUtensorMap* map, const void* base, uint64_t cols,
                                  uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return BSMMA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSMMA_OK : BSMMA_ERR_INVALID_ARG;
}

namespace {

__global__ void wait_probe_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait must give up and latch a timeout.
  if (threadIdx.x == 0) mbar_wait(&bar, 0, limit_ns, &abort_flag, status);
}

constexpr int64_t kMaxTmaDim = (int64_t(1) << 32) - 1;
constexpr int64_t kMaxStride = (int64_t(1) << 40) - 16;

// Workspace of at least `bytes` for (current device, stream).
bsmma_status get_workspace(int64_t bytes, cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSMMA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace* w = nullptr;
  for (auto& e : g_ws)
    if (e.device == dev && e.stream == stream) w = &e;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return BSMMA_ERR_CUDA;
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  if (w && w->bytes >= bytes) {
    if (capturing) w->captured = true;
    *out = w->ptr;
    return BSMMA_OK;
  }
  if (capturing) return BSMMA_ERR_WORKSPACE;
  int64_t grow = bytes + bytes / 4 + 4096;
  void* p = nullptr;
  if (cudaMalloc(&p, static_cast<size_t>(grow)) != cudaSuccess) return BSMMA_ERR_CUDA;
  if (w) {
    if (w->captured) {
      g_ws_kept.push_back(w->ptr);   // a captured graph may still be replayed on it
    } else {
      // earlier kernels on this stream may still read the old buffer
      if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaFree(p);
        return BSMMA_ERR_CUDA;
      }
      cudaFree(w->ptr);
    }
    w->ptr = p;
    w->bytes = grow;
    w->captured = false;
  } else {
    g_ws.push_back(Workspace{dev, stream, p, grow, false});
  }
  *out = p;
  return BSMMA_OK;
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

}  // namespace

bsmma_status split_workspace(cudaStream_t stream, float** part, int** arrivals) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& e : g_sws)
    if (e.device == dev->device && e.stream == stream) {
      *arrivals = static_cast<int*>(e.ptr);
      *part = reinterpret_cast<float*>(static_cast<uint8_t*>(e.ptr) + e.counter_bytes);
      return BSMMA_OK;
    }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return BSMMA_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return BSMMA_ERR_WORKSPACE;
  const int64_t sms = dev->sm_count;
  const int64_t counter_bytes = align_up(sms * 8 * 4, 256);
  const int64_t bytes = counter_bytes + 2 * sms * 128 * 256 * 4;
  void* p = nullptr;
  if (cudaMalloc(&p, static_cast<size_t>(bytes)) != cudaSuccess) return BSMMA_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, static_cast<size_t>(counter_bytes), stream) != cudaSuccess) {
    cudaFree(p);
    return BSMMA_ERR_CUDA;
  }
  g_sws.push_back(SplitWorkspace{dev->device, stream, p, counter_bytes});
  *arrivals = static_cast<int*>(p);
  *part = reinterpret_cast<float*>(static_cast<uint8_t*>(p) + counter_bytes);
  return BSMMA_OK;
}

bsmma_status validate_dense(const void* A, const void* sA, const void* B, const void* sB,
                            const void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                            bsmma_fmt a_fmt, bsmma_fmt b_fmt) {
  if (M < 0 || N < 0 || K < 0 || K % 32 != 0) return BSMMA_ERR_INVALID_ARG;
  if (layout < BSMMA_NT || layout > BSMMA_TN) return BSMMA_ERR_INVALID_ARG;
  if (a_fmt < BSMMA_E4M3 || a_fmt > BSMMA_E2M1 || b_fmt < BSMMA_E4M3 || b_fmt > BSMMA_E2M1)
    return BSMMA_ERR_INVALID_ARG;
  const bool fp4a = a_fmt == BSMMA_E2M1, fp4b = b_fmt == BSMMA_E2M1;
  if (fp4a != fp4b) return BSMMA_ERR_UNSUPPORTED;
  if (fp4a && layout != BSMMA_NT) return BSMMA_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return BSMMA_OK;
  if (!D) return BSMMA_ERR_INVALID_ARG;
  if (N % 8 != 0 || !aligned16(D)) return BSMMA_ERR_MISALIGNED;
  if (K == 0) return BSMMA_OK;
  if (!A || !B || !sA || !sB) return BSMMA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(sA) || !aligned16(sB))
    return BSMMA_ERR_MISALIGNED;
  if (layout != BSMMA_NT && N % 16 != 0) return BSMMA_ERR_MISALIGNED;
  if (layout == BSMMA_TN && M % 16 != 0) return BSMMA_ERR_MISALIGNED;
  if (M > kMaxTmaDim || N > kMaxTmaDim || K > kMaxTmaDim) return BSMMA_ERR_INVALID_ARG;
  // tensor-copy coordinates are 32-bit signed
  if (M >= INT32_MAX || N >= INT32_MAX || K >= INT32_MAX) return BSMMA_ERR_INVALID_ARG;
  if (M > kMaxStride || N > kMaxStride || K > kMaxStride) return BSMMA_ERR_INVALID_ARG;
  // tile ids are 32-bit
  if ((M + 127) / 128 * ((N + 255) / 256) > INT32_MAX / 2) return BSMMA_ERR_INVALID_ARG;
  return BSMMA_OK;
}

// Validation of the fused output stage's extra arguments.
bsmma_status check_epilogue(const void* bias, bsmma_activation act) {
  if (act < BSMMA_ACT_NONE || act > BSMMA_ACT_SILU) return BSMMA_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return BSMMA_ERR_MISALIGNED;
  return BSMMA_OK;
}

namespace {
// D[m][n] = act(bias[n]) (the output stage of an all-zero accumulator, K == 0).
__global__ void bias_act_fill_kernel(Epilogue e, __nv_bfloat16* D, int64_t M, int64_t N) {
  const uint32_t zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int64_t vecs = M * (N / 8);
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < vecs;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = v / (N / 8), c = (v - m * (N / 8)) * 8;
    store8(D + m * N + c, zero, c, e);
  }
}
}  // namespace

// K == 0: no products, so D = act(bias) per column (zero without a bias: every activation
// maps 0 to 0).
bsmma_status zero_k_epilogue(const void* bias, bsmma_activation act, void* D, int64_t M, int64_t N,
                             cudaStream_t s) {
  if (!bias) return cuda_ok(cudaMemsetAsync(D, 0, static_cast<size_t>(M * N * 2), s));
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  Epilogue e;
  e.bias = static_cast<const __nv_bfloat16*>(bias);
  e.act = static_cast<int>(act);
  bias_act_fill_kernel<<<dev->sm_count * 4, 256, 0, s>>>(e, static_cast<__nv_bfloat16*>(D), M, N);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace bsmma

using namespace bsmma;

extern "C" {

int64_t mx_scale_tiled_bytes(int64_t rows, int64_t kblocks, bsmma_scale_role role) {
  if (role != BSMMA_SCALES_A && role != BSMMA_SCALES_B) return 0;
  return wide_scale_bytes(rows, kblocks, static_cast<int>(role));
}

bsmma_status mx_scale_relayout(const uint8_t* s_plain, int64_t rows, int64_t kblocks,
                               bsmma_scale_role role, uint8_t* s_tiled, bsmma_stream stream) {
  if (rows < 0 || kblocks < 0) return BSMMA_ERR_INVALID_ARG;
  if (role != BSMMA_SCALES_A && role != BSMMA_SCALES_B) return BSMMA_ERR_INVALID_ARG;
  if (rows == 0 || kblocks == 0) return BSMMA_OK;
  if (!s_plain || !s_tiled) return BSMMA_ERR_INVALID_ARG;
  if (!aligned16(s_tiled)) return BSMMA_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (role == BSMMA_SCALES_A)
    return launch_wide_relayout(s_plain, rows, s_tiled, nullptr, 0, nullptr, kblocks, s);
  return launch_wide_relayout(nullptr, 0, nullptr, s_plain, rows, s_tiled, kblocks, s);
}

bsmma_status mx_gemm_tiled(const void* A, const uint8_t* sA_tiled, const void* B,
                           const uint8_t* sB_tiled, void* D, int64_t M, int64_t N, int64_t K,
                           bsmma_layout layout, bsmma_fmt a_fmt, bsmma_fmt b_fmt,
                           bsmma_stream stream) {
  bsmma_status st = validate_dense(A, sA_tiled, B, sB_tiled, D, M, N, K, layout, a_fmt, b_fmt);
  if (st != BSMMA_OK || M == 0 || N == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_ok(cudaMemsetAsync(D, 0, static_cast<size_t>(M * N * 2), s));
  return launch_mx_gemm(A, sA_tiled, B, sB_tiled, D, M, N, K, layout, a_fmt, b_fmt, s);
}

bsmma_status mx_gemm(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB, void* D,
                     int64_t M, int64_t N, int64_t K, bsmma_layout layout, bsmma_fmt a_fmt,
                     bsmma_fmt b_fmt, bsmma_stream stream) {
  bsmma_status st = validate_dense(A, sA, B, sB, D, M, N, K, layout, a_fmt, b_fmt);
  if (st != BSMMA_OK || M == 0 || N == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_ok(cudaMemsetAsync(D, 0, static_cast<size_t>(M * N * 2), s));
  const int64_t bytes_a = align_up(wide_scale_bytes(M, K / 32, 0), 256);
  const int64_t bytes_b = wide_scale_bytes(N, K / 32, 1);
  void* ws = nullptr;
  st = get_workspace(bytes_a + bytes_b, s, &ws);
  if (st != BSMMA_OK) return st;
  uint8_t* ta = static_cast<uint8_t*>(ws);
  uint8_t* tb = ta + bytes_a;
  st = launch_wide_relayout(sA, M, ta, sB, N, tb, K / 32, s);
  if (st != BSMMA_OK) return st;
  return launch_mx_gemm(A, ta, B, tb, D, M, N, K, layout, a_fmt, b_fmt, s);
}


bsmma_status mx_gemm_tiled_bias_act(const void* A, const uint8_t* sA_tiled, const void* B,
                                    const uint8_t* sB_tiled, const void* bias,
                                    bsmma_activation act, void* D, int64_t M, int64_t N,
                                    int64_t K, bsmma_layout layout, bsmma_fmt a_fmt,
                                    bsmma_fmt b_fmt, bsmma_stream stream) {
  bsmma_status st = validate_dense(A, sA_tiled, B, sB_tiled, D, M, N, K, layout, a_fmt, b_fmt);
  if (st == BSMMA_OK) st = check_epilogue(bias, act);
  if (st != BSMMA_OK || M == 0 || N == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return zero_k_epilogue(bias, act, D, M, N, s);
  return launch_mx_gemm(A, sA_tiled, B, sB_tiled, D, M, N, K, layout, a_fmt, b_fmt, s, bias,
                        static_cast<int>(act));
}

bsmma_status mx_gemm_bias_act(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                              const void* bias, bsmma_activation act, void* D, int64_t M,
                              int64_t N, int64_t K, bsmma_layout layout, bsmma_fmt a_fmt,
                              bsmma_fmt b_fmt, bsmma_stream stream) {
  bsmma_status st = validate_dense(A, sA, B, sB, D, M, N, K, layout, a_fmt, b_fmt);
  if (st == BSMMA_OK) st = check_epilogue(bias, act);
  if (st != BSMMA_OK || M == 0 || N == 0) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return zero_k_epilogue(bias, act, D, M, N, s);
  const int64_t bytes_a = align_up(wide_scale_bytes(M, K / 32, 0), 256);
  const int64_t bytes_b = wide_scale_bytes(N, K / 32, 1);
  void* ws = nullptr;
  st = get_workspace(bytes_a + bytes_b, s, &ws);
  if (st != BSMMA_OK) return st;
  uint8_t* ta = static_cast<uint8_t*>(ws);
  uint8_t* tb = ta + bytes_a;
  st = launch_wide_relayout(sA, M, ta, sB, N, tb, K / 32, s);
  if (st != BSMMA_OK) return st;
  return launch_mx_gemm(A, ta, B, tb, D, M, N, K, layout, a_fmt, b_fmt, s, bias,
                        static_cast<int>(act));
}

namespace {
bsmma_status check_grouped(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                           const void* D, const int64_t* m_sizes, int64_t total_M, int G,
                           int64_t N, int64_t K) {
  if (G < 1 || G > 64 || total_M < 0 || N <= 0 || K <= 0) return BSMMA_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return BSMMA_ERR_INVALID_ARG;
  if (!B || !sB || !m_sizes) return BSMMA_ERR_INVALID_ARG;
  if (total_M > 0 && (!A || !sA || !D)) return BSMMA_ERR_INVALID_ARG;
  if (!aligned16(B) || (total_M > 0 && (!aligned16(A) || !aligned16(D))) ||
      (reinterpret_cast<uintptr_t>(m_sizes) & 7u) != 0)
    return BSMMA_ERR_MISALIGNED;
  if (total_M >= INT32_MAX || static_cast<int64_t>(G) * N >= INT32_MAX || K > kMaxStride)
    return BSMMA_ERR_INVALID_ARG;
  return BSMMA_OK;
}
}  // namespace

bsmma_status grouped_fp8_gemm(const uint8_t* A, const float* sA, const uint8_t* B,
                              const float* sB, void* D, const int64_t* m_sizes, int64_t total_M,
                              int G, int64_t N, int64_t K, bsmma_stream stream) {
  const bsmma_status st = check_grouped(A, sA, B, sB, D, m_sizes, total_M, G, N, K);
  if (st != BSMMA_OK) return st;
  return launch_grouped(A, sA, B, sB, D, m_sizes, total_M, G, N, K,
                        reinterpret_cast<cudaStream_t>(stream));
}

bsmma_status grouped_fp8_gemm_packed(const uint8_t* A, const float* sA, const uint8_t* B_packed,
                                     const float* sB, void* D, const int64_t* m_sizes,
                                     int64_t total_M, int G, int64_t N, int64_t K,
                                     bsmma_stream stream) {
  const bsmma_status st = check_grouped(A, sA, B_packed, sB, D, m_sizes, total_M, G, N, K);
  if (st != BSMMA_OK) return st;
  return launch_grouped(A, sA, B_packed, sB, D, m_sizes, total_M, G, N, K,
                        reinterpret_cast<cudaStream_t>(stream), true);
}

bsmma_status grouped_fp8_pack_weights(const uint8_t* W, int64_t G, int64_t N, int64_t K,
                                      uint8_t* W_packed, bsmma_stream stream) {
  if (G < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 128 != 0) return BSMMA_ERR_INVALID_ARG;
  if (G == 0 || N == 0 || K == 0) return BSMMA_OK;
  if (!W || !W_packed) return BSMMA_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(W_packed)) return BSMMA_ERR_MISALIGNED;
  if (W == W_packed) return BSMMA_ERR_INVALID_ARG;   // not in place
  return launch_pack_weights(W, G, N, K, W_packed, reinterpret_cast<cudaStream_t>(stream));
}

bsmma_status grouped_bf16_gemm(const void* X, const void* W, void* D, const int64_t* m_sizes,
                               int64_t total_M, int G, int64_t N, int64_t K,
                               bsmma_stream stream) {
  if (G < 1 || G > 64 || total_M < 0 || N <= 0 || K <= 0) return BSMMA_ERR_INVALID_ARG;
  if (N % 8 != 0 || K % 8 != 0) return BSMMA_ERR_INVALID_ARG;
  if (!W || !m_sizes) return BSMMA_ERR_INVALID_ARG;
  if (total_M > 0 && (!X || !D)) return BSMMA_ERR_INVALID_ARG;
  if (!aligned16(W) || (total_M > 0 && (!aligned16(X) || !aligned16(D))) ||
      (reinterpret_cast<uintptr_t>(m_sizes) & 7u) != 0)
    return BSMMA_ERR_MISALIGNED;
  if (total_M >= INT32_MAX || static_cast<int64_t>(G) * N >= INT32_MAX || 2 * K > kMaxStride)
    return BSMMA_ERR_INVALID_ARG;
  return launch_grouped_bf16(X, W, D, m_sizes, total_M, G, N, K,
                             reinterpret_cast<cudaStream_t>(stream));
}

bsmma_status mx_quantize(const void* x, bsmma_dtype x_dtype, int64_t rows, int64_t cols,
                         bsmma_fmt fmt, int colwise, uint8_t* codes, uint8_t* scales,
                         bsmma_stream stream) {
  if (x_dtype != BSMMA_BF16 && x_dtype != BSMMA_F32) return BSMMA_ERR_INVALID_ARG;
  if (fmt != BSMMA_E4M3 && fmt != BSMMA_E5M2 && fmt != BSMMA_E2M1) return BSMMA_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || (colwise != 0 && colwise != 1)) return BSMMA_ERR_INVALID_ARG;
  if (colwise && fmt == BSMMA_E2M1) return BSMMA_ERR_UNSUPPORTED;
  if (colwise ? (rows % 32 != 0 || cols % 16 != 0) : (cols % 32 != 0)) return BSMMA_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return BSMMA_OK;
  if (!x || !codes || !scales) return BSMMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes)) return BSMMA_ERR_MISALIGNED;
  return launch_mx_quantize(x, x_dtype == BSMMA_F32, rows, cols, fmt, colwise != 0, codes, scales,
                            reinterpret_cast<cudaStream_t>(stream));
}

bsmma_status fp8_group_quantize(const void* x, bsmma_dtype x_dtype, int64_t total_M, int64_t K,
                                const int64_t* m_sizes, int G, uint8_t* codes, float* scales,
                                bsmma_stream stream) {
  if (x_dtype != BSMMA_BF16 && x_dtype != BSMMA_F32) return BSMMA_ERR_INVALID_ARG;
  if (G < 1 || G > 64 || total_M < 0 || K <= 0 || K % 128 != 0) return BSMMA_ERR_INVALID_ARG;
  if (!m_sizes) return BSMMA_ERR_INVALID_ARG;
  if (total_M > 0 && (!x || !codes || !scales)) return BSMMA_ERR_INVALID_ARG;
  if ((total_M + 63) / 64 * (K / 128) >= INT32_MAX) return BSMMA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(m_sizes) & 7u) != 0) return BSMMA_ERR_MISALIGNED;
  if (total_M > 0 && (!aligned16(x) || !aligned16(codes) ||
                      (reinterpret_cast<uintptr_t>(scales) & 3u) != 0))
    return BSMMA_ERR_MISALIGNED;
  return launch_group_quantize(x, x_dtype == BSMMA_F32, total_M, K, m_sizes, G, codes, scales,
                               reinterpret_cast<cudaStream_t>(stream));
}

bsmma_status fp8_block_quantize(const void* w, bsmma_dtype w_dtype, int64_t G, int64_t N,
                                int64_t K, uint8_t* codes, float* scales, bsmma_stream stream) {
  if (w_dtype != BSMMA_BF16 && w_dtype != BSMMA_F32) return BSMMA_ERR_INVALID_ARG;
  if (G < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 128 != 0) return BSMMA_ERR_INVALID_ARG;
  if (G == 0 || N == 0 || K == 0) return BSMMA_OK;
  if (G * (N / 128) * (K / 128) >= INT32_MAX) return BSMMA_ERR_INVALID_ARG;
  if (!w || !codes || !scales) return BSMMA_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return BSMMA_ERR_MISALIGNED;
  return launch_block_quantize(w, w_dtype == BSMMA_F32, G, N, K, codes, scales,
                               reinterpret_cast<cudaStream_t>(stream));
}

bsmma_status bsmma_reserve_workspace(int64_t bytes, bsmma_stream stream) {
  if (bytes < 0) return BSMMA_ERR_INVALID_ARG;
  void* p = nullptr;
  bsmma_status st = get_workspace(bytes, reinterpret_cast<cudaStream_t>(stream), &p);
  if (st != BSMMA_OK) return st;
  float* part = nullptr;
  int* arrivals = nullptr;
  return split_workspace(reinterpret_cast<cudaStream_t>(stream), &part, &arrivals);
}

bsmma_status bsmma_device_status(bsmma_stream stream) {
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0, zero = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSMMA_ERR_CUDA;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return BSMMA_ERR_CUDA;
  if (v == BSMMA_DEV_TIMEOUT) {
    // a dense launch that gave up may have left split-unit arrival counts behind
    if (cudaDeviceSynchronize() != cudaSuccess) return BSMMA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& e : g_sws)
      if (e.device == dev->device &&
          cudaMemset(e.ptr, 0, static_cast<size_t>(e.counter_bytes)) != cudaSuccess)
        return BSMMA_ERR_CUDA;
  }
  return static_cast<bsmma_status>(v);
}

bsmma_status bsmma_set_wait_limit_ns(int64_t ns) {
  if (ns <= 0) return BSMMA_ERR_INVALID_ARG;
  g_wait_limit_ns = static_cast<uint64_t>(ns);
  return BSMMA_OK;
}

bsmma_status bsmma_set_dense_variant(int variant) {
  if (variant != 0 && variant != 1 && variant != 3) return BSMMA_ERR_INVALID_ARG;
  g_dense_variant = variant;
  return BSMMA_OK;
}

bsmma_status bsmma_set_grouped_tile_width(int width) {
  if (width != 0 && width != 128 && width != 256) return BSMMA_ERR_INVALID_ARG;
  g_grouped_width = width;
  return BSMMA_OK;
}

bsmma_status bsmma_set_grouped_variant(int variant) {
  if (variant != 0 && variant != 1 && variant != 3) return BSMMA_ERR_INVALID_ARG;
  g_grouped_variant = variant;
  return BSMMA_OK;
}

const char* bsmma_status_string(bsmma_status s) {
  switch (s) {
    case BSMMA_ERR_SCRATCH_LIMIT: return "BSMMA_ERR_SCRATCH_LIMIT";
    case BSMMA_OK: return "BSMMA_OK";
    case BSMMA_ERR_INVALID_ARG: return "BSMMA_ERR_INVALID_ARG";
    case BSMMA_ERR_UNSUPPORTED: return "BSMMA_ERR_UNSUPPORTED";
    case BSMMA_ERR_MISALIGNED: return "BSMMA_ERR_MISALIGNED";
    case BSMMA_ERR_WORKSPACE: return "BSMMA_ERR_WORKSPACE";
    case BSMMA_ERR_CUDA: return "BSMMA_ERR_CUDA";
    case BSMMA_DEV_TIMEOUT: return "BSMMA_DEV_TIMEOUT";
    case BSMMA_DEV_BAD_MSIZES: return "BSMMA_DEV_BAD_MSIZES";
    default: return "BSMMA_UNKNOWN_STATUS";
  }
}

int64_t bsmma_launch_count(void) { return g_launches.load(); }

bsmma_status bsmma_probe_wait_timeout(int64_t limit_ns, bsmma_stream stream) {
  if (limit_ns <= 0 || limit_ns > 10000000000ll) return BSMMA_ERR_INVALID_ARG;
  bsmma_status st;
  const DeviceInfo* dev = current_device(&st);
  if (!dev) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = bsmma_device_status(stream);   // clear anything latched before
  if (st == BSMMA_ERR_CUDA) return st;
  wait_probe_kernel<<<1, 32, 0, s>>>(dev->status, static_cast<uint64_t>(limit_ns));
  count_launches(1);
  if (cudaGetLastError() != cudaSuccess) return BSMMA_ERR_CUDA;
  return bsmma_device_status(stream);
}

}  // extern "C"
