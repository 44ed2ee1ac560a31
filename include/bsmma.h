/*
 * bsmma.h -- C ABI of the GB300 (sm_103a) block-scaled GEMM library (libbsmma.so).
 *
 * Operations
 *   D = (A (.) sA) . (B (.) sB)^T, FP32 accumulation, BF16 output, where A and B
 *   hold FP8 (E4M3 / E5M2) or packed FP4 (E2M1) codes and sA / sB hold one E8M0
 *   scale per 32 consecutive values along K (MXFP8 / MXFP4).  Source: "PyTorch on
 *   AMD GPUs gains a FlyDSL backend", Interpretation (FP8 or packed FP4 operands,
 *   one E8M0 scale per 32 values along the reduction dimension, MXFP8 and MXFP4
 *   scaled GEMM); "Experimental FlyDSL GEMM backend for TE PyTorch", Supported
 *   Data Types (MXFP8, mixed E4M3/E5M2) and Validation (TN, NN and NT layouts).
 *
 *   The grouped groupwise FP8 GEMM: X E4M3 with one FP32 scale per row per 128-K
 *   block, W[G][N][K] E4M3 with one FP32 scale per 128x128 block, uneven or empty
 *   groups, BF16 output.  Source: "Add FlyDSL grouped groupwise FP8 GEMM for
 *   ROCm", introduction, Testing, and the commit that fixes the activation-scale
 *   layout (per-group blocks).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is caller-owned DEVICE memory of the current CUDA device;
 *     D is caller-allocated.  The library never frees or retains caller memory.
 *   - Matrices are dense and row-major with int64 extents.  Base pointers must be
 *     16-byte aligned.
 *   - All work is enqueued on `stream` (the CUDA stream handle, cudaStream_t; NULL
 *     is the legacy default stream).  No entry point synchronises the stream,
 *     except bsmma_device_status, bsmma_probe_wait_timeout and the growth of a
 *     workspace (see mx_gemm).
 *   - Errors are return codes; nothing is thrown across the ABI.  Argument errors
 *     are detected on the host before any launch and leave D untouched.  Errors
 *     detected on the device (a timed-out wait, inconsistent m_sizes) are latched
 *     in a per-device status word that bsmma_device_status reads and clears.
 *   - Entry points may be called from several host threads.
 */
#ifndef BSMMA_H
#define BSMMA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                        /* identical to cudaStream_t */
typedef struct CUstream_st* bsmma_stream;

typedef enum {
  BSMMA_OK = 0,
  BSMMA_ERR_INVALID_ARG = 1,   /* bad size, null pointer, bad enum value          */
  BSMMA_ERR_UNSUPPORTED = 2,   /* valid but unsupported format / layout combination */
  BSMMA_ERR_MISALIGNED = 3,    /* pointer or row stride violates 16-byte alignment */
  BSMMA_ERR_WORKSPACE = 4,     /* workspace would have to grow during stream capture */
  BSMMA_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed               */
  BSMMA_DEV_TIMEOUT = 6,       /* a device-side wait exceeded its limit           */
  BSMMA_DEV_BAD_MSIZES = 7,    /* m_sizes negative or not summing to total_M      */
  BSMMA_ERR_SCRATCH_LIMIT = 8  /* problem too large for mx_gemm_noalloc's fixed scratch */
} bsmma_status;

/* Layout letters in row-major operator form: NT D = A . B^T, NN D = A . B,
 * TN D = A^T . B (the Linear forward, dgrad and wgrad GEMMs). */
typedef enum { BSMMA_NT = 0, BSMMA_NN = 1, BSMMA_TN = 2 } bsmma_layout;

typedef enum { BSMMA_E4M3 = 0, BSMMA_E5M2 = 1, BSMMA_E2M1 = 2 } bsmma_fmt;

/* Which operand a set of scales belongs to: the rows of op(A) (rows of D) or the
 * rows of op(B) (columns of D).  The two sides use different tiled layouts. */
typedef enum { BSMMA_SCALES_A = 0, BSMMA_SCALES_B = 1 } bsmma_scale_role;

/*
 * mx_gemm -- dense MXFP8 / MXFP4 GEMM, D[M][N] (BF16) = op(A) . op(B)^T.
 *
 *   layout NT: A is [M][K], B is [N][K]   (both K-contiguous)
 *          NN: A is [M][K], B is [K][N]   (B N-contiguous)
 *          TN: A is [K][M], B is [K][N]   (both MN-contiguous)
 *   FP8 codes take one byte each.  E2M1 is packed two per byte along K (even k in
 *   the low nibble), rows of K/2 bytes, and is supported for NT only and only with
 *   both operands E2M1; other combinations return BSMMA_ERR_UNSUPPORTED.
 *   sA is [M][K/32], sB is [N][K/32] E8M0 codes (uint8), always indexed by
 *   (row of the logical operand op(X), K block), whatever the data layout.
 *
 * Preconditions: M, N, K >= 0; K % 32 == 0; row strides of A, B a multiple of 16
 * bytes (NN/TN: N % 16 == 0, TN: M % 16 == 0); N % 8 == 0 (16-byte rows of D).
 * M == 0 or N == 0 is a no-op; K == 0 writes D = 0.
 *
 * The scales are first rearranged (mx_scale_relayout, both roles in one launch) into
 * a library-owned device workspace kept per (device, stream), which grows when needed.
 * Growing returns BSMMA_ERR_WORKSPACE if the stream is being captured (call
 * bsmma_reserve_workspace before capture).  Otherwise it allocates a larger buffer
 * and, if no CUDA graph captured a call that used the old buffer, synchronises
 * `stream` once and frees the old one; a buffer that a captured graph uses is kept
 * until the process exits, so replaying that graph stays valid after growth.  Calls
 * on the same stream are ordered; calls on different streams use different
 * workspaces.  The workspace is keyed by the stream handle: let a stream's pending
 * mx_gemm work finish before destroying the stream, since a stream created later
 * may get the same handle and with it the same workspace.
 * When the last wave of 256 x 256 output units would leave most SM pairs idle, the
 * kernel splits those units' K range over the idle pairs and the last pair to finish
 * a unit adds the others' FP32 partial sums, in K order (the result does not depend on
 * which pair finishes last).  The partial sums live in a second per-(device, stream)
 * workspace of fixed size (two 128 KB slots per SM), allocated, its counters zeroed,
 * by the stream's first dense call outside a graph capture (bsmma_reserve_workspace
 * allocates it too).  A call captured on a stream that has none splits no unit: it
 * computes the same result, its split units' last bits rounded as unsplit ones are.
 * Two kernel launches per call (relayout, GEMM).
 */
bsmma_status mx_gemm(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                     void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                     bsmma_fmt a_fmt, bsmma_fmt b_fmt, bsmma_stream stream);

/*
 * mx_gemm_tiled -- mx_gemm with the scales already in the tiled layouts produced by
 * mx_scale_relayout: sA_tiled with role BSMMA_SCALES_A for the M rows
 * (mx_scale_tiled_bytes(M, K/32, BSMMA_SCALES_A) bytes), sB_tiled with role
 * BSMMA_SCALES_B for the N rows.  Lets callers relayout static weight scales once.
 * One kernel launch.  It allocates nothing but the fixed-size split workspace of
 * mx_gemm, on the stream's first dense call outside a graph capture; it needs no
 * reservation before capture.
 */
bsmma_status mx_gemm_tiled(const void* A, const uint8_t* sA_tiled, const void* B,
                           const uint8_t* sB_tiled, void* D, int64_t M, int64_t N, int64_t K,
                           bsmma_layout layout, bsmma_fmt a_fmt, bsmma_fmt b_fmt,
                           bsmma_stream stream);

/*
 * mx_gemm_noalloc -- mx_gemm for callers that cannot allocate device memory.
 *
 * (The source pages have no counterpart; this entry point exists for callers of
 * this library.)  mx_gemm may call cudaMalloc the first time a stream needs a
 * bigger scale workspace.  Some callers cannot allow that: code being captured
 * into a CUDA graph, code that must stay within a framework's own memory pool or a
 * fixed memory budget, and code on a path that must not synchronise (cudaMalloc
 * and cudaFree can).  mx_gemm_noalloc computes exactly what mx_gemm computes, with
 * the same arguments, preconditions and two launches, but rearranges the scales
 * into a fixed array of BSMMA_NOALLOC_SCRATCH_BYTES (16 MiB) in device memory that
 * belongs to the library; every GPU that loads the library holds that array until
 * the process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Limit: mx_scale_tiled_bytes(M, K/32, BSMMA_SCALES_A) rounded up to 256, plus
 * mx_scale_tiled_bytes(N, K/32, BSMMA_SCALES_B), must not exceed BSMMA_NOALLOC_SCRATCH_BYTES;
 * larger problems return BSMMA_ERR_SCRATCH_LIMIT before any launch.
 * The first call on a device looks up the array's device address on that device
 * (cudaGetSymbolAddress) and caches it; make that first call before any stream
 * capture.  All calls on a device share the one array and overwrite it completely,
 * so calls that can overlap on the GPU (different streams without ordering between
 * them) race with each other; order them on one stream.  It never splits output units
 * (their workspace is allocated on first use), and it never runs the
 * autotuner's timing runs (they create events and synchronise): with tuning enabled
 * it takes the stored choice for the shape class, else the SM-pair kernel.
 */
#define BSMMA_NOALLOC_SCRATCH_BYTES (16ll << 20)
bsmma_status mx_gemm_noalloc(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                             void* D, int64_t M, int64_t N, int64_t K, bsmma_layout layout,
                             bsmma_fmt a_fmt, bsmma_fmt b_fmt, bsmma_stream stream);

/*
 * grouped_fp8_gemm -- grouped groupwise FP8 GEMM, one launch.
 *
 *   A = X [total_M][K] E4M3 codes, rows of group g are [M_start_g, M_start_g+m_g)
 *       with M_start_g = m_sizes[0] + ... + m_sizes[g-1].
 *   sA  FP32 activation scales, one per row per 128-K block, in the per-group block
 *       layout: group g starts at element M_start_g*(K/128) and holds (local row l,
 *       block kb) at l + kb*m_g.
 *   B = W [G][N][K] E4M3 codes;  sB FP32 [G][N/128][K/128] weight scales.
 *   D [total_M][N] BF16: row r of group g gets
 *       sum_kb sA(g,l,kb) * sB[g][n/128][kb] * sum_{k in kb} X[r][k] * W[g][n][k].
 *   m_sizes: int64 [G] in DEVICE memory; the host never reads it (the call is
 *       capture-safe).  total_M is the row count of X and D.  Empty groups produce
 *       no work and no writes.  If an entry is negative or the entries do not sum
 *       to total_M, the kernel writes nothing and latches BSMMA_DEV_BAD_MSIZES.
 * Preconditions: N % 128 == 0, K % 128 == 0, 1 <= G <= 64, total_M >= 0.
 */
bsmma_status grouped_fp8_gemm(const uint8_t* A, const float* sA, const uint8_t* B,
                              const float* sB, void* D, const int64_t* m_sizes, int64_t total_M,
                              int G, int64_t N, int64_t K, bsmma_stream stream);

/*
 * grouped_fp8_pack_weights / grouped_fp8_gemm_packed -- the grouped GEMM with weights
 * rearranged once ahead of time, as the pages' preshuffled sibling op rearranges its
 * weights at load time ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm", introduction
 * and Performance: the _preshuffle variant).  The layout is this library's own, made
 * for sm_103a: each 128-row x 128-K tile of W is one contiguous 16 KB block that holds
 * the tile exactly as the MMA reads it from shared memory, so a kernel stage loads its
 * weight tile with one bulk copy.
 *   grouped_fp8_pack_weights: W [G][N][K] E4M3 codes -> W_packed, G*N*K bytes, where
 *     the tile (g, 128-K block kb, 128-row block nb) starts at byte
 *     ((g*(K/128) + kb)*(N/128) + nb) * 16384, row r of the tile (W row nb*128 + r) at
 *     r*128 bytes into it, and the 16-byte piece c of that row (K offsets kb*128 + 16c ..
 *     +15) at position c ^ (r % 8) of the row.  Not in place (W != W_packed).  One launch.
 *   grouped_fp8_gemm_packed: grouped_fp8_gemm with B = W_packed; every other argument,
 *     the result, preconditions and errors as for grouped_fp8_gemm.
 * Preconditions: N % 128 == 0, K % 128 == 0, G >= 0, 16-byte-aligned W and W_packed.
 */
bsmma_status grouped_fp8_pack_weights(const uint8_t* W, int64_t G, int64_t N, int64_t K,
                                      uint8_t* W_packed, bsmma_stream stream);
bsmma_status grouped_fp8_gemm_packed(const uint8_t* A, const float* sA, const uint8_t* B_packed,
                                     const float* sB, void* D, const int64_t* m_sizes,
                                     int64_t total_M, int G, int64_t N, int64_t K,
                                     bsmma_stream stream);

/*
 * grouped_bf16_gemm -- grouped BF16 GEMM: for row r of group g,
 *   D[r][n] = sum_k X[r][k] * W[g][n][k]
 * with BF16 operands, FP32 accumulation and BF16 output (round to nearest even), over
 * groups of uneven or zero size.  Source: "PyTorch on AMD GPUs gains a FlyDSL backend",
 * Interpretation: grouped GEMM that tolerates uneven and empty expert groups, measured
 * on BF16 grouped-GEMM cases (F.grouped_mm).  No scales.
 *   X        [total_M][K] BF16, row-major, device.
 *   W        [G][N][K] BF16 (one [N][K] matrix per group, K contiguous), device.
 *   D        [total_M][N] BF16, row-major, device; every row of every group written.
 *   m_sizes  [G] int64, device (read by the kernel: no host synchronisation); rows of
 *            group g are the m_sizes[g] rows after those of groups 0..g-1.
 * Preconditions: 1 <= G <= 64, total_M >= 0, N > 0 and K > 0 multiples of 8 (16-byte
 * rows), 16-byte-aligned X, W and D, 8-byte-aligned m_sizes, total_M and G*N below
 * 2^31.  BSMMA_ERR_INVALID_ARG / BSMMA_ERR_MISALIGNED otherwise, with nothing launched.
 * m_sizes that has a negative entry or does not sum to total_M is found on the device:
 * nothing is written and BSMMA_DEV_BAD_MSIZES is latched (bsmma_device_status).  One
 * launch; the caller owns every buffer; asynchronous on `stream`; allocates nothing.
 */
bsmma_status grouped_bf16_gemm(const void* X, const void* W, void* D, const int64_t* m_sizes,
                               int64_t total_M, int G, int64_t N, int64_t K,
                               bsmma_stream stream);

/*
 * mx_scale_relayout -- rearranges plain E8M0 scales s_plain [rows][kblocks] into the
 * tiled layout the GEMM kernels copy into tensor memory (128 lanes x 32 bytes per
 * copy).  Source: "[gfx1250] Add MXFP4 GEMM support to FlyDSL backend", Description
 * (the GEMM takes plain scales and rearranges them into the hardware's preferred
 * order inside the backend; a caller that keeps static weight scales can do it once,
 * here, and call mx_gemm_tiled).  The target layout is this library's own, made for
 * the sm_103a tensor-memory copy; the pages fix only that plain scales go in.  Byte (lane l, column c, byte b) of a block sits at
 * (l/8)*256 + (c/4)*128 + (l%8)*16 + (c%4)*4 + b.
 *   role BSMMA_SCALES_A: one 4096-byte chunk per 128 rows and 8 K-blocks, chunk
 *     (rb, kq) at (rb*KQ + kq)*4096, RB = 2*ceil(rows/256) row blocks,
 *     KQ = ceil(kblocks/8); lane l = row rb*128+l; column 4g + l/32 holds the row's
 *     four scales of K group g (0, 1) of the chunk; other columns are padding.
 *   role BSMMA_SCALES_B: one 4096-byte block per 256 rows and one K group (4
 *     K-blocks), block (nb, kg) at (nb*KG + kg)*4096, KG = 2*ceil(kblocks/8); four
 *     identical 1024-byte quarters in which lane i, column c holds the four scales of
 *     row nb*256 + 32c + i.
 * Padding holds 127 (the code of 1.0).  s_tiled must hold
 * mx_scale_tiled_bytes(rows, kblocks, role) bytes.  One launch.
 */
bsmma_status mx_scale_relayout(const uint8_t* s_plain, int64_t rows, int64_t kblocks,
                               bsmma_scale_role role, uint8_t* s_tiled, bsmma_stream stream);

/* Size in bytes of the tiled layout of [rows][kblocks] scales of the given role
 * (the buffer mx_scale_relayout fills; same source as mx_scale_relayout).  Returns 0
 * for an unknown role or an empty tensor. */
int64_t mx_scale_tiled_bytes(int64_t rows, int64_t kblocks, bsmma_scale_role role);

/* Activation of the fused epilogue (mx_gemm_bias_act). */
typedef enum {
  BSMMA_ACT_NONE = 0,
  BSMMA_ACT_RELU = 1,   /* max(x, 0)                          */
  BSMMA_ACT_GELU = 2,   /* x * (1 + erf(x / sqrt 2)) / 2       */
  BSMMA_ACT_SILU = 3    /* x / (1 + exp(-x))                   */
} bsmma_activation;

/*
 * mx_gemm_bias_act / mx_gemm_tiled_bias_act -- mx_gemm / mx_gemm_tiled with the output
 * stage fused: D[m][n] = act(acc[m][n] + bias[n]) rounded to BF16, where acc is the
 * FP32 accumulation mx_gemm rounds directly.  Activation and bias are the follow-up
 * named in "[gfx1250] Add MXFP4 GEMM support to FlyDSL backend", Description (the
 * plain GEMM has neither); the activation set and the erf form of GELU are this
 * library's reading.  Accuracy before the BF16 rounding: GELU's erf is evaluated by
 * Abramowitz & Stegun formula 7.1.26 (erfc form for negative inputs), so the activation
 * is within about 5e-7 |x| of the exact one; SiLU uses the fast exponential and divide
 * (a few ulp).  Both are far below the BF16 output step.
 *   bias  BF16 [N] in device memory, 16-byte aligned, or NULL for none.
 *   act   a bsmma_activation.
 * Everything else, including preconditions and errors, is as for mx_gemm / mx_gemm_tiled.
 */
bsmma_status mx_gemm_bias_act(const void* A, const uint8_t* sA, const void* B, const uint8_t* sB,
                              const void* bias, bsmma_activation act, void* D, int64_t M,
                              int64_t N, int64_t K, bsmma_layout layout, bsmma_fmt a_fmt,
                              bsmma_fmt b_fmt, bsmma_stream stream);
bsmma_status mx_gemm_tiled_bias_act(const void* A, const uint8_t* sA_tiled, const void* B,
                                    const uint8_t* sB_tiled, const void* bias,
                                    bsmma_activation act, void* D, int64_t M, int64_t N,
                                    int64_t K, bsmma_layout layout, bsmma_fmt a_fmt,
                                    bsmma_fmt b_fmt, bsmma_stream stream);

/*
 * Autotuning (opt-in).  "Add FlyDSL grouped groupwise FP8 GEMM for ROCm", Tile
 * selection: candidates are timed once per shape class and the winner persisted to
 * disk, behind a gate, with a fixed choice when the gate is off and no tuning during
 * graph capture.
 *   Shape classes and candidates: grouped_fp8_gemm per (nextPow2(total_M), N, K, G),
 *   tile widths 256 and 128 (when N % 256 == 0); grouped_bf16_gemm likewise (when
 *   N > 128), with SM-pair 256 x 256 tiles as a third candidate (2); the dense GEMMs
 *   per (nextPow2(M), N, K, layout, a_fmt, b_fmt), the SM-pair and single-CTA kernels
 *   (3, 1).
 *   The first call of a new class on a non-capturing stream runs each candidate twice
 *   and waits for it (it synchronises that stream); later calls, and calls in any
 *   process that reads the same cache file, use the stored choice.  A variant or width
 *   set with bsmma_set_dense_variant / bsmma_set_grouped_tile_width /
 *   bsmma_set_grouped_variant takes precedence.
 *   Every candidate computes the same result.
 * bsmma_autotune_configure -- enable: 1 on, 0 off, -1 from the environment
 *   (BSMMA_AUTOTUNE=1 turns it on); cache_path: the file, or NULL for
 *   BSMMA_AUTOTUNE_CACHE, else $XDG_CACHE_HOME/bsmma/autotune.txt, else
 *   $HOME/.cache/bsmma/autotune.txt.  Reloads the cache.  Without a call the
 *   environment decides at the first GEMM.  The file holds one line per class:
 *   "grouped <T> <N> <K> <G> <width>" or "dense <M> <N> <K> <layout> <a_fmt> <b_fmt>
 *   <variant>" (T, M rounded up to powers of two).
 * bsmma_autotune_lookup -- the stored choice for a key (a line without its last
 *   field), or -1.
 */
bsmma_status bsmma_autotune_configure(int enable, const char* cache_path);
int bsmma_autotune_lookup(const char* key);

/* Element type of the high-precision inputs of the quantisers. */
typedef enum { BSMMA_BF16 = 0, BSMMA_F32 = 1 } bsmma_dtype;

/*
 * mx_quantize -- MX quantisation, the step that makes mx_gemm's operands.  Source:
 * "[gfx1250] Add MXFP4 GEMM support to FlyDSL backend", the MXFP4 test helpers and
 * their review (rowwise and columnwise data are quantised separately, each the
 * layout one GEMM operand reads; BF16 input, FP32 input asked for as well).
 *   x        [rows][cols] BF16 or FP32 (x_dtype), row-major.
 *   Per block of 32 consecutive values along the quantised dimension:
 *     amax = max |x|;  e = floor(log2 amax) - emax, emax = 8 (E4M3), 15 (E5M2) or
 *     2 (E2M1), clamped to [-127, 127];  scale code = e + 127 (127 if amax == 0);
 *     code = round-to-nearest-even of the FP32 product x * 2^-e, saturated to the
 *     largest finite value (448, 57344, 6), with the sign bit of x.
 *   colwise == 0 (rowwise): blocks run along cols.  codes [rows][cols] (E2M1:
 *     [rows][cols/2], the even column in the low nibble); scales [rows][cols/32].
 *     This is mx_gemm's A or B of an NT GEMM, its A of NN, ...: an operand whose
 *     reduction dimension is contiguous.
 *   colwise == 1: blocks run along rows.  codes [rows][cols] (same layout as x);
 *     scales [cols][rows/32] (indexed by column, then row block).  This is the
 *     MN-major B of NN and the A and B of TN.  E4M3 and E5M2 only.
 * Preconditions: 16-byte-aligned x and codes; rowwise cols % 32 == 0, columnwise
 *   rows % 32 == 0 and cols % 16 == 0.  Inputs must be finite.  One launch (none
 *   for an empty tensor).
 */
bsmma_status mx_quantize(const void* x, bsmma_dtype x_dtype, int64_t rows, int64_t cols,
                         bsmma_fmt fmt, int colwise, uint8_t* codes, uint8_t* scales,
                         bsmma_stream stream);

/*
 * fp8_group_quantize -- groupwise E4M3 quantisation of the grouped GEMM's activations
 * (quantize_fp8_group(m_sizes=...) in "Add FlyDSL grouped groupwise FP8 GEMM for
 * ROCm", and the commit that fixes the activation-scale layout).
 *   x [total_M][K] BF16 or FP32; per row and 128-K block: s = amax / 448 (1 when
 *   amax == 0, both FP32), code = RNE-saturate(x / s) in E4M3 (FP32 division).
 *   codes [total_M][K] E4M3;  scales FP32 in the per-group block layout that
 *   grouped_fp8_gemm reads: group g starts at M_start_g*(K/128) and holds (local row
 *   l, block kb) at l + kb*m_g.
 *   m_sizes: int64 [G] in DEVICE memory; if an entry is negative or the entries do
 *   not sum to total_M, nothing is written and BSMMA_DEV_BAD_MSIZES is latched.
 * Preconditions: K % 128 == 0, 1 <= G <= 64, total_M >= 0, 16-byte-aligned x and
 *   codes.  One launch.
 */
bsmma_status fp8_group_quantize(const void* x, bsmma_dtype x_dtype, int64_t total_M, int64_t K,
                                const int64_t* m_sizes, int G, uint8_t* codes, float* scales,
                                bsmma_stream stream);

/*
 * fp8_block_quantize -- blockwise E4M3 quantisation of the grouped GEMM's weights
 * (128x128 blocks; same source).
 *   w [G][N][K] BF16 or FP32; per 128x128 block: s = amax / 448 (1 when amax == 0),
 *   code = RNE-saturate(w / s).  codes [G][N][K] E4M3;  scales FP32 [G][N/128][K/128].
 * Preconditions: N % 128 == 0, K % 128 == 0, G >= 0, 16-byte-aligned w and codes.
 *   One launch.
 */
bsmma_status fp8_block_quantize(const void* w, bsmma_dtype w_dtype, int64_t G, int64_t N,
                                int64_t K, uint8_t* codes, float* scales, bsmma_stream stream);

/* Grows the current (device, stream) scale workspace to at least `bytes` and allocates
 * the stream's split workspace if it has none (call before capturing mx_gemm or
 * mx_gemm_tiled into a CUDA graph).  The stream argument is this library's addition to
 * the boundary: workspaces are kept per stream, so the ones that a later capture on
 * `stream` will use are the ones reserved.  After bsmma_device_status has returned
 * BSMMA_DEV_TIMEOUT, the split workspaces' counters are cleared before it returns. */
bsmma_status bsmma_reserve_workspace(int64_t bytes, bsmma_stream stream);

/* Synchronises `stream`, then returns and clears the current device's latched
 * device-side status (BSMMA_OK, BSMMA_DEV_TIMEOUT or BSMMA_DEV_BAD_MSIZES). */
bsmma_status bsmma_device_status(bsmma_stream stream);

/* Sets the limit of every device-side wait, in nanoseconds (default 2e9). */
bsmma_status bsmma_set_wait_limit_ns(int64_t ns);

/* Selects the dense kernel variant for later mx_gemm / mx_gemm_tiled calls:
 * 0 automatic (default: SM-pair MMAs), 1 one CTA per 128x256 tile, 3 SM-pair MMAs
 * (2-CTA clusters issuing one 256x256 MMA over both SMs); any other value returns
 * BSMMA_ERR_INVALID_ARG.  Both variants compute the same result; this is a tuning and
 * testing control. */
bsmma_status bsmma_set_dense_variant(int variant);

/* Selects the grouped kernels' tile width for later grouped_fp8_gemm and
 * grouped_bf16_gemm calls: 0 automatic (default: 256 when the wide tiles fill the GPU
 * at least twice and, for grouped_fp8_gemm, N % 256 == 0; else 128), 128 or 256
 * (grouped_fp8_gemm: used only when N % 256 == 0).  Same result; a tuning and testing
 * control. */
bsmma_status bsmma_set_grouped_tile_width(int width);

/* Selects grouped_bf16_gemm's tiles for later calls: 0 automatic (default: 256 x 256 tiles
 * on SM pairs -- 2-CTA clusters issuing M = 256 MMAs -- when N > 128 and the groups average
 * at least 128 rows, else one CTA per 128-row tile of 128 or 256 columns), 1 one CTA per
 * tile, 3 SM-pair tiles.  Any other value returns BSMMA_ERR_INVALID_ARG.  Same result; a
 * tuning and testing control.  (grouped_fp8_gemm always uses one CTA per tile.) */
bsmma_status bsmma_set_grouped_variant(int variant);

/* Human-readable name of a status code (static storage). */
const char* bsmma_status_string(bsmma_status status);

/* Number of kernels this library has launched in this process. */
int64_t bsmma_launch_count(void);

/*
 * bsmma_probe_wait_timeout -- runs the library's bounded mbarrier wait on a
 * barrier that nothing ever completes, with a limit of `limit_ns`, and returns the
 * device status it latches (expected: BSMMA_DEV_TIMEOUT).  Exercises the failure
 * path of every kernel's waits without faulting or hanging the GPU; the context
 * stays usable.  Synchronises `stream`.
 */
bsmma_status bsmma_probe_wait_timeout(int64_t limit_ns, bsmma_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* BSMMA_H */
