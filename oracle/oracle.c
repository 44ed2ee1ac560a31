/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the block-scaled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file; only the tests, the smoke check and the CPU baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (in FP64, no blocking, no fusion):
 *
 *   dense block-scaled GEMM (MXFP8 / MXFP4; "PyTorch on AMD GPUs gains a FlyDSL
 *   backend", Interpretation: FP8 or packed FP4 operands with one E8M0 scale per
 *   32 values along the reduction dimension; "Experimental FlyDSL GEMM backend
 *   for TE PyTorch", Supported Data Types: MXFP8):
 *
 *     D[m][n] = sum_k  dec_a(Aop[m][k]) * 2^(sA[m][k/32]-127)
 *                     * dec_b(Bop[n][k]) * 2^(sB[n][k/32]-127)
 *
 *   grouped groupwise FP8 ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm",
 *   introduction and the commit that fixes the activation-scale layout):
 *
 *     for row r of group g (local row l = r - M_start_g):
 *     D[r][n] = sum_kb sX(g,l,kb) * sW[g][n/128][kb]
 *                      * sum_{k in block kb} e4m3(X[r][k]) * e4m3(W[g][n][k])
 *     with sX(g,l,kb) = sA[M_start_g*(K/128) + l + kb*m_g]  (per-group blocks).
 *
 *   grouped BF16 ("PyTorch on AMD GPUs gains a FlyDSL backend", Interpretation:
 *   grouped GEMM over uneven and empty groups, BF16 cases):
 *
 *     for row r of group g:  D[r][n] = sum_k bf16(X[r][k]) * bf16(W[g][n][k])
 *
 * Decoding is by 256-entry (16 for E2M1) tables built from the format
 * definitions (OCP E4M3FN, E5M2, E2M1, E8M0).  Every operand row is decoded
 * once into an FP64 buffer, then plain sequential dot products are taken.
 *
 *   quantisers (the step before the GEMM): MX rowwise / columnwise with E8M0 block
 *   scales, and the groupwise FP8 activation (1x128) and weight (128x128)
 *   quantisers with FP32 scales; see the section at the end of this file.
 *
 * Parity is pinned by the CPU test-suite: closed-form decode points, exact
 * rational brute force on tiny inputs, unit-scale = plain matmul, power-of-two
 * equivariance, layout equivalence, grouped = per-group dense concatenation,
 * bijection / padding / hand-derived positions of the scale relayouts, and for
 * the quantisers closed-form codes (ties, saturation, zero blocks, nibble order),
 * exact round trips of representable values, an independent numpy/torch
 * quantiser, and the half-step error bound.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { FMT_E4M3 = 0, FMT_E5M2 = 1, FMT_E2M1 = 2 };
enum { LAYOUT_NT = 0, LAYOUT_NN = 1, LAYOUT_TN = 2 };

/* ------------------------------------------------------------------------ */
/* Decode tables, from the bit-level definitions of each format.             */
/* ------------------------------------------------------------------------ */
static double T_E4M3[256], T_E5M2[256], T_E2M1[16], T_E8M0[256];
static pthread_once_t tables_once = PTHREAD_ONCE_INIT;

static void build_tables(void) {
  for (int c = 0; c < 256; ++c) {
    /* E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa; S.1111.111 is NaN, no inf. */
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0) v = ldexp((double)m, -9);            /* m/8 * 2^(1-7) */
    else v = ldexp(8.0 + m, e - 10);                        /* (1+m/8) * 2^(e-7) */
    T_E4M3[c] = s ? -v : v;

    /* E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa; exponent 31 is inf/NaN. */
    e = (c >> 2) & 31; m = c & 3;
    if (e == 31) v = (m == 0) ? INFINITY : NAN;
    else if (e == 0) v = ldexp((double)m, -16);            /* m/4 * 2^(1-15) */
    else v = ldexp(4.0 + m, e - 17);                        /* (1+m/4) * 2^(e-15) */
    T_E5M2[c] = s ? -v : v;

    /* E8M0: unsigned power of two 2^(c-127); 0xFF is NaN. */
    T_E8M0[c] = (c == 255) ? NAN : ldexp(1.0, c - 127);
  }
  for (int c = 0; c < 16; ++c) {
    /* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa, no inf/NaN. */
    int s = c >> 3, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(2.0 + m, e - 2);  /* (1+m/2)*2^(e-1) */
    T_E2M1[c] = s ? -v : v;
  }
}

static void init_tables(void) { pthread_once(&tables_once, build_tables); }

/* Copies one decode table out (fmt 0 E4M3, 1 E5M2, 2 E2M1, 3 E8M0). */
int oracle_decode_table(int which, double* out) {
  init_tables();
  switch (which) {
    case 0: memcpy(out, T_E4M3, sizeof T_E4M3); return 256;
    case 1: memcpy(out, T_E5M2, sizeof T_E5M2); return 256;
    case 2: memcpy(out, T_E2M1, sizeof T_E2M1); return 16;
    case 3: memcpy(out, T_E8M0, sizeof T_E8M0); return 256;
    default: return -1;
  }
}

/* Element (i, k) of the logical [rows, K] view of an operand.
 * rowmajor_k: the data is stored [rows][K] (K contiguous);
 * otherwise it is stored [K][rows] (rows contiguous).
 * FP4 is packed two per byte along K, even k in the low nibble. */
static double elem(const uint8_t* X, int fmt, int rowmajor_k, int64_t rows, int64_t K,
                   int64_t i, int64_t k) {
  if (fmt == FMT_E2M1) {
    /* packed FP4 exists only K-contiguous */
    uint8_t byte = X[i * (K / 2) + k / 2];
    return T_E2M1[(k & 1) ? (byte >> 4) : (byte & 15)];
  }
  uint8_t code = rowmajor_k ? X[i * K + k] : X[k * rows + i];
  return fmt == FMT_E4M3 ? T_E4M3[code] : T_E5M2[code];
}

/* Decode logical row i of an operand, with its E8M0 block scales applied, into out[K]. */
static void decode_row_scaled(const uint8_t* X, const uint8_t* S, int fmt, int rowmajor_k,
                              int64_t rows, int64_t K, int64_t i, double* out) {
  int64_t kb = K / 32;
  for (int64_t k = 0; k < K; ++k)
    out[k] = elem(X, fmt, rowmajor_k, rows, K, i, k) * T_E8M0[S[i * kb + k / 32]];
}

/* ------------------------------------------------------------------------ */
/* Dense MX GEMM.                                                            */
/* ------------------------------------------------------------------------ */
typedef struct {
  const uint8_t *A, *sA, *B, *sB;
  int64_t M, N, K;
  int a_fmt, b_fmt, a_kcontig, b_kcontig;
  const int64_t* rows; int64_t nrows;   /* output rows to evaluate */
  const double* Adec;                   /* [nrows][K] decoded, scaled rows of op(A) */
  double* D;                            /* [nrows][N] */
  int64_t n0, n1;                       /* this worker's column range */
} dense_job;

static void* dense_worker(void* p) {
  dense_job* j = (dense_job*)p;
  double* brow = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
  for (int64_t n = j->n0; n < j->n1; ++n) {
    decode_row_scaled(j->B, j->sB, j->b_fmt, j->b_kcontig, j->N, j->K, n, brow);
    for (int64_t r = 0; r < j->nrows; ++r) {
      const double* a = j->Adec + r * j->K;
      double acc = 0.0;
      for (int64_t k = 0; k < j->K; ++k) acc += a[k] * brow[k];
      j->D[r * j->N + n] = acc;
    }
  }
  free(brow);
  return NULL;
}

/* Splits [0, n) across nthreads workers and runs fn on each. */
static int run_parallel(void* jobs, size_t job_size, int nthreads, void* (*fn)(void*)) {
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  for (int t = 0; t < nthreads; ++t)
    pthread_create(&th[t], NULL, fn, (char*)jobs + (size_t)t * job_size);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  return 0;
}

/*
 * D[r][n] for r over `rows` (or all M rows when rows == NULL) and all n.
 * layout: 0 NT (A[M][K], B[N][K]), 1 NN (A[M][K], B[K][N]), 2 TN (A[K][M], B[K][N]).
 * sA is [M][K/32], sB is [N][K/32], always indexed by (row of op(X), K block).
 * Returns 0 on success, -1 on an unsupported combination.
 */
int oracle_mx_gemm(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                   int64_t M, int64_t N, int64_t K, int layout, int a_fmt, int b_fmt,
                   const int64_t* rows, int64_t nrows, double* D, int nthreads) {
  init_tables();
  if (K % 32 != 0 || M < 0 || N < 0 || K < 0) return -1;
  if ((a_fmt == FMT_E2M1) != (b_fmt == FMT_E2M1)) return -1;
  if (a_fmt == FMT_E2M1 && layout != LAYOUT_NT) return -1;
  int a_kcontig = (layout != LAYOUT_TN);
  int b_kcontig = (layout == LAYOUT_NT);
  if (rows == NULL) nrows = M;
  if (nrows == 0 || N == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > N) nthreads = (int)N;

  double* Adec = (double*)malloc(sizeof(double) * (size_t)(nrows * (K > 0 ? K : 1)));
  for (int64_t r = 0; r < nrows; ++r)
    decode_row_scaled(A, sA, a_fmt, a_kcontig, M, K, rows ? rows[r] : r, Adec + r * K);

  dense_job* jobs = (dense_job*)malloc(sizeof(dense_job) * (size_t)nthreads);
  for (int t = 0; t < nthreads; ++t) {
    dense_job j = {A, sA, B, sB, M, N, K, a_fmt, b_fmt, a_kcontig, b_kcontig,
                   rows, nrows, Adec, D, N * t / nthreads, N * (t + 1) / nthreads};
    jobs[t] = j;
  }
  run_parallel(jobs, sizeof(dense_job), nthreads, dense_worker);
  free(jobs);
  free(Adec);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped groupwise FP8 GEMM.                                               */
/* ------------------------------------------------------------------------ */
typedef struct {
  const uint8_t *W;
  const double* Xdec;                   /* [nrows][K] decoded sampled rows of X */
  const float *sX, *sW;
  int64_t N, K, KB;
  int64_t nrows;
  const int64_t *row_of, *grp_of, *loc_of, *start_of, *msz_of; /* per sampled row */
  int G;
  double* D;
  int64_t n0, n1;
} grouped_job;

static void* grouped_worker(void* p) {
  grouped_job* j = (grouped_job*)p;
  double* wrow = (double*)malloc(sizeof(double) * (size_t)j->K);
  for (int g = 0; g < j->G; ++g) {
    int any = 0;
    for (int64_t r = 0; r < j->nrows; ++r) any |= (j->grp_of[r] == g);
    if (!any) continue;
    for (int64_t n = j->n0; n < j->n1; ++n) {
      const uint8_t* w = j->W + ((int64_t)g * j->N + n) * j->K;
      for (int64_t k = 0; k < j->K; ++k) wrow[k] = T_E4M3[w[k]];
      for (int64_t r = 0; r < j->nrows; ++r) {
        if (j->grp_of[r] != g) continue;
        const double* xrow = j->Xdec + r * j->K;
        double acc = 0.0;
        for (int64_t kb = 0; kb < j->KB; ++kb) {
          double part = 0.0;
          for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) part += xrow[k] * wrow[k];
          double sx = (double)j->sX[j->start_of[r] * j->KB + j->loc_of[r] + kb * j->msz_of[r]];
          double sw = (double)j->sW[((int64_t)g * (j->N / 128) + n / 128) * j->KB + kb];
          acc += sx * sw * part;
        }
        j->D[r * j->N + n] = acc;
      }
    }
  }
  free(wrow);
  return 0;
}

/*
 * X [total_M][K] E4M3, sX per-group block layout FP32, W [G][N][K] E4M3,
 * sW [G][N/128][K/128] FP32, m_sizes [G] int64 (host).  Output rows `rows`
 * (global row ids; NULL = all total_M rows) into D[nrows][N].
 * Returns 0, or -1 on bad arguments (negative size, sum != total_M, N or K % 128).
 */
int oracle_grouped_fp8_gemm(const uint8_t* X, const float* sX, const uint8_t* W, const float* sW,
                            const int64_t* m_sizes, int G, int64_t total_M, int64_t N, int64_t K,
                            const int64_t* rows, int64_t nrows, double* D, int nthreads) {
  init_tables();
  if (N % 128 != 0 || K % 128 != 0 || G < 1) return -1;
  int64_t sum = 0;
  for (int g = 0; g < G; ++g) { if (m_sizes[g] < 0) return -1; sum += m_sizes[g]; }
  if (sum != total_M) return -1;
  if (rows == NULL) nrows = total_M;
  if (nrows == 0 || N == 0) return 0;

  int64_t* meta = (int64_t*)malloc(sizeof(int64_t) * (size_t)(5 * nrows));
  int64_t *row_of = meta, *grp_of = meta + nrows, *loc_of = meta + 2 * nrows,
          *start_of = meta + 3 * nrows, *msz_of = meta + 4 * nrows;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t row = rows ? rows[r] : r;
    if (row < 0 || row >= total_M) { free(meta); return -1; }
    int64_t start = 0;
    int g = 0;
    while (row >= start + m_sizes[g]) { start += m_sizes[g]; ++g; }
    row_of[r] = row; grp_of[r] = g; loc_of[r] = row - start; start_of[r] = start;
    msz_of[r] = m_sizes[g];
  }
  double* Xdec = (double*)malloc(sizeof(double) * (size_t)(nrows * K));
  for (int64_t r = 0; r < nrows; ++r)
    for (int64_t k = 0; k < K; ++k) Xdec[r * K + k] = T_E4M3[X[row_of[r] * K + k]];
  if (nthreads < 1) nthreads = 1;
  if (nthreads > N) nthreads = (int)N;
  grouped_job* jobs = (grouped_job*)malloc(sizeof(grouped_job) * (size_t)nthreads);
  for (int t = 0; t < nthreads; ++t) {
    grouped_job j = {W, Xdec, sX, sW, N, K, K / 128, nrows, row_of, grp_of, loc_of, start_of,
                     msz_of, G, D, N * t / nthreads, N * (t + 1) / nthreads};
    jobs[t] = j;
  }
  run_parallel(jobs, sizeof(grouped_job), nthreads, grouped_worker);
  free(jobs);
  free(Xdec);
  free(meta);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped BF16 GEMM ("PyTorch on AMD GPUs gains a FlyDSL backend",          */
/* Interpretation: grouped GEMM over uneven and empty expert groups, BF16    */
/* cases).  The plain reading: for row r of group g,                         */
/*   D[r][n] = sum_k bf16(X[r][k]) * bf16(W[g][n][k])                         */
/* with no scales.  BF16 is decoded from its bit fields (1 sign, 8 exponent  */
/* bits with bias 127, 7 mantissa bits).                                     */
/* ------------------------------------------------------------------------ */
static double bf16_value(uint16_t c) {
  int s = c >> 15, e = (c >> 7) & 255, m = c & 127;
  double v;
  if (e == 255) v = (m == 0) ? INFINITY : NAN;
  else if (e == 0) v = ldexp((double)m, -133);             /* m/128 * 2^(1-127) */
  else v = ldexp(128.0 + m, e - 134);                       /* (1+m/128) * 2^(e-127) */
  return s ? -v : v;
}

typedef struct {
  const uint16_t* W;
  const double* Xdec;                    /* [nrows][K] decoded sampled rows of X */
  int64_t N, K, nrows;
  const int64_t* grp_of;
  int G;
  double* D;
  int64_t n0, n1;
} grouped_bf16_job;

static void* grouped_bf16_worker(void* p) {
  grouped_bf16_job* j = (grouped_bf16_job*)p;
  double* wrow = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
  for (int g = 0; g < j->G; ++g) {
    int any = 0;
    for (int64_t r = 0; r < j->nrows; ++r) any |= (j->grp_of[r] == g);
    if (!any) continue;
    for (int64_t n = j->n0; n < j->n1; ++n) {
      const uint16_t* w = j->W + ((int64_t)g * j->N + n) * j->K;
      for (int64_t k = 0; k < j->K; ++k) wrow[k] = bf16_value(w[k]);
      for (int64_t r = 0; r < j->nrows; ++r) {
        if (j->grp_of[r] != g) continue;
        const double* xrow = j->Xdec + r * j->K;
        double acc = 0.0;
        for (int64_t k = 0; k < j->K; ++k) acc += xrow[k] * wrow[k];
        j->D[r * j->N + n] = acc;
      }
    }
  }
  free(wrow);
  return 0;
}

/*
 * X [total_M][K] BF16 bit patterns, W [G][N][K] BF16 bit patterns, m_sizes [G]
 * int64 (host).  Output rows `rows` (global row ids; NULL = all total_M rows) into
 * D[nrows][N].  Returns 0, or -1 on bad arguments (negative size, sum != total_M,
 * row id out of range).
 */
int oracle_grouped_bf16_gemm(const uint16_t* X, const uint16_t* W, const int64_t* m_sizes, int G,
                             int64_t total_M, int64_t N, int64_t K, const int64_t* rows,
                             int64_t nrows, double* D, int nthreads) {
  if (G < 1 || N < 0 || K < 0) return -1;
  int64_t sum = 0;
  for (int g = 0; g < G; ++g) { if (m_sizes[g] < 0) return -1; sum += m_sizes[g]; }
  if (sum != total_M) return -1;
  if (rows == NULL) nrows = total_M;
  if (nrows == 0 || N == 0) return 0;
  int64_t* grp_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)nrows);
  double* Xdec = (double*)malloc(sizeof(double) * (size_t)(nrows * (K > 0 ? K : 1)));
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t row = rows ? rows[r] : r;
    if (row < 0 || row >= total_M) { free(grp_of); free(Xdec); return -1; }
    int64_t start = 0;
    int g = 0;
    while (row >= start + m_sizes[g]) { start += m_sizes[g]; ++g; }
    grp_of[r] = g;
    for (int64_t k = 0; k < K; ++k) Xdec[r * K + k] = bf16_value(X[row * K + k]);
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > N) nthreads = (int)N;
  grouped_bf16_job* jobs = (grouped_bf16_job*)malloc(sizeof(grouped_bf16_job) * (size_t)nthreads);
  for (int t = 0; t < nthreads; ++t) {
    grouped_bf16_job j = {W, Xdec, N, K, nrows, grp_of, G, D, N * t / nthreads,
                          N * (t + 1) / nthreads};
    jobs[t] = j;
  }
  run_parallel(jobs, sizeof(grouped_bf16_job), nthreads, grouped_bf16_worker);
  free(jobs);
  free(Xdec);
  free(grp_of);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Wide scale layouts (integer permutations with padding), read by the      */
/* tensor core's 128-lane x 32-byte copies.                                 */
/*                                                                          */
/* Byte position of (lane l, column c, byte b) inside a block, in the order */
/* the copy walks its source: 8-lane groups of 256 bytes, each holding two  */
/* 128-byte halves (columns 0-3, 4-7) of 8 lanes x 16 bytes.               */
/*                                                                          */
/* Row role (op(A) rows): 4096-byte chunk per 128 rows and 8 K-blocks.      */
/*   Lane l is row l of the block, in lane quarter q = l/32.  Column c holds */
/*   row l's 4 scales of K group c/4 of the chunk when c%4 == q; every other */
/*   column is padding.  Chunk (rb, kq) at (rb*KQ + kq)*4096,               */
/*   RB = 2*ceil(rows/256), KQ = ceil(kblocks/8).                           */
/* Column role (op(B) rows): 4096-byte block per 256 rows and one K group:  */
/*   four identical 1024-byte quarters, one per lane quarter (q*1024);      */
/*   in each, lane i (0..31), column c holds the 4 scales of row 32c + i.   */
/*   Block (nb, kg) at (nb*KG + kg)*4096, NB = ceil(rows/256),              */
/*   KG = 2*ceil(kblocks/8).                                                */
/* Padding holds 127 (the E8M0 code of 1.0).                                */
/* ------------------------------------------------------------------------ */
static int64_t lane_col_byte(int64_t l, int64_t c, int64_t b) {
  return (l / 8) * 256 + (c / 4) * 128 + (l % 8) * 16 + (c % 4) * 4 + b;
}

int64_t oracle_wide_scale_bytes(int64_t rows, int64_t kblocks, int role) {
  if (rows <= 0 || kblocks <= 0) return 0;
  if (role == 0) return 2 * ((rows + 255) / 256) * ((kblocks + 7) / 8) * 4096;
  return ((rows + 255) / 256) * 2 * ((kblocks + 7) / 8) * 4096;
}

void oracle_wide_scale_relayout(const uint8_t* s, int64_t rows, int64_t kblocks, int role,
                                uint8_t* out) {
  int64_t total = oracle_wide_scale_bytes(rows, kblocks, role);
  for (int64_t i = 0; i < total; ++i) out[i] = 127;
  if (role == 0) {
    int64_t KQ = (kblocks + 7) / 8;
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t kb = 0; kb < kblocks; ++kb) {
        int64_t rb = r / 128, l = r % 128, kg = kb / 4, kq = kg / 2, g = kg % 2;
        int64_t c = 4 * g + l / 32;
        out[(rb * KQ + kq) * 4096 + lane_col_byte(l, c, kb % 4)] = s[r * kblocks + kb];
      }
  } else {
    int64_t KG = 2 * ((kblocks + 7) / 8);
    for (int64_t n = 0; n < rows; ++n)
      for (int64_t kb = 0; kb < kblocks; ++kb) {
        int64_t nb = n / 256, nn = n % 256, kg = kb / 4;
        for (int64_t q = 0; q < 4; ++q)
          out[(nb * KG + kg) * 4096 + q * 1024 + lane_col_byte(nn % 32, nn / 32, kb % 4)] =
              s[n * kblocks + kb];
      }
  }
}

/* ------------------------------------------------------------------------ */
/* Quantisers: the step before the GEMM.                                     */
/*                                                                           */
/* MX ("[gfx1250] Add MXFP4 GEMM support to FlyDSL backend", the MXFP4 test   */
/* helpers and their review: rowwise and columnwise data are quantised        */
/* separately; the quantiser takes BF16 input, FP32 asked for as well): per    */
/* block of 32 values along the quantised dimension, amax = max|x|, E8M0 scale */
/* 2^e with e = floor(log2 amax) - emax (emax 8 / 15 / 2 for E4M3 / E5M2 /     */
/* E2M1), clamped to [-127, 127]; amax == 0 gives scale code 127.  Codes are   */
/* round-to-nearest-even of x * 2^-e (an FP32 product), saturated to the       */
/* largest finite value, with the sign of x.                                   */
/*                                                                           */
/* Groupwise FP8 ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm":            */
/* quantize_fp8_group(m_sizes=...) and the per-group block layout of its       */
/* scales; 1x128 activation blocks, 128x128 weight blocks): FP32 scale          */
/* s = amax / 448 (1 when amax == 0, at least 2^-149), codes =                  */
/* RNE-saturate(x / s) in E4M3, both divisions in FP32.  Inputs are FP32        */
/* values (BF16 converts exactly).                                            */
/* ------------------------------------------------------------------------ */
static int fmt_emax(int fmt) { return fmt == FMT_E4M3 ? 8 : fmt == FMT_E5M2 ? 15 : 2; }
static int fmt_top(int fmt) { return fmt == FMT_E4M3 ? 0x7E : fmt == FMT_E5M2 ? 0x7B : 7; }
static const double* fmt_table(int fmt) {
  return fmt == FMT_E4M3 ? T_E4M3 : fmt == FMT_E5M2 ? T_E5M2 : T_E2M1;
}

/* Nearest finite code of |v| (ties to the even code, i.e. even mantissa), saturated at
 * the largest finite magnitude; the sign bit follows the sign of v (so -0 and small
 * negatives that round to zero keep it). */
static uint8_t encode_rne_sat(double v, int fmt) {
  const double* T = fmt_table(fmt);
  const int top = fmt_top(fmt);
  const double a = fabs(v);
  int c;
  if (a >= T[top]) {
    c = top;
  } else {
    int lo = 0, hi = top;            /* T[lo] <= a < T[hi]; positive codes increase with value */
    while (hi - lo > 1) {
      const int mid = (lo + hi) / 2;
      if (T[mid] <= a) lo = mid;
      else hi = mid;
    }
    const double below = a - T[lo], above = T[hi] - a;
    if (below < above) c = lo;
    else if (above < below) c = hi;
    else c = (lo & 1) ? hi : lo;
  }
  if (signbit(v)) c |= (fmt == FMT_E2M1) ? 0x8 : 0x80;
  return (uint8_t)c;
}

/* floor(log2 a) for a finite a > 0, exactly (frexp gives a = f * 2^p, f in [0.5, 1)). */
static int floor_log2(double a) {
  int p;
  (void)frexp(a, &p);
  return p - 1;
}

/* MX quantisation of x[rows][cols] (row-major FP32 values).
 *   colwise == 0: blocks of 32 along cols; codes [rows][cols] (E2M1: [rows][cols/2],
 *                 even column in the low nibble); scales [rows][cols/32].
 *   colwise == 1: blocks of 32 along rows; codes [rows][cols] (same layout as x);
 *                 scales [cols][rows/32].  Not for E2M1.
 * Returns 0, or -1 for unsupported arguments. */
int oracle_mx_quantize(const float* x, int64_t rows, int64_t cols, int fmt, int colwise,
                       uint8_t* codes, uint8_t* scales) {
  init_tables();
  if (rows < 0 || cols < 0 || fmt < FMT_E4M3 || fmt > FMT_E2M1) return -1;
  if (colwise ? (rows % 32 != 0 || fmt == FMT_E2M1) : (cols % 32 != 0)) return -1;
  const int64_t outer = colwise ? cols : rows;       /* one line of blocks per row / column */
  const int64_t len = colwise ? rows : cols;         /* values along the quantised dimension */
  for (int64_t o = 0; o < outer; ++o)
    for (int64_t b = 0; b < len / 32; ++b) {
      float amax = 0.0f;
      for (int64_t t = 0; t < 32; ++t) {
        const int64_t i = colwise ? (b * 32 + t) * cols + o : o * cols + b * 32 + t;
        const float m = fabsf(x[i]);
        if (m > amax) amax = m;
      }
      int e = 0;
      if (amax > 0.0f) {
        e = floor_log2((double)amax) - fmt_emax(fmt);
        if (e < -127) e = -127;
        if (e > 127) e = 127;
      }
      const uint8_t scode = (uint8_t)(amax > 0.0f ? e + 127 : 127);
      scales[o * (len / 32) + b] = scode;
      const float inv = ldexpf(1.0f, 127 - (int)scode);   /* 2^-e */
      for (int64_t t = 0; t < 32; ++t) {
        const int64_t i = colwise ? (b * 32 + t) * cols + o : o * cols + b * 32 + t;
        const float y = x[i] * inv;
        const uint8_t q = encode_rne_sat((double)y, fmt);
        if (fmt == FMT_E2M1) {
          const int64_t k = b * 32 + t;
          uint8_t* byte = &codes[o * (cols / 2) + k / 2];
          if ((k & 1) == 0) *byte = (uint8_t)((*byte & 0xF0) | q);
          else *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
        } else {
          codes[i] = q;
        }
      }
    }
  return 0;
}

/* FP32 scale of one block: s = amax / 448, 1 when amax == 0, and never below the
 * smallest positive FP32 (2^-149), so that a block whose amax / 448 underflows (FP32
 * inputs under 448 * 2^-150) still divides by a positive number. */
static float group_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  const float s = amax / 448.0f;
  const float tiny = ldexpf(1.0f, -149);
  return s > tiny ? s : tiny;
}

/* Groupwise quantisation of activations X[total_M][K] (FP32 values) over 1x128 blocks.
 * codes [total_M][K]; sx in the per-group block layout: group g starts at
 * M_start_g * (K/128) and holds (local row l, block kb) at l + kb * m_g.
 * Returns 0, or -1 when K % 128 != 0 or m_sizes do not partition total_M. */
int oracle_fp8_group_quantize(const float* x, int64_t total_M, int64_t K,
                              const int64_t* m_sizes, int G, uint8_t* codes, float* sx) {
  init_tables();
  if (K % 128 != 0 || G < 1 || total_M < 0) return -1;
  int64_t sum = 0;
  for (int g = 0; g < G; ++g) {
    if (m_sizes[g] < 0) return -1;
    sum += m_sizes[g];
  }
  if (sum != total_M) return -1;
  const int64_t KB = K / 128;
  int64_t start = 0;
  for (int g = 0; g < G; ++g) {
    const int64_t mg = m_sizes[g];
    for (int64_t l = 0; l < mg; ++l) {
      const int64_t r = start + l;
      for (int64_t kb = 0; kb < KB; ++kb) {
        float amax = 0.0f;
        for (int64_t t = 0; t < 128; ++t) {
          const float m = fabsf(x[r * K + kb * 128 + t]);
          if (m > amax) amax = m;
        }
        const float s = group_scale(amax);
        sx[start * KB + l + kb * mg] = s;
        for (int64_t t = 0; t < 128; ++t) {
          const int64_t i = r * K + kb * 128 + t;
          codes[i] = encode_rne_sat((double)(x[i] / s), FMT_E4M3);
        }
      }
    }
    start += mg;
  }
  return 0;
}

/* Blockwise quantisation of weights W[G][N][K] (FP32 values) over 128x128 blocks.
 * codes [G][N][K]; sw [G][N/128][K/128].  Returns 0, or -1 unless N, K % 128 == 0. */
int oracle_fp8_block_quantize(const float* w, int64_t G, int64_t N, int64_t K, uint8_t* codes,
                              float* sw) {
  init_tables();
  if (N % 128 != 0 || K % 128 != 0 || G < 0) return -1;
  for (int64_t g = 0; g < G; ++g)
    for (int64_t nb = 0; nb < N / 128; ++nb)
      for (int64_t kb = 0; kb < K / 128; ++kb) {
        float amax = 0.0f;
        for (int64_t n = nb * 128; n < nb * 128 + 128; ++n)
          for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
            const float m = fabsf(w[(g * N + n) * K + k]);
            if (m > amax) amax = m;
          }
        const float s = group_scale(amax);
        sw[(g * (N / 128) + nb) * (K / 128) + kb] = s;
        for (int64_t n = nb * 128; n < nb * 128 + 128; ++n)
          for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
            const int64_t i = (g * N + n) * K + k;
            codes[i] = encode_rne_sat((double)(w[i] / s), FMT_E4M3);
          }
      }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Bias and activation after the GEMM ("[gfx1250] Add MXFP4 GEMM support to   */
/* FlyDSL backend", Description: activation and bias are a follow-up to the   */
/* plain GEMM).  D[i][n] <- act(D[i][n] + bias[n]) in FP64, bias optional      */
/* (FP32 values of the BF16 bias).  act: 0 none, 1 ReLU, 2 GELU (erf form:     */
/* x * (1 + erf(x / sqrt 2)) / 2), 3 SiLU (x / (1 + exp(-x))).                 */
/* ------------------------------------------------------------------------ */
int oracle_bias_act(double* D, int64_t rows, int64_t N, const float* bias, int act) {
  if (act < 0 || act > 3 || rows < 0 || N < 0) return -1;
  for (int64_t i = 0; i < rows; ++i)
    for (int64_t n = 0; n < N; ++n) {
      double v = D[i * N + n] + (bias ? (double)bias[n] : 0.0);
      switch (act) {
        case 1: v = v > 0.0 ? v : 0.0; break;
        case 2: v = 0.5 * v * (1.0 + erf(v / sqrt(2.0))); break;
        case 3: v = v / (1.0 + exp(-v)); break;
        default: break;
      }
      D[i * N + n] = v;
    }
  return 0;
}
