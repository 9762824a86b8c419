/*
 * gemm_oracle.c -- CPU oracle for the dense GEMM  C = alpha * op(A) * op(B) + beta * C0.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The GPU library never
 * links, loads or calls it, and it shares no code, header or table with the
 * GPU library.
 *
 * What it computes (the plain definition, written out):
 *   "CUDA GEMM 矩阵乘法优化指南", section 2.1 (GEMM): C = alpha*A*B + beta*C with
 *   A of size M x K, B of size K x N, C of size M x N; every output element
 *   takes K multiply-adds (2K floating-point operations).
 *   The page in m.lqnn.cn/news/285670, section 1.2, checks GPU results against
 *   a double-precision CPU product; this oracle does the same, in fp64, over
 *   the exact values of the bf16 / fp16 inputs the GPU receives.
 *
 *   For every (i, j):
 *     s_ij = sum_{k = 0 .. K-1} a(i, k) * b(k, j)        (fp64, k ascending)
 *     r_ij = alpha * s_ij + beta * c0_ij                  (c0 not read if beta == 0)
 *     m_ij = |alpha| * sum_k |a(i, k) * b(k, j)| + |beta| * |c0_ij|
 *   m_ij is the magnitude the comparison tolerance scales with.
 *
 * Storage convention (row-major, as C and PyTorch store matrices):
 *   transA == 0: A is stored M x K, a(i, k) = A[i * lda + k]
 *   transA == 1: A is stored K x M, a(i, k) = A[k * lda + i]
 *   transB == 0: B is stored K x N, b(k, j) = B[k * ldb + j]
 *   transB == 1: B is stored N x K, b(k, j) = B[j * ldb + k]
 *   C0 / R / Mag are M x N row-major with leading dimensions ldc / ldr.
 *
 * The inputs are decoded from their format definitions: IEEE 754 binary16;
 * bfloat16 = sign, 8-bit exponent with bias 127, 7-bit fraction; and the two
 * 8-bit formats the tensor core takes ("CUDA GEMM 矩阵乘法优化指南", 13.2:
 * FP8 E4M3 / E5M2; their bit layouts are the usual OCP 8-bit ones):
 *   E4M3: sign, 4-bit exponent with bias 7, 3-bit fraction; no infinities,
 *         exponent 1111 with fraction 111 is NaN, so the largest value is 448;
 *   E5M2: sign, 5-bit exponent with bias 15, 2-bit fraction, with IEEE-style
 *         infinities and NaNs.
 * A and B may have different types (an E4M3 x E5M2 product is allowed).
 * fp32 inputs (the FP32 GEMM that "GPU GEMM 优化完全拆解（三）", 数值精度,
 * emulates with three TF32 products) are exact in fp64 as they are; the
 * product of two has at most 48 significant bits, so it is exact too.
 * Every such value is exactly representable in fp64, and so is every
 * product of two of them (at most 22 significant bits), so the only rounding
 * in s_ij is that of the fp64 additions.
 *
 * Block-scaled inputs ("CUDA GEMM 矩阵乘法优化指南", 13.2: block scaling with
 * the FP4 / FP8 formats; MXFP8: every 32 consecutive elements share one E8M0
 * scale factor; NVFP4: every 16 share one E4M3 scale factor):
 *   a(i, k) = elem(A, i, k) * sf(SFA[i * ld_sfa + k / block])
 *   b(k, j) = elem(B, j, k) * sf(SFB[j * ld_sfb + k / block])
 * with A stored M x K and B stored N x K (K contiguous in both) and
 *   E8M0:  2^(x - 127), 255 is NaN (an exponent-only scale);
 *   UE4M3: the E4M3 value of the code with its sign bit ignored;
 *   E2M1 elements (FP4): sign, 2-bit exponent with bias 1, 1-bit fraction
 *          (values 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte, the even
 *          element of a pair in the low four bits.
 * Each a(i, k) * b(k, j) is a product of values with at most 4 significant
 * bits times powers of two, exact in fp64.
 *
 * Rows of C are split over POSIX threads; the loop body is the definition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

enum { ORACLE_IN_BF16 = 0, ORACLE_IN_F16 = 1, ORACLE_IN_E4M3 = 2, ORACLE_IN_E5M2 = 3, ORACLE_IN_F32 = 4,
       ORACLE_IN_E2M1 = 5 };
enum { ORACLE_SF_E8M0 = 0, ORACLE_SF_UE4M3 = 1 };
enum { ORACLE_C_F32 = 0, ORACLE_C_BF16 = 1, ORACLE_C_F16 = 2 };

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xFF;
  int f = h & 0x7F;
  double v;
  if (e == 0xFF) {
    v = (f == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    v = ldexp((double)f / 128.0, -126); /* subnormal: 0.f * 2^(1-127) */
  } else {
    v = ldexp(1.0 + (double)f / 128.0, e - 127);
  }
  return sign ? -v : v;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0x1F) {
    v = (f == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    v = ldexp((double)f / 1024.0, -14); /* subnormal: 0.f * 2^(1-15) */
  } else {
    v = ldexp(1.0 + (double)f / 1024.0, e - 15);
  }
  return sign ? -v : v;
}

/* FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; S.1111.111 is NaN. */
double oracle_e4m3_value(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int f = b & 0x7;
  double v;
  if (e == 0xF && f == 0x7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)f / 8.0, -6); /* subnormal: 0.f * 2^(1-7) */
  } else {
    v = ldexp(1.0 + (double)f / 8.0, e - 7);
  }
  return sign ? -v : v;
}

/* FP8 E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits, IEEE-style specials. */
double oracle_e5m2_value(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 2) & 0x1F;
  int f = b & 0x3;
  double v;
  if (e == 0x1F) {
    v = (f == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    v = ldexp((double)f / 4.0, -14); /* subnormal: 0.f * 2^(1-15) */
  } else {
    v = ldexp(1.0 + (double)f / 4.0, e - 15);
  }
  return sign ? -v : v;
}

/* FP4 E2M1 (low four bits of x): 1 sign bit, 2 exponent bits (bias 1), 1 fraction bit. */
double oracle_e2m1_value(uint8_t x) {
  int sign = (x >> 3) & 1;
  int e = (x >> 1) & 0x3;
  int f = x & 0x1;
  double v = e == 0 ? (double)f / 2.0 /* subnormal: 0.f * 2^(1-1) */ : ldexp(1.0 + (double)f / 2.0, e - 1);
  return sign ? -v : v;
}

/* E8M0 scale factor: 2^(x - 127); 255 is NaN. */
double oracle_e8m0_value(uint8_t x) { return x == 255 ? NAN : ldexp(1.0, (int)x - 127); }

/* Unsigned E4M3 scale factor: the E4M3 value with the sign bit ignored. */
double oracle_ue4m3_value(uint8_t x) { return oracle_e4m3_value((uint8_t)(x & 0x7F)); }

/* Element idx of a stored matrix of the given input type. */
static double in_value(int in_type, const void* base, int64_t idx) {
  switch (in_type) {
    case ORACLE_IN_E2M1: {
      const uint8_t byte = ((const uint8_t*)base)[idx >> 1];
      return oracle_e2m1_value((idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF));
    }
    case ORACLE_IN_F16: return oracle_f16_value(((const uint16_t*)base)[idx]);
    case ORACLE_IN_E4M3: return oracle_e4m3_value(((const uint8_t*)base)[idx]);
    case ORACLE_IN_E5M2: return oracle_e5m2_value(((const uint8_t*)base)[idx]);
    case ORACLE_IN_F32: return (double)((const float*)base)[idx]; /* exact in fp64 */
    default: return oracle_bf16_value(((const uint16_t*)base)[idx]);
  }
}

/* Bytes per element (0 for E2M1, which packs two to a byte). */
static int64_t elem_bytes(int in_type) {
  if (in_type == ORACLE_IN_E2M1) return 0;
  return (in_type == ORACLE_IN_E4M3 || in_type == ORACLE_IN_E5M2) ? 1 : in_type == ORACLE_IN_F32 ? 4 : 2;
}

static double c0_value(int c_type, const void* C0, int64_t idx) {
  if (c_type == ORACLE_C_F32) return (double)((const float*)C0)[idx];
  if (c_type == ORACLE_C_BF16) return oracle_bf16_value(((const uint16_t*)C0)[idx]);
  return oracle_f16_value(((const uint16_t*)C0)[idx]);
}

typedef struct {
  int transA, transB, a_type, b_type, c_type;
  int64_t M, N, K, lda, ldb, ldc, ldr;
  double alpha, beta;
  const void* A;
  const void* B;
  const void* C0;
  /* block scaling (block > 0): scale factors of A's and B's blocks of k */
  int64_t block, ld_sfa, ld_sfb;
  int sf_type;
  const uint8_t* SFA;
  const uint8_t* SFB;
  /* full mode: rows [row0, row1) of R / Mag */
  double* R;
  double* Mag;
  int64_t row0, row1;
  /* sampled mode: entries [e0, e1) of (rows, cols) */
  const int64_t* rows;
  const int64_t* cols;
  int64_t e0, e1;
} job_t;

static double sf_value(int sf_type, uint8_t x) {
  return sf_type == ORACLE_SF_UE4M3 ? oracle_ue4m3_value(x) : oracle_e8m0_value(x);
}

/* One output element, straight from the definition. */
static void element(const job_t* J, int64_t i, int64_t j, double* r, double* m) {
  double s = 0.0, sa = 0.0;
  for (int64_t k = 0; k < J->K; ++k) {
    double a = in_value(J->a_type, J->A, J->transA ? k * J->lda + i : i * J->lda + k);
    double b = in_value(J->b_type, J->B, J->transB ? j * J->ldb + k : k * J->ldb + j);
    if (J->block > 0) {
      a *= sf_value(J->sf_type, J->SFA[i * J->ld_sfa + k / J->block]);
      b *= sf_value(J->sf_type, J->SFB[j * J->ld_sfb + k / J->block]);
    }
    double p = a * b;
    s += p;
    sa += fabs(p);
  }
  double rv = J->alpha * s;
  double mv = fabs(J->alpha) * sa;
  if (J->beta != 0.0) {
    double c0 = c0_value(J->c_type, J->C0, i * J->ldc + j);
    rv += J->beta * c0;
    mv += fabs(J->beta) * fabs(c0);
  }
  *r = rv;
  *m = mv;
}

static void* run_rows(void* arg) {
  const job_t* J = (const job_t*)arg;
  for (int64_t i = J->row0; i < J->row1; ++i)
    for (int64_t j = 0; j < J->N; ++j)
      element(J, i, j, &J->R[i * J->ldr + j], &J->Mag[i * J->ldr + j]);
  return NULL;
}

static void* run_entries(void* arg) {
  const job_t* J = (const job_t*)arg;
  for (int64_t e = J->e0; e < J->e1; ++e) element(J, J->rows[e], J->cols[e], &J->R[e], &J->Mag[e]);
  return NULL;
}

static int pick_threads(int nthreads, int64_t work_items) {
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > 256) nthreads = 256;
  if (work_items < nthreads) nthreads = work_items > 0 ? (int)work_items : 1;
  return nthreads;
}

static int run_jobs(job_t* jobs, int nthreads, void* (*fn)(void*)) {
  pthread_t tid[256];
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&tid[t], NULL, fn, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  /* any job whose thread could not be started runs on the caller */
  for (int t = started; t < nthreads; ++t) fn(&jobs[t]);
  return nthreads;
}

static int check_args(int transA, int transB, int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int a_type, int b_type, int c_type) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return -1;
  if (a_type < ORACLE_IN_BF16 || a_type > ORACLE_IN_E2M1) return -1;
  if (b_type < ORACLE_IN_BF16 || b_type > ORACLE_IN_E2M1) return -1;
  if (c_type != ORACLE_C_F32 && c_type != ORACLE_C_BF16 && c_type != ORACLE_C_F16) return -1;
  if (lda < (transA ? M : K) || ldb < (transB ? K : N)) return -1;
  return 0;
}

/*
 * Full oracle: R and Mag (M x N, leading dimension ldr) receive r_ij and m_ij.
 * A holds elements of a_type, B of b_type (2-byte codes for bf16 / fp16,
 * 1-byte codes for E4M3 / E5M2).  nthreads <= 0 uses every online core.
 * Returns the number of threads used, or -1 on a bad argument.
 */
int oracle_gemm_ab(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                   const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                   const void* C0, int c_type, int64_t ldc, int a_type, int b_type, double* R,
                   double* Mag, int64_t ldr, int nthreads) {
  if (check_args(transA, transB, M, N, K, lda, ldb, a_type, b_type, c_type) != 0) return -1;
  if (ldr < N || (beta != 0.0 && ldc < N)) return -1;
  if (M == 0 || N == 0) return 0;
  nthreads = pick_threads(nthreads, M);
  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  if (!jobs) return -1;
  for (int t = 0; t < nthreads; ++t) {
    job_t* J = &jobs[t];
    J->transA = transA; J->transB = transB; J->a_type = a_type; J->b_type = b_type;
    J->c_type = c_type;
    J->M = M; J->N = N; J->K = K; J->lda = lda; J->ldb = ldb; J->ldc = ldc; J->ldr = ldr;
    J->alpha = alpha; J->beta = beta; J->A = A; J->B = B; J->C0 = C0;
    J->R = R; J->Mag = Mag;
    J->row0 = M * t / nthreads;
    J->row1 = M * (t + 1) / nthreads;
  }
  int used = run_jobs(jobs, nthreads, run_rows);
  free(jobs);
  return used;
}

/* Both operands of one type. */
int oracle_gemm(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                const void* C0, int c_type, int64_t ldc, int in_type, double* R, double* Mag,
                int64_t ldr, int nthreads) {
  return oracle_gemm_ab(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C0, c_type, ldc,
                        in_type, in_type, R, Mag, ldr, nthreads);
}

/*
 * Sampled oracle: for e in [0, count), R[e] / Mag[e] receive r and m at
 * (rows[e], cols[e]).  Used where the full product would take too long.
 */
int oracle_gemm_at_ab(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                      const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                      const void* C0, int c_type, int64_t ldc, int a_type, int b_type,
                      int64_t count, const int64_t* rows, const int64_t* cols, double* R,
                      double* Mag, int nthreads) {
  if (check_args(transA, transB, M, N, K, lda, ldb, a_type, b_type, c_type) != 0) return -1;
  if (beta != 0.0 && ldc < N) return -1;
  for (int64_t e = 0; e < count; ++e)
    if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -1;
  if (count == 0) return 0;
  nthreads = pick_threads(nthreads, count);
  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  if (!jobs) return -1;
  for (int t = 0; t < nthreads; ++t) {
    job_t* J = &jobs[t];
    J->transA = transA; J->transB = transB; J->a_type = a_type; J->b_type = b_type;
    J->c_type = c_type;
    J->M = M; J->N = N; J->K = K; J->lda = lda; J->ldb = ldb; J->ldc = ldc; J->ldr = 0;
    J->alpha = alpha; J->beta = beta; J->A = A; J->B = B; J->C0 = C0;
    J->R = R; J->Mag = Mag; J->rows = rows; J->cols = cols;
    J->e0 = count * t / nthreads;
    J->e1 = count * (t + 1) / nthreads;
  }
  int used = run_jobs(jobs, nthreads, run_entries);
  free(jobs);
  return used;
}

int oracle_gemm_at(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                   const void* A, int64_t lda, const void* B, int64_t ldb, double beta,
                   const void* C0, int c_type, int64_t ldc, int in_type, int64_t count,
                   const int64_t* rows, const int64_t* cols, double* R, double* Mag,
                   int nthreads) {
  return oracle_gemm_at_ab(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C0, c_type, ldc,
                           in_type, in_type, count, rows, cols, R, Mag, nthreads);
}

/*
 * Fused epilogue, applied in place to R / Mag produced by oracle_gemm (M x N,
 * leading dimension ldr).  The pages name the operations fused into a GEMM's
 * write-back: "第4章：经典算子实现 —— GEMM", section 7.2 (GEMM + bias +
 * activation) and "GPU GEMM 优化完全拆解（三）", mainloop 与 epilogue (elementwise
 * ReLU and quantisation scaling before the store).  Written out:
 *   z_ij   = r_ij + bias_j                    (bias: N fp32 values, or NULL)
 *   d_ij   = act(z_ij)                        act 0: z;  1 (ReLU): max(z, 0);
 *                                             2 (GELU): z * Phi(z) = z * (1 + erf(z / sqrt 2)) / 2
 *   out_ij = scale * d_ij
 * and the tolerance magnitude follows the same steps:
 *   m'_ij  = |scale| * L * (m_ij + |bias_j|),  L = 1 (identity, ReLU) or 1.13 (GELU, whose
 *                                             slope lies in [-0.129, 1.129]).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_epilogue(int64_t M, int64_t N, double* R, double* Mag, int64_t ldr, const float* bias,
                    int act, double scale) {
  if (M < 0 || N < 0 || ldr < N || act < 0 || act > 2) return -1;
  const double lip = act == 2 ? 1.13 : 1.0;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double z = R[i * ldr + j];
      double m = Mag[i * ldr + j];
      if (bias) {
        z += (double)bias[j];
        m += fabs((double)bias[j]);
      }
      double d = z;
      if (act == 1) d = z > 0.0 ? z : 0.0;
      if (act == 2) d = 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
      R[i * ldr + j] = scale * d;
      Mag[i * ldr + j] = fabs(scale) * lip * m;
    }
  }
  return 0;
}

/*
 * Strided batched oracle: for b in [0, batch), the GEMM above on
 *   A_b = A + b * strideA,  B_b = B + b * strideB,  C0_b / R_b / Mag_b = ... + b * stride
 * (strides in elements; a stride of 0 reuses one operand for every batch).
 * This is the product a batched attention score or value GEMM computes per
 * (batch, head) pair ("第4章：经典算子实现 —— GEMM", section 1: Q (B*H, S, d) x K^T).
 * R / Mag hold batch x M x N, leading dimension ldr, batch stride M * ldr.
 * Returns the threads used by the last batch, or -1 on a bad argument.
 */
int oracle_gemm_batched(int transA, int transB, int64_t M, int64_t N, int64_t K, double alpha,
                        const void* A, int64_t lda, int64_t strideA, const void* B, int64_t ldb,
                        int64_t strideB, double beta, const void* C0, int c_type, int64_t ldc,
                        int64_t strideC, int a_type, int b_type, int64_t batch, double* R,
                        double* Mag, int64_t ldr, int nthreads) {
  if (batch < 0 || strideA < 0 || strideB < 0 || strideC < 0) return -1;
  const int64_t ea = elem_bytes(a_type);
  const int64_t eb = elem_bytes(b_type);
  if (ea == 0 || eb == 0) return -1;  /* packed FP4: block-scaled entry point only */
  const int64_t ec = c_type == ORACLE_C_F32 ? 4 : 2;
  int used = 0;
  for (int64_t b = 0; b < batch; ++b) {
    const char* Ab = (const char*)A + b * strideA * ea;
    const char* Bb = (const char*)B + b * strideB * eb;
    const char* Cb = C0 ? (const char*)C0 + b * strideC * ec : NULL;
    used = oracle_gemm_ab(transA, transB, M, N, K, alpha, Ab, lda, Bb, ldb, beta, Cb, c_type, ldc,
                          a_type, b_type, R + b * M * ldr, Mag + b * M * ldr, ldr, nthreads);
    if (used < 0) return -1;
  }
  return used;
}

/*
 * Grouped oracle (mixture-of-experts routing, the grouped GEMM of DeepGEMM that
 * "第4章：经典算子实现 —— GEMM" points to for MoE): `groups` GEMMs whose
 * rows are stacked.  Group g owns rows [off_g, off_g + m_sizes[g]) of A (stored
 * sum(m) x K, row-major, lda) and of C / R / Mag (sum(m) x N), off_g being the
 * sum of the sizes before it, and multiplies them by its own B_g = B + g * strideB
 * (transB as in oracle_gemm):
 *   R[off_g + i][j] = alpha * sum_k A[off_g + i][k] * b_g(k, j) + beta * C0[off_g + i][j].
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm_grouped(int transB, int64_t groups, const int64_t* m_sizes, int64_t N, int64_t K,
                        double alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                        int64_t strideB, double beta, const void* C0, int c_type, int64_t ldc,
                        int a_type, int b_type, double* R, double* Mag, int64_t ldr, int nthreads) {
  if (groups < 0 || strideB < 0) return -1;
  const int64_t ea = elem_bytes(a_type);
  const int64_t eb = elem_bytes(b_type);
  if (ea == 0 || eb == 0) return -1;  /* packed FP4: block-scaled entry point only */
  const int64_t ec = c_type == ORACLE_C_F32 ? 4 : 2;
  int64_t off = 0;
  for (int64_t g = 0; g < groups; ++g) {
    const int64_t m = m_sizes[g];
    if (m < 0) return -1;
    const char* Ag = (const char*)A + off * lda * ea;
    const char* Bg = (const char*)B + g * strideB * eb;
    const char* Cg = C0 ? (const char*)C0 + off * ldc * ec : NULL;
    if (m > 0 && oracle_gemm_ab(0, transB, m, N, K, alpha, Ag, lda, Bg, ldb, beta, Cg, c_type, ldc,
                                a_type, b_type, R + off * ldr, Mag + off * ldr, ldr, nthreads) < 0)
      return -1;
    off += m;
  }
  return 0;
}

/*
 * Block-scaled oracle (see the header): A stored M x K, B stored N x K, both
 * with K contiguous (lda, ldb in elements; even for E2M1), a_type / b_type
 * E4M3, E5M2 or E2M1; SFA M x ceil(K / block) and SFB N x ceil(K / block)
 * scale codes of sf_type, row pitches ld_sfa / ld_sfb.  Full mode when rows ==
 * NULL (R, Mag M x N with leading dimension ldr), else the `count` entries
 * (rows[e], cols[e]).  Returns the number of threads used, or -1.
 */
int oracle_gemm_block_scaled(int64_t M, int64_t N, int64_t K, double alpha, const void* A, int64_t lda,
                             const uint8_t* SFA, int64_t ld_sfa, const void* B, int64_t ldb,
                             const uint8_t* SFB, int64_t ld_sfb, double beta, const void* C0,
                             int c_type, int64_t ldc, int a_type, int b_type, int sf_type, int64_t block,
                             int64_t count, const int64_t* rows, const int64_t* cols, double* R,
                             double* Mag, int64_t ldr, int nthreads) {
  if (check_args(0, 1, M, N, K, lda, ldb, a_type, b_type, c_type) != 0) return -1;
  if (block <= 0 || (sf_type != ORACLE_SF_E8M0 && sf_type != ORACLE_SF_UE4M3)) return -1;
  const int64_t nblk = (K + block - 1) / block;
  if (ld_sfa < nblk || ld_sfb < nblk || (K > 0 && (!SFA || !SFB))) return -1;
  if (beta != 0.0 && ldc < N) return -1;
  if (!rows && ldr < N) return -1;
  if (rows)
    for (int64_t e = 0; e < count; ++e)
      if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -1;
  const int64_t items = rows ? count : M;
  if (items == 0 || (!rows && N == 0)) return 0;
  nthreads = pick_threads(nthreads, items);
  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  if (!jobs) return -1;
  for (int t = 0; t < nthreads; ++t) {
    job_t* J = &jobs[t];
    J->transA = 0; J->transB = 1; J->a_type = a_type; J->b_type = b_type; J->c_type = c_type;
    J->M = M; J->N = N; J->K = K; J->lda = lda; J->ldb = ldb; J->ldc = ldc; J->ldr = ldr;
    J->alpha = alpha; J->beta = beta; J->A = A; J->B = B; J->C0 = C0;
    J->block = block; J->ld_sfa = ld_sfa; J->ld_sfb = ld_sfb; J->sf_type = sf_type;
    J->SFA = SFA; J->SFB = SFB;
    J->R = R; J->Mag = Mag; J->rows = rows; J->cols = cols;
    if (rows) {
      J->e0 = count * t / nthreads;
      J->e1 = count * (t + 1) / nthreads;
    } else {
      J->row0 = M * t / nthreads;
      J->row1 = M * (t + 1) / nthreads;
    }
  }
  int used = run_jobs(jobs, nthreads, rows ? run_entries : run_rows);
  free(jobs);
  return used;
}
