/*
 * gemm_gb300.h -- C ABI of a GB300 (sm_103a) dense GEMM library.
 *
 * The operation (all entry points):
 *   C = alpha * op(A) * op(B) + beta * C
 * with op(A) of size M x K, op(B) of size K x N and C of size M x N; 2*M*N*K
 * floating-point operations.  This is the GEMM of "CUDA GEMM 矩阵乘法优化指南"
 * (blog.zhenwei.site), section 2.1, with the op / alpha / beta calling shape of
 * the cuBLAS call in "第4章：经典算子实现 —— GEMM" (aiinfra.vidrealm.tech),
 * section 7.1.  Inputs are bf16, fp16 or 8-bit floats (E4M3 / E5M2; see
 * gemm_dtype_t), products are accumulated in fp32 on
 * the tensor cores (tcgen05.mma into Tensor Memory), and alpha / beta are
 * applied in fp32 before the result is rounded (round-to-nearest-even) to the
 * type of C.
 *
 * Storage is row-major (the C / PyTorch convention):
 *   transA == GEMM_OP_N : A is stored M x K, element (i, k) at A[i * lda + k], lda >= K
 *   transA == GEMM_OP_T : A is stored K x M, element (i, k) at A[k * lda + i], lda >= M
 *   transB == GEMM_OP_N : B is stored K x N, element (k, j) at B[k * ldb + j], ldb >= N
 *   transB == GEMM_OP_T : B is stored N x K, element (k, j) at B[j * ldb + k], ldb >= K
 *   C is M x N, element (i, j) at C[i * ldc + j], ldc >= N.
 * So "A row-major, B column-major" is (GEMM_OP_N, GEMM_OP_T), the NT layout.
 *
 * Every entry point returns a gemm_status_t and never throws.  No call here
 * allocates or frees the caller's A, B or C.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque library handle, bound to one CUDA device. */
typedef struct gemm_handle_s* gemm_handle_t;

typedef enum { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op_t;

/*
 * Input types -> type of C.  Accumulation is fp32 in every case.
 *
 * The 8-bit float inputs are the tensor core's FP8 formats ("CUDA GEMM
 * 矩阵乘法优化指南", section 13.2: E4M3 / E5M2, issued as tcgen05.mma
 * kind::f8f6f4 with 32 products of k per instruction), in the OCP 8-bit
 * layouts: E4M3 = sign, 4-bit exponent (bias 7), 3-bit fraction, no
 * infinities, largest value 448; E5M2 = sign, 5-bit exponent (bias 15),
 * 2-bit fraction, IEEE-style infinities and NaNs.  A and B may differ.  With
 * 8-bit inputs both operands must be K-major (transA == GEMM_OP_N and
 * transB == GEMM_OP_T: A stored M x K, B stored N x K, the usual layout of
 * FP8 weights); other layouts return GEMM_ERR_UNSUPPORTED.  Leading dimensions
 * are in elements (= bytes); the code is 16 + (A is E5M2) + 2 * (B is E5M2) +
 * 4 * (0 for fp32 C, 1 for bf16 C, 2 for fp16 C, 3 for E4M3 C).  Per-tensor
 * scale factors of FP8 data fold into alpha.
 *
 * fp32 inputs ("GPU GEMM 优化完全拆解（三）", section 数值精度: the tensor cores
 * take no fp32 operands; TF32 keeps the sign, the 8-bit exponent and 10
 * fraction bits; three TF32 products emulate one fp32 product) run on the
 * tensor core's TF32 kind (tcgen05.mma kind::tf32, 8 products of k per
 * instruction) and write fp32 C:
 *   GEMM_F32_F32   the fp32 GEMM: each value x is split into hi = TF32(x) and
 *                  lo = TF32(x - hi) (rounded to nearest) and every product is
 *                  lo_a hi_b + hi_a lo_b + hi_a hi_b, which misses a * b by
 *                  about 2^-21 of |a b|.  Both operands are first written
 *                  K-major into the workspace as two TF32 segments (two more
 *                  launches, twice the operand bytes), then one TF32 GEMM
 *                  over three segments of k sums the three products.
 *   GEMM_TF32_F32  one TF32 product per product: the 13 low fraction bits of
 *                  every input are dropped (about 2^-10 of each value).  A
 *                  K-major operand (A with transA == GEMM_OP_N, B with transB
 *                  == GEMM_OP_T) that the copy engine can load is read as it
 *                  is; any other is first written K-major, cut the same way.
 * Leading dimensions and strides are in elements (4 bytes).
 *
 * E4M3 C is a quantised output: the fp32 result (after the fused epilogue of
 * gemm_run_ex, whose out_scale is the quantisation scale) is rounded to
 * nearest even and saturated to +-448.  It is written only: beta must be 0
 * (else GEMM_ERR_UNSUPPORTED).
 */
typedef enum {
  GEMM_BF16_F32 = 0,  /* A, B bf16; C fp32 */
  GEMM_BF16_BF16 = 1, /* A, B bf16; C bf16 */
  GEMM_F16_F32 = 2,   /* A, B fp16; C fp32 */
  GEMM_F16_F16 = 3,   /* A, B fp16; C fp16 */
  GEMM_BF16_E4M3 = 4, /* A, B bf16; C E4M3 (quantised output) */
  GEMM_F16_E4M3 = 5,  /* A, B fp16; C E4M3 (quantised output) */
  GEMM_F32_F32 = 6,   /* A, B fp32; C fp32: three TF32 products per product */
  GEMM_TF32_F32 = 7,  /* A, B fp32 read as TF32; C fp32: one TF32 product */
  GEMM_E4M3_F32 = 16,        /* A, B E4M3; C fp32 */
  GEMM_E5M2_E4M3_F32 = 17,   /* A E5M2, B E4M3; C fp32 */
  GEMM_E4M3_E5M2_F32 = 18,   /* A E4M3, B E5M2; C fp32 */
  GEMM_E5M2_F32 = 19,        /* A, B E5M2; C fp32 */
  GEMM_E4M3_BF16 = 20,       /* ... the same pairs with bf16 C */
  GEMM_E5M2_E4M3_BF16 = 21,
  GEMM_E4M3_E5M2_BF16 = 22,
  GEMM_E5M2_BF16 = 23,
  GEMM_E4M3_F16 = 24,        /* ... and with fp16 C */
  GEMM_E5M2_E4M3_F16 = 25,
  GEMM_E4M3_E5M2_F16 = 26,
  GEMM_E5M2_F16 = 27,
  GEMM_E4M3_E4M3OUT = 28,      /* ... and with E4M3 C (quantised output) */
  GEMM_E5M2_E4M3_E4M3OUT = 29,
  GEMM_E4M3_E5M2_E4M3OUT = 30,
  GEMM_E5M2_E4M3OUT = 31,
  /* Block-scaled inputs, gemm_run_block_scaled only (see there):
     MXFP8: 32 + (A is E5M2) + 2 * (B is E5M2) + 4 * (0 fp32, 1 bf16, 2 fp16 C) */
  GEMM_MXFP8_F32 = 32,         /* A, B E4M3 with E8M0 scales per 32; C fp32 */
  GEMM_MXFP8_E5M2_F16 = 43,    /* the last MXFP8 code: A, B E5M2; C fp16 */
  GEMM_NVFP4_F32 = 48,         /* A, B E2M1 (packed) with unsigned E4M3 scales per 16; C fp32 */
  GEMM_NVFP4_BF16 = 49,
  GEMM_NVFP4_F16 = 50
} gemm_dtype_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1, /* null pointer, negative size, leading dimension too small, bad enum */
  GEMM_ERR_UNSUPPORTED = 2, /* a size the library cannot index (an extent >= 2^31), or an
                               8-bit input layout other than A M x K, B N x K */
  GEMM_ERR_NO_DEVICE = 3,   /* the device is absent or is not sm_103 */
  GEMM_ERR_CUDA = 4,        /* a CUDA runtime call failed; gemm_last_cuda_error() tells which */
  GEMM_ERR_TENSORMAP = 5,   /* cuTensorMapEncodeTiled refused an operand description */
  GEMM_ERR_TIMEOUT = 6,     /* a kernel gave up waiting on one of its barriers (see gemm_get_status) */
  GEMM_ERR_WORKSPACE = 7    /* the handle could not grow its device workspace */
} gemm_status_t;

/*
 * gemm_create: make a handle for CUDA device `device` (the ordinal).
 * Allocates the handle's device status word and tile counters on that
 * device.  *out is set to NULL on failure.  Errors: GEMM_ERR_INVALID_ARG (out
 * is NULL), GEMM_ERR_NO_DEVICE, GEMM_ERR_CUDA.
 */
gemm_status_t gemm_create(gemm_handle_t* out, int device);

/*
 * gemm_run: enqueue C = alpha * op(A) * op(B) + beta * C on `stream`
 * (a cudaStream_t; NULL is the legacy default stream).  Asynchronous: it
 * returns once the kernels are launched and never synchronises.
 *
 *   transA, transB  GEMM_OP_N / GEMM_OP_T, layouts above.
 *   M, N, K         sizes, >= 0.  M == 0 or N == 0 is a no-op returning GEMM_OK.
 *                   K == 0 sets C = beta * C (C = 0 when beta == 0).
 *   alpha, beta     fp32 scalars, read on the host.  When beta == 0, C is not
 *                   read, so C may hold anything (NaN included) on entry.
 *   A, B, C         caller-owned device pointers, of the types `dtype` names.
 *                   A and B are read only; C is read (beta != 0) and written.
 *                   C must not overlap A or B.
 *   lda, ldb, ldc   leading dimensions in elements, per the layouts above.
 *   dtype           gemm_dtype_t.
 *
 * Operands whose base address is not 16-byte aligned, or whose row pitch in
 * bytes is not a multiple of 16, are first copied by a device kernel into an
 * aligned buffer owned by the handle (the tensor-memory-accelerator copy
 * engine reads only 16-byte aligned rows); a C with such a pitch is written by
 * the scalar-store epilogue.  The handle's workspace grows on demand with
 * cudaMalloc (synchronous), so the first call of a new shape may block.
 *
 * The handle's workspace is shared by all calls on it: do not run one handle
 * on two streams at once.  Errors are returned synchronously for bad
 * arguments and failed launches; a kernel that times out on a barrier is
 * reported later by gemm_get_status.
 */
gemm_status_t gemm_run(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N,
                       int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                       int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtype_t dtype,
                       void* stream);

/*
 * Fused epilogue: elementwise operations applied to each element of the
 * result before it is stored, in this order ("第4章：经典算子实现 —— GEMM",
 * section 7.2: GEMM + bias + activation; "GPU GEMM 优化完全拆解（三）",
 * mainloop 与 epilogue: ReLU and quantisation scaling before write-back):
 *   z = alpha * op(A) * op(B) + beta * C + bias[j]
 *   C = convert(out_scale * act(z))
 * act: GEMM_ACT_NONE (identity), GEMM_ACT_RELU max(z, 0), GEMM_ACT_GELU
 * z * Phi(z) = z * (1 + erf(z / sqrt 2)) / 2 (the exact form, evaluated in
 * fp32 with the device erff).
 */
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU = 2 } gemm_activation_t;

typedef struct {
  const float* bias;   /* device pointer to N fp32 values, one per column j of C, read only;
                          NULL for none.  Must be 4-byte aligned. */
  int32_t activation;  /* gemm_activation_t */
  float out_scale;     /* finite; multiplies act(z) before the conversion to C's type (the
                          quantisation scale for E4M3 C); 1 for none */
} gemm_epilogue_t;

/*
 * gemm_run_ex: gemm_run with the fused epilogue `epi` (NULL = none, the same as
 * gemm_run).  The operations cost no extra pass over C: they are applied in the
 * kernel's epilogue (and by the K == 0 kernel, where z = beta * C + bias).
 * Errors: those of gemm_run, and GEMM_ERR_INVALID_ARG for an unknown
 * activation, a non-finite out_scale or a misaligned bias.
 */
gemm_status_t gemm_run_ex(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N,
                          int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                          int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtype_t dtype,
                          const gemm_epilogue_t* epi, void* stream);

/*
 * gemm_run_strided_batched: `batch` independent GEMMs in one launch,
 *   C_b = alpha * op(A_b) * op(B_b) + beta * C_b   (with the fused epilogue epi, may be NULL)
 * where A_b = A + b * strideA, B_b = B + b * strideB and C_b = C + b * strideC
 * (strides in elements of each matrix's type), b = 0 .. batch - 1.  This is
 * the shape of attention's per-(batch, head) products, Q (B*H, S, d) x K^T
 * ("第4章：经典算子实现 —— GEMM", section 1), with the batch taken as a third
 * dimension of the tensor-memory-accelerator copies ("CUDA GEMM 矩阵乘法优化
 * 指南", 12.2: 3-D copies for attention heads).  All batches share one
 * persistent schedule (their tiles follow one another), so a batch of small
 * GEMMs still fills the GPU.
 *   strideA / strideB  >= 0; 0 reuses one A (or B) for every batch.
 *   strideC            >= (M - 1) * ldc + N when batch > 1 (no two C_b overlap).
 *   bias (epi)         one value per column, the same for every batch.
 * batch == 0 is a no-op.  Other arguments, layouts and errors as in gemm_run
 * and gemm_run_ex; GEMM_ERR_UNSUPPORTED when the tiles of all batches exceed
 * 2^30.
 */
gemm_status_t gemm_run_strided_batched(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M,
                                       int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                                       int64_t strideA, const void* B, int64_t ldb, int64_t strideB,
                                       float beta, void* C, int64_t ldc, int64_t strideC, int64_t batch,
                                       gemm_dtype_t dtype, const gemm_epilogue_t* epi, void* stream);

/*
 * gemm_get_status: synchronise `stream`, then read and clear the handle's
 * device status word.  Returns GEMM_OK, GEMM_ERR_TIMEOUT (a kernel waited
 * longer than the wait limit on one of its barriers and returned early; C is
 * then incomplete) or GEMM_ERR_CUDA (the synchronisation itself failed).
 * *detail (may be NULL) receives the raw status word: 0, or the role and
 * barrier that gave up (see gemm_status_string for the code only).
 */
gemm_status_t gemm_get_status(gemm_handle_t h, void* stream, int32_t* detail);

/* A static, human-readable string for a status code. */
const char* gemm_status_string(gemm_status_t s);

/* The last CUDA error code (cudaError_t as int) the handle saw, 0 if none. */
int gemm_last_cuda_error(gemm_handle_t h);

/*
 * gemm_destroy: free the handle and its device memory.  Synchronises the
 * device first.  Passing NULL is a no-op returning GEMM_OK.
 */
gemm_status_t gemm_destroy(gemm_handle_t h);

/* ---------------------------------------------------------------------------
 * Planning and tuning.
 *
 * The planner maps a call to one kernel configuration: the operands' major
 * modes, the output tile, the k-split for shapes with too few tiles to fill
 * the GPU, and whether the operands must be swapped (C^T = op(B)^T op(A)^T)
 * so that a short M rides on the MMA's N dimension.  These choices follow the
 * tiling, split-K and rasterisation designs of "GPU GEMM 优化完全拆解（三）"
 * (pinghaoyang.com.cn), sections "双缓冲的两个 scope、rasterization 与 Split-K"
 * and "Hopper 时代的三种 kernel 设计".
 * ------------------------------------------------------------------------- */

typedef enum {
  GEMM_PATH_NOOP = 0,      /* M == 0 or N == 0 */
  GEMM_PATH_SCALE_C = 1,   /* K == 0: C = beta * C */
  GEMM_PATH_TC_1CTA = 2,   /* persistent tcgen05 kernel, one CTA per output tile (cta_group::1) */
  GEMM_PATH_TC_2CTA = 3    /* persistent tcgen05 kernel, CTA pairs share a 256-row tile (cta_group::2) */
} gemm_path_t;

/* How C leaves the epilogue (gemm_plan_t.bulk_store). */
typedef enum {
  GEMM_BULK_NONE = 0,       /* direct stores by the epilogue warps (beta != 0, 8-bit C, grouped GEMMs,
                               small C that bulk stores cannot write) */
  GEMM_BULK_ROWS = 1,       /* bulk tensor stores of rows of C */
  GEMM_BULK_TRANSPOSED = 2, /* bulk tensor stores of transposed blocks (swapped problems) */
  GEMM_BULK_STAGED = 3,     /* C's rows are misaligned, or end inside a 16-byte piece, K < 2048 and
                               GEMM_BULK_ROW_CLASSES does not apply:
                               bulk tensor stores write an aligned copy of C in the handle's workspace
                               and a copy kernel then writes C's M x N elements (one more launch;
                               beta == 0, unswapped, one GEMM, M * N >= 2^20) */
  GEMM_BULK_ROW_COPIES = 4, /* C's rows are misaligned, or end inside a 16-byte piece (beta == 0,
                               unswapped, not grouped; where GEMM_BULK_STAGED is not chosen): each
                               row of a block leaves through one 1-D bulk copy of its whole 16-byte
                               pieces; the partial pieces at a tile's first and last columns are
                               written by plain stores.  No workspace for C, no second launch */
  GEMM_BULK_ROW_CLASSES = 5 /* fp32 C whose rows are misaligned (beta == 0, unswapped, one GEMM, at
                               least 4 rows): the rows fall into 1, 2 or 4 classes of one misalignment
                               each, whose rows lie a multiple of 16 bytes apart; each class is
                               described as a tensor of its own and a block of C leaves through one
                               bulk tensor store per class; the partial pieces at a tile's first and
                               last columns are written by plain stores */
} gemm_bulk_store_t;

typedef struct {
  int32_t path;            /* gemm_path_t */
  int32_t swap_ab;         /* 1: the kernel computes C^T = op(B)^T * op(A)^T */
  int32_t a_kmajor;        /* MMA A operand (rows of the MMA) has K contiguous */
  int32_t b_kmajor;        /* MMA B operand (columns of the MMA) has K contiguous */
  int32_t bm, bn, bk;      /* output tile (bm x bn; a CTA pair shares bm = 256) and the k-block
                              of one stage: kdepth 128-byte k-slices (64 k for 16-bit
                              inputs, 128 for 8-bit, 32 for fp32/TF32) */
  int32_t stages;          /* shared-memory ring depth, in stages of bk */
  int32_t split_k;         /* k-splits per output tile (1 = none) */
  int32_t raster_group;    /* tile rows per raster group */
  int32_t repack_a;        /* A copied to an aligned workspace first (fp32: written as TF32 parts) */
  int32_t repack_b;        /* B copied to an aligned workspace first (fp32: written as TF32 parts) */
  int32_t vector_store;    /* epilogue writes C rows with 16-byte (or bulk tensor) stores */
  int32_t grid;            /* CTAs launched for the main kernel */
  int32_t launches;        /* kernels launched by one gemm_run */
  int32_t schedule;        /* 0: whole (or split-K) tiles; 1: stream-K tail */
  int64_t tiles;           /* schedule tiles = tiles_i * tiles_j * batch */
  int64_t units;           /* work units over all CTAs (tiles, split pieces or stream-K pieces) */
  int64_t workspace_bytes; /* handle workspace this call needs */
  int32_t tiles_i;         /* schedule tiles along the MMA rows (M, or N when swapped) */
  int32_t tiles_j;         /* schedule tiles along the MMA columns (N, or M when swapped) */
  int32_t num_kb;          /* k-blocks of bk per tile (GEMM_F32_F32: over 3K) */
  int32_t dp_tiles;        /* tiles run whole (stream-K: the complete waves) */
  int32_t sk_slots;        /* stream-K: clusters sharing the remaining tiles' k-blocks */
  int32_t cluster;         /* CTAs per schedule slot: 1, or 2 (a CTA pair) */
  int32_t kdepth;          /* 128-byte k-slices per ring stage (1 or 2): each stage's copies
                              complete one barrier */
  int32_t bulk_store;      /* how C leaves: gemm_bulk_store_t */
  int32_t batch;           /* GEMMs in the call (1 unless strided batched); tiles counts all */
  int32_t epilogue_warps;  /* warps storing C: 4 (one per 32-lane quarter of the accumulator), or
                              8 (two per quarter, each storing half of a tile's columns; for
                              256-wide CTA-pair 16-bit tiles whose C leaves through direct
                              stores, row classes or per-row copies) */
} gemm_plan_t;

/*
 * gemm_plan: the configuration gemm_run would use for these arguments, written
 * to *plan.  Host-only: touches no device, so it can be called without a GPU.
 * With h == NULL the default options and a GPU of `sm_count` SMs (all of them
 * usable by CTA pairs) are assumed; with a handle, its options
 * (gemm_set_option) and its device's measured residency apply and sm_count is
 * ignored.  Pointers are used only for their alignment.  Returns the same
 * argument errors as gemm_run.
 */
gemm_status_t gemm_plan(gemm_handle_t h, int sm_count, gemm_op_t transA, gemm_op_t transB,
                        int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                        const void* B, int64_t ldb, float beta, const void* C, int64_t ldc,
                        gemm_dtype_t dtype, gemm_plan_t* plan);

/*
 * gemm_run_grouped: `groups` GEMMs with stacked rows, the grouped GEMM of
 * mixture-of-experts layers (DeepGEMM's, which "第4章：经典算子实现 —— GEMM"
 * cites for MoE routing): tokens sorted by expert, expert g owning
 * m_sizes[g] consecutive rows (m_sizes: a host array; 0 is allowed):
 *   C[off_g + i, :] = alpha * A[off_g + i, :] * op(B_g) + beta * C[off_g + i, :],  i < m_sizes[g]
 * with off_g the sum of the sizes before g.  A is stored sum(m) x K row-major
 * (lda >= K); B_g = B + g * strideB (elements) is N x K when transB ==
 * GEMM_OP_T, else K x N; C is sum(m) x N (ldc).  strideB == 0 gives every group
 * the same B.  One launch covers every group: the groups' tiles share one
 * persistent schedule, a group's last tile rows are masked at its edge, and C
 * leaves through direct stores.  8-bit inputs need transB == GEMM_OP_T.
 * groups == 0 is a no-op.  The fused epilogue `epi` (may be NULL) applies as
 * in gemm_run_ex.  Errors as gemm_run_ex; GEMM_ERR_INVALID_ARG for a negative
 * size or a missing m_sizes.
 */
gemm_status_t gemm_run_grouped(gemm_handle_t h, gemm_op_t transB, int64_t groups, const int64_t* m_sizes,
                               int64_t N, int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                               int64_t ldb, int64_t strideB, float beta, void* C, int64_t ldc,
                               gemm_dtype_t dtype, const gemm_epilogue_t* epi, void* stream);

/* gemm_plan for a grouped call (arguments as gemm_run_grouped; tiles_i counts
   every group's tile rows). */
gemm_status_t gemm_plan_grouped(gemm_handle_t h, int sm_count, gemm_op_t transB, int64_t groups,
                                const int64_t* m_sizes, int64_t N, int64_t K, const void* A, int64_t lda,
                                const void* B, int64_t ldb, int64_t strideB, float beta, const void* C,
                                int64_t ldc, gemm_dtype_t dtype, gemm_plan_t* plan);

/*
 * gemm_run_block_scaled: C = alpha * A' * B'^T + beta * C for block-scaled
 * operands, as the Blackwell section of "CUDA GEMM 矩阵乘法优化指南" (13.2)
 * describes them: narrow codes sharing one scale factor per block of k:
 *   a'(i, k) = code(A, i, k) * scale(SFA[i * ld_sfa + k / block])
 *   b'(j, k) = code(B, j, k) * scale(SFB[j * ld_sfb + k / block])
 * MXFP8 (GEMM_MXFP8_*): E4M3 / E5M2 codes, block 32, E8M0 scales (2^(s - 127)).
 * NVFP4 (GEMM_NVFP4_*): E2M1 codes (sign, 2-bit exponent with bias 1, 1-bit
 *   fraction), two a byte with the even k in the low four bits; block 16;
 *   unsigned E4M3 scales (sign bit ignored).  A per-tensor scale folds into alpha.
 * A is stored M x K and B N x K, K contiguous; lda / ldb count values (even
 * for NVFP4).  SFA is M rows and SFB N rows of at least ceil(K / block) scale
 * codes, row pitches ld_sfa / ld_sfb in bytes.  Codes past K in a row and scale
 * codes past ceil(K / block) are never read.  C is M x N (ldc) in fp32, bf16
 * or fp16.  The fused epilogue `epi` (may be NULL) applies as in gemm_run_ex.
 * All pointers are device pointers owned by the caller.
 * How it runs: one launch per operand writes a'(., k) as bf16 into the handle's
 * workspace (exact: a code times a scale has at most 6 significant bits, so
 * every value inside bf16's exponent range is held exactly; values below
 * 2^-133 flush), then the bf16 tensor-core GEMM computes the product, so the
 * result is the block-scaled product with fp32 accumulation at bf16 speed.
 * With M <= 64 < N (a decode-batch GEMM against a weight matrix, bound by
 * reading B), B instead stays in its codes: only A goes through the pass, and
 * four more warps of the GEMM convert B's codes and scales into the tensor
 * core's operand tiles as they arrive (NVFP4 as fp16, exact; MXFP8 as bf16),
 * so B's bytes are read once, at their code size.  This needs B and SFB
 * 16-byte aligned with rows of a multiple of 16 bytes (ldb / 2 bytes for
 * NVFP4, ldb for MXFP8; ld_sfb); otherwise, or with the option
 * GEMM_OPT_DEQUANT_IN_KERNEL = 1, both operands take the pass.
 * (The tensor core's own block-scaled kinds are not used.)
 * Returns GEMM_ERR_INVALID_ARG for a non-block-scaled dtype, null scales,
 * scale pitches below ceil(K / block), odd NVFP4 pitches, or the argument
 * errors of gemm_run.
 */
gemm_status_t gemm_run_block_scaled(gemm_handle_t h, int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                                    int64_t lda, const void* SFA, int64_t ld_sfa, const void* B, int64_t ldb,
                                    const void* SFB, int64_t ld_sfb, float beta, void* C, int64_t ldc,
                                    gemm_dtype_t dtype, const gemm_epilogue_t* epi, void* stream);

/* gemm_plan for a block-scaled call (arguments as gemm_run_block_scaled). */
gemm_status_t gemm_plan_block_scaled(gemm_handle_t h, int sm_count, int64_t M, int64_t N, int64_t K, const void* A,
                                     int64_t lda, const void* SFA, int64_t ld_sfa, const void* B, int64_t ldb,
                                     const void* SFB, int64_t ld_sfb, float beta, const void* C, int64_t ldc,
                                     gemm_dtype_t dtype, gemm_plan_t* plan);

/*
 * gemm_run_host: gemm_run on HOST buffers.  A, B and C are host pointers
 * (page-locked memory lets the copies overlap the GEMM; pageable memory works
 * but serialises them); sizes, leading dimensions, dtypes and errors as
 * gemm_run (block-scaled types: GEMM_ERR_UNSUPPORTED).  The handle keeps device
 * copies of A, B and C (grown as needed: a larger call synchronises the device
 * once) and two copy streams, one per direction.  C is processed in blocks of
 * up to four row chunks by four column chunks (M or N of 1024 or more is cut
 * in four): A's row chunks and B's column chunks travel to the device
 * alternately, each block of C (its old values first when beta != 0) is
 * multiplied as soon as its rows of A and columns of B are there, and goes
 * back to the host while the next inputs travel.  Everything
 * is ordered after the work already queued on `stream`, and `stream` waits
 * for the last copy back: C on the host is complete once `stream` is
 * synchronised.  The host buffers must stay valid and unchanged until then.
 */
gemm_status_t gemm_run_host(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N, int64_t K,
                            float alpha, const void* A, int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                            int64_t ldc, gemm_dtype_t dtype, void* stream);

/* gemm_plan for a strided batched call (arguments as gemm_run_strided_batched). */
gemm_status_t gemm_plan_strided_batched(gemm_handle_t h, int sm_count, gemm_op_t transA, gemm_op_t transB,
                                        int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                        int64_t strideA, const void* B, int64_t ldb, int64_t strideB,
                                        float beta, const void* C, int64_t ldc, int64_t strideC,
                                        int64_t batch, gemm_dtype_t dtype, gemm_plan_t* plan);

typedef enum {
  GEMM_OPT_WAIT_LIMIT_NS = 0, /* barrier wait limit in ns (default 2e9; >= 1e6) */
  GEMM_OPT_FORCE_PATH = 1,    /* 0 auto, or GEMM_PATH_TC_1CTA / GEMM_PATH_TC_2CTA */
  GEMM_OPT_SPLIT_K = 2,       /* 0 auto, else the k-split to use (clamped to the k-blocks) */
  GEMM_OPT_RASTER_GROUP = 3,  /* 0 auto, else tile rows per raster group */
  GEMM_OPT_FORCE_BN = 4,      /* 0 auto, else 64, 128 or 256 */
  GEMM_OPT_TEST_DROP_LOAD = 5, /* tests only: 0 off; n > 0 makes CTA 0 skip its n-th k-block
                                  load, so a barrier is never completed and the bounded wait
                                  must end the kernel with GEMM_ERR_TIMEOUT */
  GEMM_OPT_MAX_GRID = 6,       /* 0 auto, else at most this many CTAs (persistent CTAs then
                                  walk more tiles each) */
  GEMM_OPT_STREAM_K = 7,       /* 0 auto, 1 never, 2 always when the last wave is incomplete */
  GEMM_OPT_STAGES = 8,         /* 0 auto (deepest ring that fits), else at most this many stages */
  GEMM_OPT_EPILOGUE = 10,      /* 0 auto: C tiles leave through shared-memory staging and bulk
                                  tensor stores when rows start 16-byte aligned and N is a whole
                                  number of 16-byte pieces (beta != 0: old C arrives by tensor
                                  loads); else, with beta == 0 and unswapped, through an aligned
                                  copy in the workspace and a second kernel (GEMM_BULK_STAGED;
                                  one GEMM, M * N >= 2^20, K < 2048) or by per-row bulk copies
                                  (GEMM_BULK_ROW_COPIES); 2: always direct stores from
                                  registers; 3: prefer GEMM_BULK_STAGED where allowed;
                                  4: prefer GEMM_BULK_ROW_COPIES.  In auto mode fp32 C of one
                                  GEMM takes GEMM_BULK_ROW_CLASSES before either */
  GEMM_OPT_KDEPTH = 11,        /* 0 auto, else 1 or 2 128-byte k-slices per ring stage (2 halves
                                  the barrier round trips per byte; falls back to 1 where the
                                  ring would hold fewer than two stages) */
  GEMM_OPT_PDL = 12,           /* 1 (default): the main kernel is launched as a programmatic
                                  dependent of the stream's previous kernel, so its launch and
                                  set-up overlap that kernel's end; it reads and writes memory only
                                  after the previous kernel has finished.  0: ordinary launch */
  GEMM_OPT_PLAN_CACHE = 13,    /* 1 (default): plain and strided-batched calls reuse the plan of
                                  an earlier call with the same sizes, leading dimensions,
                                  strides, dtype, beta, options and pointer alignments (32
                                  plans per handle, least recently used replaced); 0: plan
                                  every call */
  GEMM_OPT_DEQUANT_IN_KERNEL = 15, /* block-scaled GEMMs with M <= 64 < N: 0 (default) the weights
                                  B stay in their codes and the GEMM converts them as they
                                  arrive (see gemm_run_block_scaled); 1: a pass writes both
                                  operands as 16-bit values first */
  GEMM_OPT_EPILOGUE_WARPS = 16  /* 0 auto (eight where C leaves through direct stores, row
                                  classes or per-row copies and the tile has such a kernel),
                                  else 4 or 8: the kernel with that many epilogue warps where
                                  the tile has one (gemm_plan_t.epilogue_warps) */
} gemm_option_t;

/* Set an option on a handle.  Errors: GEMM_ERR_INVALID_ARG for an unknown
   option or an out-of-range value. */
gemm_status_t gemm_set_option(gemm_handle_t h, gemm_option_t opt, int64_t value);

/* Kernels launched by gemm_run on this handle since it was created. */
gemm_status_t gemm_launch_count(gemm_handle_t h, uint64_t* count);

/* Plan-cache counters of the handle since its creation: calls whose plan was
   reused (*hits) and calls that planned anew (*misses). */
gemm_status_t gemm_plan_cache_stats(gemm_handle_t h, uint64_t* hits, uint64_t* misses);

/* Tensor-map cache counters of the handle since its creation.  Each launch
   needs two or three tensor maps (A, B and, for bulk stores, C); a map whose
   description (base address, extents, strides, box, type, swizzle) matches
   one encoded by a recent call is copied from the handle's cache (*hits)
   instead of being encoded again (*misses).  256 maps are kept (64 sets of 4,
   least recently used replaced). */
gemm_status_t gemm_tensor_map_cache_stats(gemm_handle_t h, uint64_t* hits, uint64_t* misses);

/*
 * gemm_probe_tma_tile (test support): load one tile of a row-major 16-bit
 * matrix into shared memory exactly as the GEMM loads a K-major operand tile
 * (a tensor-memory-accelerator copy with the 128-byte swizzle; box of 64
 * elements = 128 bytes by `rows` rows, starting at element (0, 0)), then copy
 * the tile's shared-memory bytes unchanged to `dst`: rows * 64 16-bit values
 * in shared-memory order, so that dst[p] is the element the copy engine put at
 * 16-bit position p.  Elements past `cols` arrive as zeros.  The layout the
 * MMA descriptors assume is element (r, c) at r * 64 + (c ^ ((r & 7) << 3))
 * ("[CUDA 优化实战] hgemm sm120 - 100KB SMEM 中的“微雕”战争", section 4).
 *   src: device pointer, 16-byte aligned; ld (elements, >= cols) with ld * 2 a
 *        multiple of 16; 1 <= rows <= 256; cols >= 1.
 *   dst: device pointer to rows * 64 uint16 values (caller-owned).
 * Asynchronous on `stream`.  GEMM_ERR_INVALID_ARG for a bad argument (checked
 * before any CUDA call), GEMM_ERR_TENSORMAP if the tile cannot be described,
 * GEMM_ERR_CUDA on a launch failure; a copy that never lands is reported by
 * gemm_get_status as GEMM_ERR_TIMEOUT.  After that report the caller launches
 * no further probe in the process: the timed-out copy may still land in the
 * shared memory of an exited block.
 */
gemm_status_t gemm_probe_tma_tile(gemm_handle_t h, const void* src, int64_t ld, int64_t cols, int64_t rows, void* dst,
                                  void* stream);

/* ---------------------------------------------------------------------------
 * gemm_run_noalloc: the GEMM of gemm_run for callers that must not allocate
 * device memory -- for example a caller whose device memory is fully reserved
 * up front by its own allocator, or one that cannot afford the device-wide
 * synchronisation that cudaMalloc / cudaFree can imply.  (The source pages
 * have no counterpart; this is a property of the library's interface.)
 *
 * Same arguments and semantics as gemm_run, on the current CUDA device and
 * without a handle; default options apply.  It calls no cudaMalloc, cudaFree
 * or other allocating routine.  Its scratch -- repacked copies of operands the
 * copy engine cannot read directly, partial sums of tiles split by the
 * stream-K schedule, their arrival counters and a status word -- lives in
 * fixed file-scope device arrays of the library: 16 MiB of scratch and 4096
 * counters, which every GPU that loads the library holds until the process
 * exits.  A call whose plan would need more (a larger repack, or more partial
 * sums than fit) is first re-planned without the stream-K tail, which needs
 * no partial sums; if it still does not fit, the call returns
 * GEMM_ERR_WORKSPACE and launches nothing.
 *
 * The first call on a device sets that device up (looks up the arrays'
 * device addresses, opts the kernels in to their shared memory); later calls
 * only plan and launch.  Every call shares the same arrays
 * and each call clears the counters and status word it uses, so calls that
 * overlap on the GPU (two streams, or two host threads) race on them: order
 * them on one stream.  A kernel that gives up on a barrier records it in the
 * path's own status word; gemm_noalloc_get_status reads it.
 * Returns GEMM_OK, the argument errors of gemm_run, GEMM_ERR_NO_DEVICE,
 * GEMM_ERR_WORKSPACE or GEMM_ERR_CUDA.
 * ------------------------------------------------------------------------- */
gemm_status_t gemm_run_noalloc(gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N, int64_t K,
                               float alpha, const void* A, int64_t lda, const void* B, int64_t ldb,
                               float beta, void* C, int64_t ldc, gemm_dtype_t dtype, void* stream);

/*
 * gemm_noalloc_get_status: the status of the no-allocation path on the
 * current device, like gemm_get_status for a handle.  Synchronises `stream`,
 * reads the path's device status word and clears it.  Returns GEMM_OK,
 * GEMM_ERR_TIMEOUT (a kernel of an earlier gemm_run_noalloc gave up waiting on
 * a barrier and returned early; its C is incomplete) or GEMM_ERR_CUDA;
 * *detail (may be NULL) receives the raw word (layout as gemm_get_status).
 * Allocates nothing.  The word is shared by every no-allocation call on the
 * device, so read it after the calls it should cover, on their stream.
 */
gemm_status_t gemm_noalloc_get_status(void* stream, int32_t* detail);

/*
 * gemm_noalloc_set_option: process-wide options of the no-allocation path.
 * Only GEMM_OPT_WAIT_LIMIT_NS (>= 1e6) and GEMM_OPT_TEST_DROP_LOAD (tests:
 * make CTA 0 skip its n-th k-block load, 0 off) are accepted; any other option
 * returns GEMM_ERR_INVALID_ARG.  Takes effect from the next gemm_run_noalloc.
 */
gemm_status_t gemm_noalloc_set_option(gemm_option_t opt, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
