// gemm_internal.h -- declarations shared by the host planner (gemm_api.cu) and
// the kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "schedule.h"

namespace g10 {

constexpr int kBM = 128;          // MMA M (rows of the output tile held in TMEM lanes)
constexpr int kSliceBytes = 128;  // a k-slice: one 128-byte swizzle row of every tile row
constexpr int kBK = 64;           // k-slice of 16-bit elements (64 x 2 bytes)
// Warps of a GEMM CTA: warp 0 TMA producer, warp 1 MMA issuer, then `ew`
// epilogue warps (four, one per 32-lane quarter of tensor memory; or eight,
// two per quarter, each of a pair storing half of the tile's columns), then in
// DQ kernels kConvWarps warps converting block-scaled codes.
constexpr int kConvWarps = 8;
__host__ __device__ constexpr int threads_of(int ew, bool dq) { return 64 + 32 * (ew + (dq ? kConvWarps : 0)); }

// k elements of one k-slice for an element of eb bytes (2: bf16 / fp16, 1: FP8).
__host__ __device__ constexpr int slice_k(int eb) { return kSliceBytes / eb; }

// Element type of C.
enum CType : int32_t { kCF32 = 0, kCBF16 = 1, kCF16 = 2, kCE4M3 = 3 };

// Elementwise operations fused into the store of C (after the alpha / beta
// blend): z += bias, z = act(z), z *= out_scale, then the conversion to C's type.
enum Activation : int32_t { kActNone = 0, kActRelu = 1, kActGelu = 2 };
struct EpiOps {
  const float* bias = nullptr;  // one fp32 value per column of the caller's C, or null
  int32_t bias_on_i = 0;        // the bias runs along the kernel's I (a swapped problem)
  int32_t act = kActNone;
  float out_scale = 1.0f;
  __host__ __device__ bool any() const { return bias != nullptr || act != kActNone || out_scale != 1.0f; }
};

// Status-word layout written by a kernel that gives up on a barrier:
//   bits 0-7 = 6 (GEMM_ERR_TIMEOUT), bits 8-11 = role, bits 12-15 = barrier.
enum : int32_t { kStatusTimeout = 6 };
enum WaitRole : int32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleConvert = 4 };
enum WaitBarrier : int32_t {
  kBarEmpty = 1, kBarFull = 2, kBarAccEmpty = 3, kBarAccFull = 4, kBarDrain = 5, kBarCLoad = 6, kBarCodeFull = 7
};

// Arguments of the persistent tcgen05 GEMM kernel, in the kernel's own terms:
//   D (I x J) = P (I x K) * Q (K x J),  C[i * c_si + j * c_sj] = alpha * D[i][j] + beta * C[...]
// P is the MMA "A" operand (tile rows on TMEM lanes), Q the MMA "B" operand.
struct TcArgs {
  int32_t I, J, K;
  Sched sched;           // work assignment (schedule.h); num_kb = ceil(K / (slice_k * kdepth))
  int32_t p_kmajor;      // P has K contiguous (else I contiguous)
  int32_t q_kmajor;      // Q has K contiguous (else J contiguous)
  uint32_t idesc;        // tcgen05 instruction descriptor
  int32_t stages;        // ring stages in use, 1 .. the configuration's maximum / kdepth
  int32_t kdepth;        // k-slices per stage (1 or 2); one barrier per stage
  float alpha, beta;
  void* C;
  int64_t c_si, c_sj;
  int32_t c_type;        // CType
  int32_t vec_store;     // c_sj == 1 and every row of C starts 16-byte aligned
  int32_t tma_store;     // BulkStore: how C tiles leave through shared-memory staging
  float* partials;       // partial tiles of split tiles, [partial_slots * CG][BN][kBM] fp32
  int32_t* counters;     // per split tile (x CG) arrival counters, zero between calls
  int32_t* status;       // device status word
  uint64_t wait_limit_ns;
  int32_t drop_load;     // tests only: CTA 0 skips its drop_load-th k-block load (1-based)
  int32_t pdl;           // launch as a programmatic dependent of the stream's previous kernel
  // TF32 operands stored as two segments of seg_slices 128-byte k-slices
  // (0: no segments): logical segment s of K reads stored segment bit s of
  // p_seg (P) / q_seg (Q)
  int32_t seg_slices;
  int32_t p_seg, q_seg;
  EpiOps ops;            // fused elementwise operations of the epilogue
  int64_t c_sb;          // batch stride of C in elements (strided batches; tile batch in Unit::tb)
  int32_t p_bcast;       // P is one matrix shared by every batch (its tensor map has one batch)
  int32_t q_bcast;
  // grouped GEMMs (sched.groups > 0): group g's rows of P and C start at row
  // group_row[g] and number group_m[g]; the tile's group is Unit::tb
  const int64_t* group_row;
  const int32_t* group_m;
  int32_t c_classes;     // kBulkRowCopies with fp32 C: P row classes with tensor maps in CMaps (0: per-row copies)
  // DQ kernels: P arrives as block-scaled codes (map_p: the codes, CMaps m[0]:
  // their scale codes) and converter warps write its 16-bit values into the
  // ring.  dq_fmt: 1 E2M1 codes with unsigned E4M3 scales per 16 values (to
  // fp16), 2 / 3 E4M3 / E5M2 codes with E8M0 scales per 32 values (to bf16).
  int32_t dq_fmt;
  int32_t code_bytes;    // code bytes of one row of a k-slice (32 for E2M1, 64 for the 8-bit codes)
  int32_t spk;           // scale codes of one row of a k-slice (4 or 2)
  int32_t code_stages;       // stages of the code ring (<= 16)
  int32_t code_stage_bytes;  // Q's tile, 128 rows of codes, 128 x 16 bytes of scale codes (a multiple of 1024)
};

// Epilogue store paths: direct stores, or staged bulk tensor stores of rows of
// C, or (for swapped problems, whose C is stored J x I) of transposed blocks,
// or, for rows of C that bulk tensor stores cannot write (not 16-byte aligned,
// or ending inside a 16-byte piece), one 1-D bulk copy per row of a block.
enum BulkStore : int32_t { kBulkNone = 0, kBulkRows = 1, kBulkTransposed = 2, kBulkRowCopies = 3 };

// Tensor maps of fp32 C whose rows start off 16-byte boundaries (c_classes
// P > 0 in TcArgs): the rows i = r, r + P, r + 2P, ... (class r) all start the
// same s_r values past a 16-byte boundary and lie P * ldc * 4 bytes apart, a
// multiple of 16, so each class is a tensor of its own whose columns are C's
// shifted by s_r.  m[r]: class r, boxes of 32 columns by 32 / P rows, 128-byte
// swizzle; m[4 + r]: the same class, boxes of 28 columns (unswizzled 112-byte
// rows) for a tile's first block, whose first 16-byte piece holds values of
// the tile to its left.
struct CMaps {
  CUtensorMap m[8];
};

// Tile configurations: a tile of (128 * cg) x bn per CTA (cg == 1) or CTA
// pair (cg == 2).  eb is the input element size in bytes: 2 for bf16 / fp16
// (tcgen05.mma kind::f16), 1 for the 8-bit formats (kind::f8f6f4), 4 for TF32
// (kind::tf32).
struct TileConfig {
  int bn, cg, eb;
  int dq;  // 1: P arrives as block-scaled codes, converted in the kernel (four more warps)
  int ew;  // epilogue warps: 4, or 8 (two per tensor-memory lane quarter)
};
constexpr int kNumTileConfigs = 15;
extern const TileConfig kTileConfigs[kNumTileConfigs];
int tc_stages(int cfg);  // ring depth in k-slices
int tc_code_ring_bytes(int cfg);  // DQ kernels: shared memory of the code ring (0 for the others)
// One-time per device: opt in to the kernel's shared memory; for clusters also
// report how many can be resident at once.
cudaError_t tc_prepare(int cfg, int* max_clusters);
// grid = CTAs (a multiple of cg).
// map_c describes C for the bulk-store epilogue (ignored unless args.tma_store).
cudaError_t tc_launch(int cfg, const CUtensorMap& map_p, const CUtensorMap& map_q,
                      const CUtensorMap& map_c, const CMaps& cmaps, const TcArgs& args, int grid,
                      cudaStream_t stream);

// dst[b * dbs + r * ldd + c] = src[b * sbs + r * lds + c] for elements of
// esize (1 or 2) bytes, b < nb, r < rows, c < cols; strides in elements.
cudaError_t repack_launch(const void* src, int64_t lds, int64_t sbs, void* dst, int64_t ldd, int64_t dbs,
                          int64_t rows, int64_t cols, int64_t nb, int esize, int sm_count,
                          cudaStream_t stream);

// One 128-byte-swizzled tile load (box 64 x rows of 16-bit elements) into
// shared memory, written back out in shared-memory order (probe.cu).
cudaError_t tma_tile_probe_launch(const CUtensorMap& map, int rows, uint16_t* dst, int32_t* status,
                                  uint64_t wait_limit_ns, cudaStream_t stream);

// dst[r * ldd + c] = src[r * lds + c] for r < rows, c < cols, elements of
// esize (2 or 4) bytes; src 16-byte aligned with 16-byte rows (lds * esize a
// multiple of 16) that hold whole 16-byte pieces past cols.  Nothing outside
// dst's rows x cols elements is written.
cudaError_t unstage_c_launch(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                             int esize, cudaStream_t stream);

// TF32 values of fp32 operands, written K-major: row r of dst (b-th matrix at
// dbs elements) receives parts segments of seg values (seg >= K; values K ..
// seg - 1 of a segment are 0).  parts == 1: each value with its 13 low fraction
// bits dropped.  parts > 1: segment s holds lo = TF32(x - hi) when bit s of
// pattern is set, else hi = TF32(x) (both rounded to nearest).  Source element
// (r, k) is src[k * lds + r] when transposed, else src[r * lds + k].
cudaError_t split_tf32_launch(const float* src, int64_t lds, int64_t sbs, bool transposed, float* dst,
                              int64_t ldd, int64_t dbs, int64_t rows, int64_t K, int64_t seg, int64_t nb, int parts,
                              int pattern, int sm_count, cudaStream_t stream);

// Block-scaled operand -> bf16 (fp16 when f16_out), K-major: dst[r * ldd + k] = code(r, k) *
// scale(r, k / block) for k < K, 0 for K <= k < ldd (ldd a multiple of 16, dst
// 16-byte aligned).  fmt: 0 E4M3, 1 E5M2, 2 E2M1 packed two a byte (even k
// low); lds counts values; scale codes E8M0 (e8m0) or unsigned E4M3, rows of
// ld_sf codes.  block: 16 or 32.
cudaError_t dequant_launch(const void* src, int64_t lds, const void* sf, int64_t ld_sf, int fmt, bool e8m0,
                           int block, void* dst, int64_t ldd, int64_t rows, int64_t K, bool f16_out, int sm_count,
                           cudaStream_t stream);

// The whole GEMM when K == 0: C = ops(beta * C) over `batch` M x N matrices
// with leading dimension ldc, sbc elements apart (beta * C = 0 when beta == 0;
// C is then not read).
cudaError_t scale_c_launch(void* C, int32_t c_type, int64_t M, int64_t N, int64_t ldc, float beta,
                           const EpiOps& ops, int64_t batch, int64_t sbc, int sm_count,
                           cudaStream_t stream);

}  // namespace g10
