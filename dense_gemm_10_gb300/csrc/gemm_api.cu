// gemm_api.cu -- the C ABI of include/gemm_gb300.h: handles, argument checks,
// the planner, tensor-map encoding and kernel launches.
//
// The planner restates, for this GPU, the blocking choices of the pages:
// output tiles computed by one CTA ("CUDA GEMM 矩阵乘法优化指南", 5.1 and 13.2),
// a persistent grid of one CTA per SM (12.5), a k-split when there are too few
// tiles to fill the SMs ("GPU GEMM 优化完全拆解（三）", Split-K 与 Sliced-K), and
// the transpose identity C^T = B^T A^T that cuBLAS callers use to swap operand
// roles ("第4章：经典算子实现 —— GEMM", 7.1), here to put a short M on the MMA's
// N dimension.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gemm_gb300.h"
#include "gemm_internal.h"
#include "ptx.cuh"
#include "tmap_cache.h"

using namespace g10;

namespace {

constexpr int64_t kMaxExtent = (int64_t{1} << 31) - 4096;  // kernel indexes with int32
constexpr int64_t kCounterCap = 1 << 16;                    // split-K tiles per call
constexpr int64_t kDefaultWaitNs = 2000000000;              // 2 s

struct Options {
  int64_t wait_limit_ns = kDefaultWaitNs;
  int force_path = 0;
  int split_k = 0;
  int raster_group = 0;
  int force_bn = 0;
  int drop_load = 0;
  int max_grid = 0;
  int stream_k = 0;  // 0 auto, 1 off, 2 on
  int stages = 0;    // 0: the configuration's maximum ring depth
  int tma_store = 0; // GEMM_OPT_EPILOGUE: 0 auto, 1 bulk stores when possible, 2 direct stores
  int kdepth = 0;    // GEMM_OPT_KDEPTH: 0 auto, else 64-wide k-slices per ring stage
  int pdl = 1;       // GEMM_OPT_PDL: programmatic dependent launch of the main kernel
  int plan_cache = 1;  // GEMM_OPT_PLAN_CACHE: reuse the plans of recent calls
  bool stage_c = true; // C that bulk stores cannot write may go through an aligned copy
  int dq_kernel = 0;   // GEMM_OPT_DEQUANT_IN_KERNEL: 0 auto, 1 never (the dequantising pass for both operands)
  int epi_warps = 0;   // GEMM_OPT_EPILOGUE_WARPS: 0 auto, else 4 or 8 where the tile has both kernels
};

// One stored operand, as the tensor-memory-accelerator copy engine will see it.
struct Operand {
  const void* ptr = nullptr;  // stored matrix (row-major)
  int64_t rows = 0, cols = 0; // stored shape
  int64_t ld = 0;             // leading dimension in elements
  bool kmajor = false;        // K runs along stored rows (cols == K)
  bool repack = false;        // copied into the workspace first
  int64_t packed_ld = 0;
  size_t ws_offset = 0;
  int64_t bstride = 0;        // elements between batches' matrices (strided batches)
  int64_t nb = 1;             // distinct matrices: 1 when shared by every batch
  // fp32 operands written as TF32 parts (split_tf32_launch) instead of repacked:
  // the source is ptr/ld/bstride, `src_k` values of k per row, read transposed
  // when `split_trans`; the copy is rows x cols (= split_parts segments of
  // split_seg values) K-major.  seg_map: bit s = the stored segment that
  // logical segment s of the GEMM's k reads (three-product fp32 GEMM).
  int split_parts = 0;
  int split_pattern = 0;
  bool split_trans = false;
  int64_t src_k = 0;
  int64_t split_seg = 0;
  int seg_map = 0;
  // block-scaled operands written as bf16 (dequant_launch) instead: source
  // codes of format dq - 1 at ptr (ld values a row), scale codes sf (ld_sf a row)
  int dq = 0;
  const void* sf = nullptr;
  int64_t ld_sf = 0;
  // block-scaled codes read by a DQ kernel as they are (converted in the kernel)
  bool codes = false;
  bool dq_f16 = false;  // dequant_launch writes fp16 (NVFP4 operands of a DQ kernel) instead of bf16
};

struct Plan {
  gemm_plan_t pub{};
  int32_t tma_store = kBulkNone;  // BulkStore: how C leaves the epilogue
  Sched sched{};
  Operand p, q;
  int64_t I = 0, J = 0, K = 0;
  int64_t c_si = 0, c_sj = 0;
  int64_t batch = 1, c_sb = 0;  // strided batch: count, C's batch stride in elements
  // grouped GEMMs: per-group tile prefix, first row and row count (host copies)
  std::vector<int32_t> group_tiles, group_m;
  std::vector<int64_t> group_row;
  size_t group_offset = 0;      // their place in the workspace
  int32_t c_type = kCF32;
  int32_t eb = 2;                  // input element bytes (2: bf16 / fp16, 1: FP8)
  uint32_t a_fmt = 1, b_fmt = 1;   // instruction-descriptor formats of the stored A and B
  int32_t in_dtype = 0;            // CU_TENSOR_MAP data type of A and B
  int cfg = 0;                     // index into kTileConfigs
  size_t partial_offset = 0;
  // C staged in the workspace (bulk_store == GEMM_BULK_STAGED): the kernel's
  // bulk stores write an aligned copy, rows of c_ws_ld elements, which a copy
  // kernel then writes into C
  bool c_staged = false;
  int64_t c_ws_ld = 0;
  size_t c_ws_offset = 0;
  // fp32 C off 16-byte boundaries written by tensor stores per row class (CMaps)
  int32_t c_classes = 0;
  // a DQ kernel: P's block-scaled codes converted in the kernel
  int32_t dq_fmt = 0, code_bytes = 0, spk = 0;
  int64_t code_cols = 0, scale_cols = 0;  // bytes of codes and scale codes in a row of P
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool tma_aligned(const void* p, int64_t ld, int eb, int64_t bstride, int64_t nb) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * eb) % 16 == 0) &&
         (nb == 1 || (bstride * eb) % 16 == 0);
}

// The input and output types a gemm_dtype_t names.
struct DtypeInfo {
  bool valid = false;
  int32_t eb = 2;
  uint32_t a_fmt = 0, b_fmt = 0;  // kind::f16: 0 f16, 1 bf16; kind::f8f6f4: 0 E4M3, 1 E5M2
  int32_t c_type = kCF32;
  CUtensorMapDataType map_type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int parts = 0;  // fp32 inputs: TF32 products per product (1 or 3)
  // block-scaled inputs (gemm_run_block_scaled): 1 MXFP8 (E8M0 scales), 2 NVFP4
  // (unsigned E4M3 scales); values of k per scale; code formats of A and B
  // (0 E4M3, 1 E5M2, 2 E2M1).  The GEMM itself then runs on bf16 values.
  int sc = 0;
  int block = 0;
  int src_a = 0, src_b = 0;
};

// Scale codes of a block-scaled GEMM (rows of ld codes, one per block of k).
struct BlockScale {
  const void* sfa = nullptr;
  int64_t ld_sfa = 0;
  const void* sfb = nullptr;
  int64_t ld_sfb = 0;
};

DtypeInfo dtype_info(int dtype) {
  DtypeInfo d;
  if (dtype >= GEMM_BF16_F32 && dtype <= GEMM_F16_E4M3) {
    const bool bf16 = dtype == GEMM_BF16_F32 || dtype == GEMM_BF16_BF16 || dtype == GEMM_BF16_E4M3;
    d.valid = true;
    d.a_fmt = d.b_fmt = bf16 ? 1u : 0u;
    d.c_type = (dtype == GEMM_BF16_F32 || dtype == GEMM_F16_F32)    ? kCF32
               : (dtype == GEMM_BF16_E4M3 || dtype == GEMM_F16_E4M3) ? kCE4M3
               : bf16                                              ? kCBF16
                                                                   : kCF16;
    d.map_type = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  } else if ((dtype >= GEMM_MXFP8_F32 && dtype <= GEMM_MXFP8_E5M2_F16) ||
             (dtype >= GEMM_NVFP4_F32 && dtype <= GEMM_NVFP4_F16)) {
    // MXFP8: 32 + (A is E5M2) + 2 * (B is E5M2) + 4 * (C: 0 fp32, 1 bf16, 2 fp16); NVFP4: 48 + C
    static const int32_t kC[3] = {kCF32, kCBF16, kCF16};
    const bool mx = dtype <= GEMM_MXFP8_E5M2_F16;
    const int x = mx ? dtype - GEMM_MXFP8_F32 : dtype - GEMM_NVFP4_F32;
    d.valid = true;
    d.a_fmt = d.b_fmt = 1;  // the GEMM's operands: bf16
    d.c_type = kC[mx ? x >> 2 : x];
    d.map_type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    d.sc = mx ? 1 : 2;
    d.block = mx ? 32 : 16;
    d.src_a = mx ? (x & 1) : 2;
    d.src_b = mx ? ((x >> 1) & 1) : 2;
  } else if (dtype == GEMM_F32_F32 || dtype == GEMM_TF32_F32) {
    d.valid = true;
    d.eb = 4;
    d.a_fmt = d.b_fmt = 2;  // kind::tf32
    d.c_type = kCF32;
    d.map_type = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    d.parts = dtype == GEMM_F32_F32 ? 3 : 1;
  } else if (dtype >= GEMM_E4M3_F32 && dtype <= GEMM_E5M2_E4M3OUT) {
    // 16 + (A is E5M2) + 2 * (B is E5M2) + 4 * (C: 0 fp32, 1 bf16, 2 fp16, 3 E4M3)
    const int x = dtype - GEMM_E4M3_F32;
    static const int32_t kC[4] = {kCF32, kCBF16, kCF16, kCE4M3};
    d.valid = true;
    d.eb = 1;
    d.a_fmt = x & 1;
    d.b_fmt = (x >> 1) & 1;
    d.c_type = kC[x >> 2];
    d.map_type = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  }
  return d;
}

// 64-wide k-slices per ring stage unless GEMM_OPT_KDEPTH says otherwise.  The
// 64-wide tiles have small stages (20-24 KB per k-slice); two slices per stage
// halve the barrier round trips per byte, which measured 5-8% faster on the
// HBM-bound 64 x 32000 x 4096 GEMM.  The wider tiles measured no gain.
int default_kdepth(const TileConfig& c) { return c.bn == 64 ? 2 : 1; }

// Relative time of one 64-wide k-slice of one schedule tile for each tile
// configuration, in units of the CTA-pair 256 x 256 tile, from GB300
// measurements of the 4096^3 and 8192 x 12288 x 4096 bf16 GEMMs.
double tile_kb_cost(const TileConfig& c) {
  if (c.cg == 2) return c.bn == 256 ? 1.0 : c.bn == 128 ? 0.62 : 0.65;
  return c.bn == 256 ? 1.15 : c.bn == 128 ? 0.85 : 0.6;
}

// Resident schedule slots (CTAs, CTA pairs or clusters) per tile configuration.
struct SlotTable {
  int n[kNumTileConfigs];
  SlotTable() {
    for (int& x : n) x = 1;
  }
  int of(int cfg) const { return n[cfg]; }
  static SlotTable even(int sm_count) {
    SlotTable t;
    for (int i = 0; i < kNumTileConfigs; ++i)
      t.n[i] = std::max(1, sm_count / kTileConfigs[i].cg);
    return t;
  }
};

// Opt every configuration in to its shared memory on the current device and
// record how many of its clusters can be resident (a cluster sits in one GPC).
cudaError_t measure_slots(int sm_count, SlotTable* t) {
  *t = SlotTable::even(sm_count);
  for (int i = 0; i < kNumTileConfigs; ++i) {
    const TileConfig& c = kTileConfigs[i];
    int clusters = 0;
    cudaError_t e = tc_prepare(i, &clusters);
    if (e != cudaSuccess) return e;
    if (c.cg > 1 && clusters > 0) t->n[i] = std::min(clusters, sm_count / c.cg);
  }
  return cudaSuccess;
}

struct Choice {
  bool valid = false;
  int cfg = 0, cg = 1, bn = 64, slots = 1, kdepth = 1;
  double cost = 1e300;
  Sched sched{};
};

bool needs_partials(const Sched& s) {
  return (s.mode == kSchedTiles && s.split_k > 1) || s.mode == kSchedStreamK;
}

// Work units over all slots (for reporting): whole tiles, split pieces, or
// stream-K range pieces (one more piece per slot edge that falls inside a tile).
int64_t count_units(const Sched& s) {
  const int64_t tiles = sched_tiles(s);
  if (s.mode == kSchedTiles) return tiles * s.split_k;
  int64_t n = s.dp_tiles + (tiles - s.dp_tiles);
  for (int32_t c = 1; c < s.sk_slots; ++c)
    if (sk_begin(s, c) % s.num_kb != 0) ++n;
  return n;
}

// Estimated time, in k-blocks of one tile, of the stream-K tail: `iters`
// k-blocks of `tiles` tiles dealt to `g` slots.  Each partial piece costs a
// store, and the tile's last contribution reads every piece of its tile.
// Time of a stream-K tail in k-blocks (one k-block = one ring stage of operand
// bytes per CTA).  Besides its share of the k-blocks, the slot that finishes a
// tile writes its fp32 partial and then reads every contribution back, and
// those bytes travel the same per-SM path as its operand loads: r k-blocks for
// the write and, measured on GB300 (4096^3 bf16 and 8-bit), ~1.5 r per
// contribution read.  r = a CTA's fp32 partial tile in stages of operand bytes.
double sk_tail_cost(int64_t tiles, int64_t num_kb, int64_t g, double r) {
  const int64_t iters = tiles * num_kb;
  const double per_slot = static_cast<double>(cdiv(iters, g));
  if (g <= tiles && tiles % g == 0) return per_slot;  // whole tiles, no partials
  const double contrib = per_slot >= static_cast<double>(num_kb)
                             ? 2.0
                             : std::ceil(static_cast<double>(num_kb) / per_slot) + 1.0;
  return per_slot + r * (1.0 + 1.5 * contrib);
}

// num_kb counts stages of kdepth 64-wide k-slices each.
Choice choose_schedule(const Options& o, int64_t tiles_i, int64_t tiles_j, int64_t batch, int64_t num_kb,
                       int kdepth, int cfg, int slots, bool hbm_bound) {
  Choice ch;
  ch.kdepth = kdepth;
  const TileConfig& tc = kTileConfigs[cfg];
  const int cl = tc.cg;  // CTAs per slot
  ch.cfg = cfg;
  ch.cg = tc.cg;
  ch.bn = tc.bn;
  ch.slots = slots;
  const int64_t tiles = tiles_i * tiles_j * batch;
  // a CTA's fp32 partial tile (bn x 128) in stages of its operand bytes
  const double stage_bytes = static_cast<double>(kdepth) * (kBM + tc.bn / tc.cg) * kSliceBytes;
  const double r = 4.0 * tc.bn * kBM / stage_bytes;
  Sched& s = ch.sched;
  s.tiles_i = static_cast<int32_t>(tiles_i);
  s.tiles_j = static_cast<int32_t>(tiles_j);
  s.batch = static_cast<int32_t>(batch);
  s.num_kb = static_cast<int32_t>(num_kb);
  s.raster_group = 8;
  s.mode = kSchedTiles;
  s.split_k = 1;
  if (o.split_k) {  // an explicit split-K request
    const int64_t split = std::min<int64_t>(o.split_k, num_kb);
    if (tiles * cl > kCounterCap) return ch;
    s.split_k = static_cast<int32_t>(split);
    ch.cost = static_cast<double>(cdiv(tiles * split, slots)) *
              (static_cast<double>(cdiv(num_kb, split)) + (split > 1 ? r * (1.0 + 1.5) : 0.0)) * kdepth *
              tile_kb_cost(tc);
    ch.valid = true;
    return ch;
  }
  // Whole tiles: ceil(tiles / slots) waves, on a grid that gives every slot the
  // same number of tiles (for an HBM-bound GEMM the slots of a last, partly
  // filled wave only compete for bandwidth).
  const int64_t waves = cdiv(tiles, slots);
  double best = static_cast<double>(waves * num_kb);
  ch.slots = static_cast<int>(cdiv(tiles, waves));
  // Stream-K tail: the tiles of the incomplete last wave shared by g slots.
  const int64_t full_waves = tiles / slots;
  const int64_t sk_tiles = tiles - full_waves * slots;
  // An HBM-bound GEMM whose whole tiles keep (nearly) every slot streaming
  // gains nothing from evening out the waves but the partial-sum traffic; one
  // that leaves a tenth of the slots idle gains their share of the bandwidth
  // (64 x 32000 x 4096: 250 tiles on 125 of 152 SMs, 49.0 us; stream-K on all
  // of them, 47.4 us).
  const bool hbm_busy = hbm_bound && tiles >= slots && 10 * ch.slots >= 9 * slots;
  const bool sk_allowed = o.stream_k == 2 || (o.stream_k == 0 && !hbm_busy);
  if (sk_allowed && sk_tiles > 0 && sk_tiles * cl <= kCounterCap) {
    const int64_t iters = sk_tiles * num_kb;
    int64_t best_g = 0;
    double best_tail = 1e300;
    for (int64_t g = 1; g <= std::min<int64_t>(slots, iters); ++g) {
      // After full waves, a tail whose share per slot exceeds half a tile is
      // mostly whole-tile work already; its partial sums and the tail tiles'
      // out-of-raster operand reads cost more than the quantisation saves
      // (measured at 8192 x 4096 x 16384).  An HBM-bound GEMM gains the idle
      // slots' bandwidth instead.
      if (o.stream_k != 2 && !hbm_bound && full_waves > 0 && 2 * cdiv(iters, g) > num_kb) continue;
      const double t = sk_tail_cost(sk_tiles, num_kb, g, r);
      if (t < best_tail - 1e-9) {
        best_tail = t;
        best_g = g;
      }
    }
    const double sk = static_cast<double>(full_waves * num_kb) + best_tail;
    if (best_g > 0 && (o.stream_k == 2 || sk < best - 1e-9)) {
      best = sk;
      ch.slots = slots;
      s.mode = kSchedStreamK;
      s.dp_tiles = static_cast<int32_t>(full_waves * slots);
      s.sk_slots = static_cast<int32_t>(best_g);
      s.sk_iters = iters;
    }
  }
  ch.cost = best * kdepth * tile_kb_cost(tc);
  ch.valid = true;
  return ch;
}

gemm_status_t make_plan(const Options& o, const SlotTable& slots, gemm_op_t transA, gemm_op_t transB,
                        int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                        int64_t ldb, float beta, const void* C, int64_t ldc, gemm_dtype_t dtype,
                        Plan* out, int64_t batch = 1, int64_t strideA = 0, int64_t strideB = 0,
                        int64_t strideC = 0, int64_t groups = 0, const int64_t* m_sizes = nullptr,
                        const BlockScale* bs = nullptr) {
  Plan pl;
  gemm_plan_t& P = pl.pub;
  if ((transA != GEMM_OP_N && transA != GEMM_OP_T) || (transB != GEMM_OP_N && transB != GEMM_OP_T))
    return GEMM_ERR_INVALID_ARG;
  const DtypeInfo dt = dtype_info(dtype);
  if (!dt.valid) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  // block-scaled types only through gemm_run_block_scaled, which passes the scales
  if ((dt.sc != 0) != (bs != nullptr)) return GEMM_ERR_INVALID_ARG;
  if (dt.sc != 0 && (batch != 1 || groups != 0)) return GEMM_ERR_UNSUPPORTED;
  pl.eb = dt.eb;
  pl.in_dtype = static_cast<int32_t>(dt.map_type);
  pl.c_type = dt.c_type;
  // E4M3 output is a quantised result, written only.
  if (dt.c_type == kCE4M3 && beta != 0.0f) return GEMM_ERR_UNSUPPORTED;
  const int64_t c_elem = pl.c_type == kCF32 ? 4 : pl.c_type == kCE4M3 ? 1 : 2;
  if (batch < 0 || strideA < 0 || strideB < 0 || strideC < 0 || groups < 0) return GEMM_ERR_INVALID_ARG;
  if (groups > 0) {  // stacked rows: A (sum m) x K row-major, one B per group
    if (!m_sizes || transA != GEMM_OP_N || batch != 1) return GEMM_ERR_INVALID_ARG;
    M = 0;
    for (int64_t g = 0; g < groups; ++g) {
      if (m_sizes[g] < 0) return GEMM_ERR_INVALID_ARG;
      M += m_sizes[g];
    }
    pl.I = M;  // the stacked rows (also what the K == 0 path scales)
  }
  P.batch = static_cast<int32_t>(batch > 1 ? batch : 1);
  if (M == 0 || N == 0 || batch == 0) {
    P.path = GEMM_PATH_NOOP;
    *out = pl;
    return GEMM_OK;
  }
  if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
  if (M > kMaxExtent || N > kMaxExtent || K > kMaxExtent || batch > kMaxExtent) return GEMM_ERR_UNSUPPORTED;
  // every batch writes its own C
  if (batch > 1 && strideC < (M - 1) * ldc + N) return GEMM_ERR_INVALID_ARG;
  pl.batch = batch;
  pl.c_sb = batch > 1 ? strideC : 0;
  if (K == 0) {
    P.path = GEMM_PATH_SCALE_C;
    P.launches = 1;
    *out = pl;
    return GEMM_OK;
  }
  if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_ARG;
  if (lda < (transA == GEMM_OP_T ? M : K) || ldb < (transB == GEMM_OP_T ? K : N))
    return GEMM_ERR_INVALID_ARG;
  if (dt.sc != 0) {  // A M x K and B N x K codes, a scale code per block of k
    const int64_t nblk = cdiv(K, dt.block);
    if (!bs->sfa || !bs->sfb || bs->ld_sfa < nblk || bs->ld_sfb < nblk) return GEMM_ERR_INVALID_ARG;
    if (dt.sc == 2 && (lda % 2 != 0 || ldb % 2 != 0)) return GEMM_ERR_INVALID_ARG;  // rows start on a byte
  }
  // 8-bit operands: K-major only (A stored M x K, B stored N x K).
  if (dt.eb == 1 && (transA != GEMM_OP_N || transB != GEMM_OP_T)) return GEMM_ERR_UNSUPPORTED;

  // Stored operands.
  Operand a, b;
  a.ptr = A; a.ld = lda; a.kmajor = transA == GEMM_OP_N;
  a.rows = a.kmajor ? M : K; a.cols = a.kmajor ? K : M;
  b.ptr = B; b.ld = ldb; b.kmajor = transB == GEMM_OP_T;
  b.rows = b.kmajor ? N : K; b.cols = b.kmajor ? K : N;
  if (dt.sc != 0) {  // both are written as bf16 into the workspace first
    a.dq = dt.src_a + 1;
    a.sf = bs->sfa;
    a.ld_sf = bs->ld_sfa;
    b.dq = dt.src_b + 1;
    b.sf = bs->sfb;
    b.ld_sf = bs->ld_sfb;
  }
  a.nb = (batch > 1 && strideA > 0) ? batch : 1;  // a stride of 0 shares one matrix
  b.nb = (batch > 1 && strideB > 0) ? batch : 1;
  if (groups > 1 && strideB > 0) b.nb = groups;  // one weight matrix per group
  a.bstride = a.nb > 1 ? strideA : 0;
  b.bstride = b.nb > 1 ? strideB : 0;
  // fp32 inputs run on the TF32 tensor-core kind, K-major.  One TF32 product
  // per product (GEMM_TF32_F32): an fp32 operand the copy engine can load
  // K-major goes in as it is (the tensor core keeps its top 19 bits); any
  // other is written K-major with its values cut to TF32 the same way.  The
  // fp32 GEMM (GEMM_F32_F32) splits every value x into hi = TF32(x) and lo =
  // TF32(x - hi) and sums lo_a hi_b + hi_a lo_b + hi_a hi_b (the small
  // products first) as one GEMM over three segments of k: A is stored as
  // [lo | hi] and read as [lo | hi | hi], B stored as [hi | lo] and read as
  // [hi | lo | hi], each segment K rounded up to a whole 32-value k-slice
  // (zeros past K) so that no k-slice straddles two segments.
  int64_t Kg = K;  // k extent of the GEMM the kernel runs
  int64_t seg = K;
  if (dt.parts > 0) {
    seg = dt.parts > 1 ? static_cast<int64_t>(round_up(static_cast<size_t>(K), slice_k(dt.eb))) : K;
    Kg = seg * dt.parts;
    for (Operand* op : {&a, &b}) {
      if (dt.parts == 1 && op->kmajor && tma_aligned(op->ptr, op->ld, dt.eb, op->bstride, op->nb)) continue;
      op->split_parts = dt.parts > 1 ? 2 : 1;
      op->split_pattern = dt.parts == 1 ? 0 : op == &a ? 0x1 : 0x2;
      op->seg_map = dt.parts == 1 ? 0 : op == &a ? 0x6 : 0x2;
      op->split_seg = seg;
      op->split_trans = !op->kmajor;
      op->src_k = K;
      op->rows = op->kmajor ? op->rows : op->cols;
      op->cols = op->split_parts * seg;
      op->kmajor = true;
    }
  }

  // A short M rides on the MMA's N dimension: compute C^T = op(B)^T op(A)^T.
  const bool swap = groups == 0 && M <= 64 && N > M;
  // Block-scaled operands of such a swapped (HBM-bound) GEMM: the weights B,
  // streamed once, stay in their codes and the DQ kernel's converter warps
  // write their 16-bit values into the ring as they arrive (fp16 for NVFP4,
  // whose code x scale products fp16 holds exactly; bf16 for MXFP8), instead
  // of a pass that writes two to four times the bytes it reads.  The copy
  // engine needs 16-byte aligned rows of codes and of scale codes.
  bool dq_kernel = false;
  if (dt.sc != 0 && swap && o.dq_kernel == 0) {
    const int64_t row_bytes = dt.sc == 2 ? ldb / 2 : ldb;
    dq_kernel = reinterpret_cast<uintptr_t>(B) % 16 == 0 && row_bytes % 16 == 0 &&
                reinterpret_cast<uintptr_t>(bs->sfb) % 16 == 0 && bs->ld_sfb % 16 == 0;
  }
  if (dq_kernel) {
    b.dq = 0;
    b.codes = true;
    a.dq_f16 = dt.sc == 2;
    pl.dq_fmt = dt.sc == 2 ? 1 : (dt.src_b == 1 ? 3 : 2);
    pl.code_bytes = dt.sc == 2 ? 32 : 64;
    pl.spk = dt.sc == 2 ? 4 : 2;
    pl.code_cols = dt.sc == 2 ? (K + 1) / 2 : K;
    pl.scale_cols = cdiv(K, dt.block);
    if (dt.sc == 2) {  // fp16 operands
      pl.in_dtype = static_cast<int32_t>(CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    }
  }
  P.swap_ab = swap ? 1 : 0;
  pl.I = swap ? N : M;
  pl.J = swap ? M : N;
  pl.K = Kg;
  pl.p = swap ? b : a;
  pl.q = swap ? a : b;
  // the schedule indexes tiles (and split-K partial slots) with 32-bit integers
  if (cdiv(pl.I, kBM) * cdiv(pl.J, 64) * batch > (int64_t{1} << 30)) return GEMM_ERR_UNSUPPORTED;
  pl.a_fmt = swap ? dt.b_fmt : dt.a_fmt;  // formats of the MMA's A (P) and B (Q) operands
  pl.b_fmt = swap ? dt.a_fmt : dt.b_fmt;
  if (dq_kernel && dt.sc == 2) pl.a_fmt = pl.b_fmt = 0;  // fp16
  pl.c_si = swap ? 1 : ldc;
  pl.c_sj = swap ? ldc : 1;
  P.a_kmajor = pl.p.kmajor ? 1 : 0;
  P.b_kmajor = pl.q.kmajor ? 1 : 0;

  const int64_t num_kslices = cdiv(Kg, slice_k(dt.eb));  // 128-byte k-slices
  // Below the machine balance (≈ 2.2 PFLOP/s over ≈ 7 TB/s ≈ 300 FLOP per byte
  // for 16-bit inputs; twice the rate for 8-bit inputs, half for TF32) the
  // GEMM is bound by HBM, not by the tensor cores.
  const double alg_bytes = dt.eb * (static_cast<double>(M) * Kg * a.nb + static_cast<double>(Kg) * N * b.nb) +
                           static_cast<double>(M) * N * batch * c_elem * (beta != 0.0f ? 2 : 1);
  const double rate = dt.eb == 1 ? 2.0 : dt.eb == 4 ? 0.5 : 1.0;
  const bool hbm_bound = 2.0 * static_cast<double>(M) * N * Kg * batch / alg_bytes < 256.0 * rate;

  // Tile configuration and schedule: the configuration with the lowest
  // estimated time, est_time() below.
  // (ties go first; the eight-epilogue-warp kernel of a tile is chosen below,
  // once the store path is known)
  static const int kPreference[kNumTileConfigs] = {4, 3, 2, 1, 5, 0, 9, 8, 7, 6, 12, 11, 10, 13, 14};
  Choice best;
  for (int cfg : kPreference) {
    const TileConfig& c = kTileConfigs[cfg];
    if (c.ew != 4) continue;
    if (c.eb != dt.eb) continue;
    if ((c.dq != 0) != dq_kernel) continue;
    const int path = c.cg == 2 ? GEMM_PATH_TC_2CTA : GEMM_PATH_TC_1CTA;
    if (o.force_path && o.force_path != path) continue;
    if (o.force_bn && c.bn != o.force_bn) continue;
    if (!o.force_bn && c.bn > 64 && pl.J <= c.bn / 2) continue;       // too wide for J
    if (!o.force_path && c.cg == 2 && pl.I <= kBM) continue;          // one row of tiles
    if (c.bn / c.cg < 64 && !pl.q.kmajor) continue;  // half-atom Q halves: K-major only
    int nslots = slots.of(cfg);
    if (o.max_grid) nslots = std::min(nslots, std::max(1, o.max_grid / c.cg));
    // Two k-slices per stage where the ring still holds at least two such stages
    // (a DQ kernel converts one k-slice a stage).
    int kdepth = c.dq ? 1 : o.kdepth ? o.kdepth : default_kdepth(c);
    if (kdepth > 1 && tc_stages(cfg) / kdepth < 2) kdepth = 1;
    // grouped: each group's rows padded to whole tiles
    int64_t tile_rows = cdiv(pl.I, kBM * c.cg);
    if (groups > 0) {
      tile_rows = 0;
      for (int64_t g = 0; g < groups; ++g) tile_rows += cdiv(m_sizes[g], kBM * c.cg);
      if (tile_rows == 0) tile_rows = 1;
    }
    Choice ch = choose_schedule(o, tile_rows, cdiv(pl.J, c.bn), batch,
                                cdiv(num_kslices, kdepth), kdepth, cfg, nslots, hbm_bound);
    if (ch.valid && ch.cost < best.cost - 1e-9) best = ch;
  }
  if (!best.valid) return GEMM_ERR_INVALID_ARG;  // forced options admit no configuration
  const int cg = best.cg;
  const int cl = best.cg;
  pl.sched = best.sched;
  pl.cfg = best.cfg;
  if (groups > 0) {
    const int64_t tile_m = kBM * best.cg;
    pl.group_tiles.assign(1, 0);
    int64_t row = 0;
    for (int64_t g = 0; g < groups; ++g) {
      pl.group_tiles.push_back(pl.group_tiles.back() +
                               static_cast<int32_t>(cdiv(m_sizes[g], tile_m) * pl.sched.tiles_j));
      pl.group_row.push_back(row);
      pl.group_m.push_back(static_cast<int32_t>(m_sizes[g]));
      row += m_sizes[g];
    }
    pl.sched.groups = static_cast<int32_t>(groups);
    pl.sched.group_tile_start = pl.group_tiles.data();  // the host copy, for planning
  }
  pl.sched.raster_group = o.raster_group ? o.raster_group : 8;
  if (pl.sched.raster_group > pl.sched.tiles_i) pl.sched.raster_group = pl.sched.tiles_i;
  P.path = cg == 2 ? GEMM_PATH_TC_2CTA : GEMM_PATH_TC_1CTA;
  P.cluster = cl;
  P.bm = kBM * cg;
  P.bn = best.bn;
  P.kdepth = best.kdepth;
  P.bk = slice_k(dt.eb) * best.kdepth;
  P.stages = tc_stages(best.cfg) / best.kdepth;
  if (o.stages > 0 && o.stages < P.stages) P.stages = o.stages;
  P.schedule = pl.sched.mode;
  P.split_k = pl.sched.mode == kSchedTiles ? pl.sched.split_k : 1;
  P.tiles_i = pl.sched.tiles_i;
  P.tiles_j = pl.sched.tiles_j;
  P.num_kb = pl.sched.num_kb;
  P.tiles = sched_tiles(pl.sched);
  P.dp_tiles = pl.sched.mode == kSchedStreamK ? pl.sched.dp_tiles : static_cast<int32_t>(P.tiles);
  P.sk_slots = pl.sched.mode == kSchedStreamK ? pl.sched.sk_slots : 0;
  P.units = count_units(pl.sched);
  P.raster_group = pl.sched.raster_group;
  P.grid = static_cast<int32_t>(std::min<int64_t>(best.slots, std::max<int64_t>(P.units, 1)) * cl);

  // Workspace: repacked operands, then partial tiles of split tiles.
  size_t ws = 0;
  for (Operand* op : {&pl.p, &pl.q}) {
    if (op->codes) continue;  // read as codes by the DQ kernel
    if (op->split_parts > 0 || op->dq > 0 || !tma_aligned(op->ptr, op->ld, dt.eb, op->bstride, op->nb)) {
      op->repack = true;  // rows padded to whole 16-byte pieces, batches packed
      // (dequantised rows: whole 16-value pieces, one per thread of dequant_launch)
      op->packed_ld = static_cast<int64_t>(round_up(static_cast<size_t>(op->cols), op->dq > 0 ? 16 : 16 / dt.eb));
      op->ws_offset = ws;
      ws = round_up(ws + static_cast<size_t>(op->rows) * op->packed_ld * dt.eb * op->nb, 256);
    }
  }
  P.repack_a = (swap ? pl.q.repack : pl.p.repack) ? 1 : 0;
  P.repack_b = (swap ? pl.p.repack : pl.q.repack) ? 1 : 0;
  if (groups > 0) {
    pl.group_offset = ws;
    ws = round_up(ws + (groups + 1) * 4 + groups * 4, 8);
    ws = round_up(ws + groups * 8, 256);
  }
  if (needs_partials(pl.sched)) {
    pl.partial_offset = ws;
    ws = round_up(ws + static_cast<size_t>(partial_slots(pl.sched)) * cl * best.bn * kBM * 4, 256);
  }
  const bool c_rows_aligned = reinterpret_cast<uintptr_t>(C) % 16 == 0 && (ldc * c_elem) % 16 == 0 &&
                              (pl.c_sb * c_elem) % 16 == 0;
  P.vector_store = (!swap && c_rows_aligned) ? 1 : 0;
  // Bulk tensor stores need 16-byte aligned rows and a row width that is a
  // whole number of 16-byte pieces (a partial piece at the right edge would be
  // written whole, past column N).  With beta != 0 the old C of each block is
  // loaded by the copy engine into the staging buffer the block then leaves
  // from (not for swapped problems, whose blocks leave transposed: they keep
  // the direct path, which reads C as it writes it).  A swapped problem stores
  // transposed blocks (C's rows run along the kernel's J).
  // (a group's rows end inside C: a bulk store could not stop at the group's edge)
  const bool bulk = c_rows_aligned && (N * c_elem) % 16 == 0 && (beta == 0.0f || !swap) && o.tma_store != 2 &&
                    pl.c_type != kCE4M3 && groups == 0;  // 8-bit C leaves through direct stores
  pl.tma_store = !bulk ? kBulkNone : swap ? kBulkTransposed : kBulkRows;
  P.bulk_store = pl.tma_store;
  P.launches = 1 + P.repack_a + P.repack_b;
  // A large C whose rows bulk stores cannot write (misaligned rows, or a width
  // that ends inside a 16-byte piece, which a bulk store would write whole):
  // the kernel writes an aligned copy in the workspace with bulk stores, and a
  // copy kernel moves it into C.  Direct stores cost more than that second pass
  // (4096 x 4097 x 1000: 80 us with direct stores, 40 us with bulk stores).
  // Otherwise, with beta == 0, either each epilogue thread writes its row's
  // whole 16-byte pieces with 1-D bulk copies (the partial pieces at a tile's
  // edges by plain stores), with no second pass over C, or (a large C, one
  // GEMM) the kernel's bulk tensor stores write an aligned copy of C in the
  // workspace that a copy kernel then moves into C.  The row copies cost one
  // copy per row of each 32-column block, which keeps the copy engine busy;
  // with a short K the epilogue is exposed and the second pass is cheaper
  // (4095 x 4097 x 1000 fp32: 86.8 us with row copies, 72.5 us through the
  // copy), with a long K it is hidden (4096 x 4097 x 4096: 102 against 116 us).
  // GEMM_OPT_EPILOGUE = 3 / 4 asks for the copy / the row copies.
  // fp32 C (one GEMM, at least P rows) has a better way: its rows fall into
  // P <= 4 classes of one misalignment each whose rows lie a multiple of 16
  // bytes apart, so each class is a tensor of its own and a block leaves
  // through P tensor stores (GEMM_BULK_ROW_CLASSES; 4095 x 4097 x 1000: see
  // DESIGN's measurements).
  const bool misaligned_ok = !bulk && o.tma_store != 2 && beta == 0.0f && !swap && groups == 0 && pl.c_type != kCE4M3;
  int classes = 0;
  if (misaligned_ok && pl.c_type == kCF32 && pl.batch == 1 && o.tma_store != 3 && o.tma_store != 4) {
    const int64_t g = (ldc * 4) % 16;  // 0, 4, 8 or 12
    const int n = g == 0 ? 1 : g == 8 ? 2 : 4;
    if (M >= n && N >= 8) classes = n;
  }
  const bool staged_ok = misaligned_ok && o.stage_c && pl.batch == 1 && M * N >= (int64_t{1} << 20);
  const bool use_staged = staged_ok && classes == 0 && (o.tma_store == 3 || (o.tma_store != 4 && K < 2048));
  if (misaligned_ok && !use_staged) {
    pl.tma_store = kBulkRowCopies;
    pl.c_classes = classes;
    P.bulk_store = classes > 0 ? GEMM_BULK_ROW_CLASSES : GEMM_BULK_ROW_COPIES;
  } else if (use_staged) {
    pl.c_staged = true;
    pl.c_ws_ld = static_cast<int64_t>(round_up(static_cast<size_t>(N), static_cast<size_t>(16 / c_elem)));
    pl.c_ws_offset = ws;
    ws = round_up(ws + static_cast<size_t>(M) * pl.c_ws_ld * c_elem, 256);
    pl.tma_store = kBulkRows;
    P.bulk_store = GEMM_BULK_STAGED;
    P.vector_store = 1;
    P.launches += 1;
  }
  // Eight epilogue warps (two per tensor-memory lane quarter, each storing half
  // of a tile's columns) where C leaves through direct stores, row classes or
  // per-row copies: there a block's own work (shifting rows across pieces,
  // plain stores at the edges) outweighs the tensor-memory reads, and two warps
  // a quarter share it (4095 x 4097 x 1000 fp32 with ldc = 4097: 69.8 -> 57.9
  // us; ldc = 4100: 56.0 -> 47.8 us).  With bulk tensor stores the tensor-memory
  // reads and shared-memory writes bound the epilogue and the smaller ring of
  // the wider kernel costs more than the warps gain (4096^3 88.3 -> 92.7 us), so
  // the four-warp kernel stays.
  const bool wide_epilogue = pl.tma_store == kBulkNone || pl.tma_store == kBulkRowCopies;
  if (o.epi_warps == 8 || (o.epi_warps == 0 && wide_epilogue)) {
    const TileConfig& c = kTileConfigs[pl.cfg];
    for (int i = 0; i < kNumTileConfigs; ++i) {
      const TileConfig& e = kTileConfigs[i];
      if (e.ew == 8 && e.bn == c.bn && e.cg == c.cg && e.eb == c.eb && e.dq == c.dq &&
          slots.of(i) >= slots.of(pl.cfg) && tc_stages(i) / P.kdepth >= 2) {
        pl.cfg = i;
        P.stages = tc_stages(i) / P.kdepth;
        if (o.stages > 0 && o.stages < P.stages) P.stages = o.stages;
        break;
      }
    }
  }
  P.epilogue_warps = kTileConfigs[pl.cfg].ew;
  P.workspace_bytes = static_cast<int64_t>(ws);
  *out = pl;
  if (out->sched.groups > 0) out->sched.group_tile_start = out->group_tiles.data();  // the copy's own table
  return GEMM_OK;
}

// ------------------------------------------------------------ tensor maps --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Encode the rank-3 tiled map that `d` describes, or copy it out of `cache`
// (when one is given) if the same description was encoded before.
gemm_status_t encode_tiled(TmapCache* cache, const TmapDesc& d, CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) return GEMM_ERR_TENSORMAP;
  auto encode = [fn](const TmapDesc& k, CUtensorMap* m) {
    cuuint64_t dims[3] = {k.dims[0], k.dims[1], k.dims[2]};
    cuuint64_t strides[2] = {k.strides[0], k.strides[1]};
    cuuint32_t box[3] = {k.box[0], k.box[1], k.box[2]};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, static_cast<CUtensorMapDataType>(k.dtype), 3, reinterpret_cast<void*>(k.base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, static_cast<CUtensorMapSwizzle>(k.swizzle),
              static_cast<CUtensorMapL2promotion>(k.promotion), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const bool ok = cache ? cache->get(d, map, encode) : encode(d, map);
  return ok ? GEMM_OK : GEMM_ERR_TENSORMAP;
}

// Describe operand `op` (possibly its repacked copy at `base`/`ld`) for 2-D tiled
// loads with the 128-byte swizzle: K-major tiles are {one 128-byte k-slice} x
// {box_rows rows} (64 16-bit or 128 8-bit elements of k); MN-major tiles
// (16-bit only) are {64 rows of M/N} x {64 k}, loaded one 64-wide atom at a time.
gemm_status_t encode_operand(CUtensorMap* map, const Operand& op, const void* base, int64_t ld,
                             int64_t bstride, int eb, int32_t map_type, int box_rows, TmapCache* cache) {
  // third dimension: the batch (one matrix when shared; its stride is then any valid value)
  uint64_t dims[3];
  dims[2] = static_cast<uint64_t>(op.nb);
  const int64_t one = round_up(static_cast<size_t>(op.rows * ld * eb), 16);
  const uint64_t strides[2] = {static_cast<uint64_t>(ld) * eb, static_cast<uint64_t>(op.nb > 1 ? bstride * eb : one)};
  uint32_t box[3];
  box[2] = 1;
  if (op.kmajor) {
    dims[0] = static_cast<uint64_t>(op.cols);  // K
    dims[1] = static_cast<uint64_t>(op.rows);  // M or N
    box[0] = static_cast<uint32_t>(slice_k(eb));
    box[1] = static_cast<uint32_t>(box_rows);
  } else {
    dims[0] = static_cast<uint64_t>(op.cols);  // M or N
    dims[1] = static_cast<uint64_t>(op.rows);  // K
    box[0] = 64;
    box[1] = kBK;
  }
  return encode_tiled(cache, tmap_desc(base, dims, strides, box, map_type, CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B), map);
}

// Describe C as stored (rows x cols, row pitch ldc) for bulk stores.  Rows:
// boxes of 32 rows x 128 bytes with the 128-byte swizzle.  Transposed: boxes
// of 32 rows x 32 elements, 128-byte swizzled for fp32, plain for 16 bits.
gemm_status_t encode_c(CUtensorMap* map, void* C, int64_t rows, int64_t cols, int64_t ldc,
                       int32_t c_type, bool transposed, int64_t batch, int64_t strideC, TmapCache* cache) {
  const int64_t esize = c_type == kCF32 ? 4 : 2;
  const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows), static_cast<uint64_t>(batch)};
  const int64_t one = round_up(static_cast<size_t>(rows * ldc * esize), 16);
  const uint64_t strides[2] = {static_cast<uint64_t>(ldc * esize),
                               static_cast<uint64_t>(batch > 1 ? strideC * esize : one)};
  const uint32_t box[3] = {static_cast<uint32_t>(transposed ? 32 : 128 / esize), 32, 1};
  const int swz = transposed && esize == 2 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  const int dt = c_type == kCF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                 : c_type == kCBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return encode_tiled(cache, tmap_desc(C, dims, strides, box, dt, swz, CU_TENSOR_MAP_L2_PROMOTION_NONE), map);
}

// A DQ kernel's P operand as it is stored: rows of block-scaled codes
// (code_cols bytes a row, ld_bytes apart; boxes of code_bytes x 128 rows,
// one k-slice) and their scale codes (scale_cols bytes a row, ld_sf apart;
// boxes of 16 x 128 rows, four or eight k-slices' worth).  Bytes past a row's
// codes or scale codes arrive as zeros.
gemm_status_t encode_codes(CUtensorMap* codes, CUtensorMap* scales, const void* ptr, int64_t rows, int64_t code_cols,
                           int64_t ld_bytes, int code_bytes, const void* sf, int64_t scale_cols, int64_t ld_sf,
                           TmapCache* cache) {
  const uint64_t dims[3] = {static_cast<uint64_t>(code_cols), static_cast<uint64_t>(rows), 1};
  const uint64_t strides[2] = {static_cast<uint64_t>(ld_bytes), round_up(static_cast<size_t>(rows * ld_bytes), 16)};
  const uint32_t box[3] = {static_cast<uint32_t>(code_bytes), static_cast<uint32_t>(kBM), 1};
  gemm_status_t s = encode_tiled(cache, tmap_desc(ptr, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                                 codes);
  if (s != GEMM_OK) return s;
  const uint64_t sdims[3] = {static_cast<uint64_t>(scale_cols), static_cast<uint64_t>(rows), 1};
  const uint64_t sstrides[2] = {static_cast<uint64_t>(ld_sf), round_up(static_cast<size_t>(rows * ld_sf), 16)};
  const uint32_t sbox[3] = {16, static_cast<uint32_t>(kBM), 1};
  return encode_tiled(cache, tmap_desc(sf, sdims, sstrides, sbox, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      scales);
}

// The row-class tensor maps of fp32 C (rows x cols, row pitch ldc elements,
// rows off 16-byte boundaries; see CMaps): class r holds rows r, r + P, ...,
// its base rounded down to 16 bytes and its columns shifted by the rounding,
// its width cut to whole 16-byte pieces.
gemm_status_t encode_c_classes(CMaps* cm, void* C, int64_t rows, int64_t cols, int64_t ldc, int P, TmapCache* cache) {
  std::memset(cm, 0, sizeof(*cm));
  for (int r = 0; r < P; ++r) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(C) + static_cast<uintptr_t>(r * ldc * 4);
    const int64_t sh = static_cast<int64_t>((addr & 15u) / 4);
    const uint64_t nrows = static_cast<uint64_t>((rows - r + P - 1) / P);
    // whole 16-byte pieces only: a tensor store writes the whole last piece of
    // a row that ends inside one, so the values past the last whole piece go
    // out by plain stores
    const uint64_t dims[3] = {static_cast<uint64_t>((cols + sh) & ~int64_t{3}), nrows, 1};
    const uint64_t strides[2] = {static_cast<uint64_t>(P * ldc * 4), round_up(nrows * P * ldc * 4, 16)};
    const void* base = reinterpret_cast<const void*>(addr - static_cast<uintptr_t>(sh * 4));
    const uint32_t rows_box = static_cast<uint32_t>(32 / P);
    const uint32_t box[3] = {32, rows_box, 1};
    const uint32_t box_first[3] = {28, rows_box, 1};
    gemm_status_t s = encode_tiled(cache, tmap_desc(base, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE),
                                   &cm->m[r]);
    if (s != GEMM_OK) return s;
    s = encode_tiled(cache, tmap_desc(base, dims, strides, box_first, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE),
                     &cm->m[4 + r]);
    if (s != GEMM_OK) return s;
  }
  return GEMM_OK;
}

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) changed = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

}  // namespace

// Plans of recent plain and strided-batched calls, so that a repeated call
// skips the planner (its schedule search costs several microseconds on the
// host).  A plan depends on the pointers only through their 16-byte alignment;
// a hit gets the call's own pointers back.
struct PlanKey {
  int32_t transA, transB, dtype;
  uint32_t align_a, align_b, align_c;
  int64_t M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC;
  float beta;
  Options opt;
};
constexpr int kPlanCache = 32;
struct PlanCache {
  PlanKey key[kPlanCache];
  Plan plan[kPlanCache];
  uint64_t used[kPlanCache] = {};  // 0: empty; else the tick of the last use
  uint64_t tick = 0;
  uint64_t hits = 0, misses = 0;
};

// gemm_run_host: device copies of A, B and C, and the two copy streams (one
// per direction) whose transfers overlap the GEMMs of neighbouring row chunks.
constexpr int kHostChunks = 4;
constexpr int kHostBlocks = kHostChunks * kHostChunks;  // blocks of C: row chunks x column chunks
struct HostStage {
  void* a = nullptr;
  void* b = nullptr;
  void* c = nullptr;
  size_t a_bytes = 0, b_bytes = 0, c_bytes = 0;
  cudaStream_t up = nullptr, down = nullptr;  // host -> device, device -> host
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t loaded[kHostBlocks] = {};       // a block's operands (and old C) are on the device
  cudaEvent_t computed[kHostBlocks] = {};     // a block's C is ready to copy back
};

struct gemm_handle_s {
  int device = -1;
  int sm_count = 0;
  int32_t* d_status = nullptr;
  int32_t* d_counters = nullptr;
  void* d_ws = nullptr;
  size_t ws_bytes = 0;
  uint64_t launches = 0;
  int last_cuda_error = 0;
  SlotTable slots;  // resident slots (CTAs, pairs, clusters) per kernel configuration
  Options opt;
  HostStage host;
  PlanCache plans;
  TmapCache tmaps;  // encoded tensor maps of recent calls
};

static gemm_status_t cuda_fail(gemm_handle_t h, cudaError_t e) {
  if (h) h->last_cuda_error = static_cast<int>(e);
  return GEMM_ERR_CUDA;
}

extern "C" {

gemm_status_t gemm_create(gemm_handle_t* out, int device) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return GEMM_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_NO_DEVICE;  // built for sm_103a only
  gemm_handle_t h = new (std::nothrow) gemm_handle_s;
  if (!h) return GEMM_ERR_WORKSPACE;
  h->device = device;
  h->sm_count = prop.multiProcessorCount;
  DeviceGuard g(device);
  // Opt every kernel configuration in to its shared memory, and count how many
  // of its clusters can be resident at once.
  cudaError_t e = measure_slots(h->sm_count, &h->slots);
  if (e == cudaSuccess) e = cudaMalloc(&h->d_status, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&h->d_counters, kCounterCap * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->d_counters, 0, kCounterCap * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->d_status);
    cudaFree(h->d_counters);
    delete h;
    return GEMM_ERR_CUDA;
  }
  *out = h;
  return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h) {
  if (!h) return GEMM_OK;
  {
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->d_ws);
    cudaFree(h->d_counters);
    cudaFree(h->d_status);
    HostStage& hs = h->host;
    cudaFree(hs.a);
    cudaFree(hs.b);
    cudaFree(hs.c);
    if (hs.up) cudaStreamDestroy(hs.up);
    if (hs.down) cudaStreamDestroy(hs.down);
    if (hs.start) cudaEventDestroy(hs.start);
    if (hs.end) cudaEventDestroy(hs.end);
    for (int i = 0; i < kHostBlocks; ++i) {
      if (hs.loaded[i]) cudaEventDestroy(hs.loaded[i]);
      if (hs.computed[i]) cudaEventDestroy(hs.computed[i]);
    }
  }
  delete h;
  return GEMM_OK;
}

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported size";
    case GEMM_ERR_NO_DEVICE: return "no sm_103 device";
    case GEMM_ERR_CUDA: return "CUDA runtime error";
    case GEMM_ERR_TENSORMAP: return "tensor map encoding failed";
    case GEMM_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case GEMM_ERR_WORKSPACE: return "workspace allocation failed";
  }
  return "unknown status";
}

int gemm_last_cuda_error(gemm_handle_t h) { return h ? h->last_cuda_error : 0; }

gemm_status_t gemm_set_option(gemm_handle_t h, gemm_option_t opt, int64_t value) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  switch (opt) {
    case GEMM_OPT_WAIT_LIMIT_NS:
      if (value < 1000000) return GEMM_ERR_INVALID_ARG;
      h->opt.wait_limit_ns = value;
      return GEMM_OK;
    case GEMM_OPT_FORCE_PATH:
      if (value != 0 && value != GEMM_PATH_TC_1CTA && value != GEMM_PATH_TC_2CTA) return GEMM_ERR_INVALID_ARG;
      h->opt.force_path = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_SPLIT_K:
      if (value < 0 || value > 64) return GEMM_ERR_INVALID_ARG;
      h->opt.split_k = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_RASTER_GROUP:
      if (value < 0 || value > 1024) return GEMM_ERR_INVALID_ARG;
      h->opt.raster_group = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_FORCE_BN:
      if (value != 0 && value != 64 && value != 128 && value != 256) return GEMM_ERR_INVALID_ARG;
      h->opt.force_bn = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_TEST_DROP_LOAD:
      if (value < 0 || value > (int64_t{1} << 30)) return GEMM_ERR_INVALID_ARG;
      h->opt.drop_load = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_MAX_GRID:
      if (value < 0 || value > (int64_t{1} << 20)) return GEMM_ERR_INVALID_ARG;
      h->opt.max_grid = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_STREAM_K:
      if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
      h->opt.stream_k = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_STAGES:
      if (value < 0 || value > 64) return GEMM_ERR_INVALID_ARG;
      h->opt.stages = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_EPILOGUE:
      if (value < 0 || value > 4) return GEMM_ERR_INVALID_ARG;
      h->opt.tma_store = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_KDEPTH:
      if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
      h->opt.kdepth = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_PDL:
      if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
      h->opt.pdl = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_PLAN_CACHE:
      if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
      h->opt.plan_cache = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_DEQUANT_IN_KERNEL:
      if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
      h->opt.dq_kernel = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_EPILOGUE_WARPS:
      if (value != 0 && value != 4 && value != 8) return GEMM_ERR_INVALID_ARG;
      h->opt.epi_warps = static_cast<int>(value);
      return GEMM_OK;
  }
  return GEMM_ERR_INVALID_ARG;
}

gemm_status_t gemm_plan_cache_stats(gemm_handle_t h, uint64_t* hits, uint64_t* misses) {
  if (!h || !hits || !misses) return GEMM_ERR_INVALID_ARG;
  *hits = h->plans.hits;
  *misses = h->plans.misses;
  return GEMM_OK;
}

gemm_status_t gemm_tensor_map_cache_stats(gemm_handle_t h, uint64_t* hits, uint64_t* misses) {
  if (!h || !hits || !misses) return GEMM_ERR_INVALID_ARG;
  *hits = h->tmaps.hits;
  *misses = h->tmaps.misses;
  return GEMM_OK;
}

gemm_status_t gemm_launch_count(gemm_handle_t h, uint64_t* count) {
  if (!h || !count) return GEMM_ERR_INVALID_ARG;
  *count = h->launches;
  return GEMM_OK;
}

gemm_status_t gemm_plan_strided_batched(gemm_handle_t h, int sm_count, gemm_op_t transA, gemm_op_t transB,
                                        int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                        int64_t strideA, const void* B, int64_t ldb, int64_t strideB,
                                        float beta, const void* C, int64_t ldc, int64_t strideC,
                                        int64_t batch, gemm_dtype_t dtype, gemm_plan_t* plan) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  if (!h && sm_count <= 0) return GEMM_ERR_INVALID_ARG;
  Options o = h ? h->opt : Options();
  const SlotTable slots = h ? h->slots : SlotTable::even(sm_count);
  Plan pl;
  gemm_status_t s = make_plan(o, slots, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl,
                              batch, strideA, strideB, strideC);
  if (s == GEMM_OK) *plan = pl.pub;
  return s;
}

gemm_status_t gemm_plan(gemm_handle_t h, int sm_count, gemm_op_t transA, gemm_op_t transB,
                        int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                        const void* B, int64_t ldb, float beta, const void* C, int64_t ldc,
                        gemm_dtype_t dtype, gemm_plan_t* plan) {
  return gemm_plan_strided_batched(h, sm_count, transA, transB, M, N, K, A, lda, 0, B, ldb, 0, beta, C, ldc,
                                   0, 1, dtype, plan);
}

// Write the operands the copy engine cannot read as they are (repacked or
// split into TF32 parts) into the workspace at `ws`; *pbase / *qbase and their
// leading dimensions then describe what the kernel loads.  Counts launches.
static cudaError_t prepare_operands(const Plan& pl, uint8_t* ws, int sm_count, cudaStream_t st,
                                    const void** pbase, int64_t* pld, const void** qbase, int64_t* qld,
                                    uint64_t* launches) {
  *pbase = pl.p.ptr;
  *qbase = pl.q.ptr;
  *pld = pl.p.ld;
  *qld = pl.q.ld;
  for (int w = 0; w < 2; ++w) {
    const Operand& op = w == 0 ? pl.p : pl.q;
    if (!op.repack) continue;
    void* dst = ws + op.ws_offset;
    cudaError_t e;
    if (op.dq > 0)
      e = dequant_launch(op.ptr, op.ld, op.sf, op.ld_sf, op.dq - 1, op.dq - 1 != 2 /* MXFP8: E8M0 */,
                         op.dq - 1 == 2 ? 16 : 32, dst, op.packed_ld, op.rows, op.cols, op.dq_f16, sm_count, st);
    else if (op.split_parts > 0)
      e = split_tf32_launch(static_cast<const float*>(op.ptr), op.ld, op.bstride, op.split_trans,
                            static_cast<float*>(dst), op.packed_ld, op.rows * op.packed_ld, op.rows, op.src_k,
                            op.split_seg, op.nb, op.split_parts, op.split_pattern, sm_count, st);
    else
      e = repack_launch(op.ptr, op.ld, op.bstride, dst, op.packed_ld, op.rows * op.packed_ld, op.rows, op.cols,
                        op.nb, pl.eb, sm_count, st);
    if (e != cudaSuccess) return e;
    if (launches) *launches += 1;
    if (w == 0) { *pbase = dst; *pld = op.packed_ld; } else { *qbase = dst; *qld = op.packed_ld; }
  }
  return cudaSuccess;
}

// make_plan through the handle's cache (plain and strided-batched calls).
static gemm_status_t cached_plan(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N,
                                 int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                                 const void* C, int64_t ldc, gemm_dtype_t dtype, Plan* pl, int64_t batch,
                                 int64_t strideA, int64_t strideB, int64_t strideC) {
  if (!h->opt.plan_cache)
    return make_plan(h->opt, h->slots, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, pl, batch,
                     strideA, strideB, strideC);
  PlanKey k;
  std::memset(&k, 0, sizeof(k));  // (padding too: keys compare bytewise)
  k.transA = transA;
  k.transB = transB;
  k.dtype = dtype;
  k.align_a = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(A) % 16) | (A ? 0u : 0x100u);
  k.align_b = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(B) % 16) | (B ? 0u : 0x100u);
  k.align_c = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(C) % 16) | (C ? 0u : 0x100u);
  k.M = M; k.N = N; k.K = K; k.lda = lda; k.ldb = ldb; k.ldc = ldc;
  k.batch = batch; k.strideA = strideA; k.strideB = strideB; k.strideC = strideC;
  k.beta = beta;
  k.opt = h->opt;
  PlanCache& pc = h->plans;
  ++pc.tick;
  int victim = 0;
  for (int e = 0; e < kPlanCache; ++e) {
    if (pc.used[e] != 0 && std::memcmp(&pc.key[e], &k, sizeof(k)) == 0) {
      pc.used[e] = pc.tick;
      ++pc.hits;
      *pl = pc.plan[e];
      // this call's operands (a swapped problem has B on the MMA's rows)
      pl->p.ptr = pl->pub.swap_ab ? B : A;
      pl->q.ptr = pl->pub.swap_ab ? A : B;
      return GEMM_OK;
    }
    if (pc.used[e] < pc.used[victim]) victim = e;
  }
  ++pc.misses;
  const gemm_status_t s = make_plan(h->opt, h->slots, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype,
                                    pl, batch, strideA, strideB, strideC);
  if (s == GEMM_OK) {
    pc.key[victim] = k;
    pc.plan[victim] = *pl;
    pc.used[victim] = pc.tick;
  }
  return s;
}

static gemm_status_t run_gemm(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M,
                              int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                              const void* B, int64_t ldb, float beta, void* C, int64_t ldc,
                              gemm_dtype_t dtype, EpiOps ops, void* stream, int64_t batch = 1,
                              int64_t strideA = 0, int64_t strideB = 0, int64_t strideC = 0,
                              int64_t groups = 0, const int64_t* m_sizes = nullptr,
                              const BlockScale* bs = nullptr, bool allow_pdl = true) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  Plan pl;
  gemm_status_t s =
      (groups == 0 && bs == nullptr)
          ? cached_plan(h, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl, batch, strideA,
                        strideB, strideC)
          : make_plan(h->opt, h->slots, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl, batch,
                      strideA, strideB, strideC, groups, m_sizes, bs);
  if (s == GEMM_OK && groups > 0) M = pl.I;  // the stacked rows
  if (s != GEMM_OK) return s;
  const gemm_plan_t& P = pl.pub;
  if (P.path == GEMM_PATH_NOOP) return GEMM_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceGuard g(h->device);
  cudaError_t e;
  if (P.path == GEMM_PATH_SCALE_C) {
    ops.bias_on_i = 0;  // C as stored: the bias runs along its columns
    e = scale_c_launch(C, pl.c_type, M, N, ldc, beta, ops, pl.batch, pl.c_sb, h->sm_count, st);
    if (e != cudaSuccess) return cuda_fail(h, e);
    h->launches += 1;
    return GEMM_OK;
  }

  // Grow the workspace (synchronous: cudaFree waits for work that may still use it).
  if (static_cast<size_t>(P.workspace_bytes) > h->ws_bytes) {
    const size_t want = round_up(static_cast<size_t>(P.workspace_bytes) + (size_t{1} << 20), 1 << 20);
    void* nw = nullptr;
    e = cudaMalloc(&nw, want);
    if (e != cudaSuccess) {
      cudaGetLastError();
      h->last_cuda_error = static_cast<int>(e);
      return GEMM_ERR_WORKSPACE;
    }
    cudaFree(h->d_ws);
    h->d_ws = nw;
    h->ws_bytes = want;
  }
  const int cg = P.bm / kBM;

  // Operands that the copy engine cannot read directly are repacked (or split) first.
  const void* pbase;
  const void* qbase;
  int64_t pld, qld;
  uint8_t* ws = static_cast<uint8_t*>(h->d_ws);
  e = prepare_operands(pl, ws, h->sm_count, st, &pbase, &pld, &qbase, &qld, &h->launches);
  if (e != cudaSuccess) return cuda_fail(h, e);

  CUtensorMap map_p, map_q;
  TmapCache* tc = &h->tmaps;
  CMaps cmaps;
  std::memset(&cmaps, 0, sizeof(cmaps));
  if (pl.p.codes)  // (a DQ kernel: P's codes, and their scale codes in cmaps.m[0])
    s = encode_codes(&map_p, &cmaps.m[0], pl.p.ptr, pl.p.rows, pl.code_cols, pl.dq_fmt == 1 ? pl.p.ld / 2 : pl.p.ld,
                     pl.code_bytes, pl.p.sf, pl.scale_cols, pl.p.ld_sf, tc);
  else
    s = encode_operand(&map_p, pl.p, pbase, pld, pl.p.repack ? pl.p.rows * pld : pl.p.bstride, pl.eb,
                       pl.in_dtype, kBM, tc);
  if (s != GEMM_OK) return s;
  s = encode_operand(&map_q, pl.q, qbase, qld, pl.q.repack ? pl.q.rows * qld : pl.q.bstride, pl.eb,
                     pl.in_dtype, P.bn / cg, tc);
  if (s != GEMM_OK) return s;
  CUtensorMap map_c;
  std::memset(&map_c, 0, sizeof(map_c));
  // (staged C: the kernel writes the aligned copy, whole rows of c_ws_ld elements)
  void* c_out = pl.c_staged ? static_cast<void*>(ws + pl.c_ws_offset) : C;
  const int64_t c_ld = pl.c_staged ? pl.c_ws_ld : ldc;
  if (pl.tma_store == kBulkRows || pl.tma_store == kBulkTransposed) {
    // C as stored: I x J, or J x I for a swapped problem
    s = pl.tma_store == kBulkRows
            ? encode_c(&map_c, c_out, pl.I, pl.c_staged ? pl.c_ws_ld : pl.J, c_ld, pl.c_type, false, pl.batch, pl.c_sb,
                       tc)
            : encode_c(&map_c, C, pl.J, pl.I, ldc, pl.c_type, true, pl.batch, pl.c_sb, tc);
    if (s != GEMM_OK) return s;
  }

  if (pl.c_classes > 0) {
    s = encode_c_classes(&cmaps, C, pl.I, pl.J, ldc, pl.c_classes, tc);
    if (s != GEMM_OK) return s;
  }

  TcArgs a;
  std::memset(&a, 0, sizeof(a));
  a.I = static_cast<int32_t>(pl.I);
  a.J = static_cast<int32_t>(pl.J);
  a.K = static_cast<int32_t>(pl.K);
  a.sched = pl.sched;
  a.p_kmajor = P.a_kmajor;
  a.q_kmajor = P.b_kmajor;
  a.stages = P.stages;
  a.kdepth = P.kdepth;
  a.idesc = make_idesc(pl.a_fmt, pl.b_fmt, !pl.p.kmajor, !pl.q.kmajor, kBM * cg, P.bn);
  a.alpha = alpha;
  a.beta = beta;
  a.c_classes = pl.c_classes;
  a.dq_fmt = pl.dq_fmt;
  a.code_bytes = pl.code_bytes;
  a.spk = pl.spk;
  if (pl.dq_fmt != 0) {  // the code ring: Q's 16-bit tile, 128 rows of codes, 128 x 16 bytes of scale codes
    a.code_stage_bytes = P.bn / cg * kSliceBytes + kBM * pl.code_bytes + kBM * 16;
    a.code_stages = std::min(16, tc_code_ring_bytes(pl.cfg) / a.code_stage_bytes);
  }
  a.C = c_out;
  a.c_si = pl.c_staged ? pl.c_ws_ld : pl.c_si;
  a.c_sj = pl.c_sj;
  a.c_sb = pl.c_sb;
  a.p_bcast = pl.p.nb == 1 ? 1 : 0;
  a.q_bcast = pl.q.nb == 1 ? 1 : 0;
  a.c_type = pl.c_type;
  a.vec_store = P.vector_store;
  a.tma_store = pl.tma_store;
  a.partials = needs_partials(pl.sched) ? reinterpret_cast<float*>(ws + pl.partial_offset) : nullptr;
  a.counters = h->d_counters;
  a.status = h->d_status;
  a.wait_limit_ns = static_cast<uint64_t>(h->opt.wait_limit_ns);
  if (pl.sched.groups > 0) {  // the group tables go to the workspace with the launch's stream
    const int64_t G = pl.sched.groups;
    uint8_t* base = ws + pl.group_offset;
    int32_t* d_tiles = reinterpret_cast<int32_t*>(base);
    int32_t* d_m = d_tiles + (G + 1);
    int64_t* d_row = reinterpret_cast<int64_t*>(base + round_up((G + 1) * 4 + G * 4, 8));
    e = cudaMemcpyAsync(d_tiles, pl.group_tiles.data(), (G + 1) * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_m, pl.group_m.data(), G * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_row, pl.group_row.data(), G * 8, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(h, e);
    a.sched.group_tile_start = d_tiles;
    a.group_m = d_m;
    a.group_row = d_row;
  }
  a.drop_load = h->opt.drop_load;
  // (grouped: the group tables are copied just before; host calls: an event wait comes just before)
  a.pdl = (pl.sched.groups > 0 || !allow_pdl) ? 0 : h->opt.pdl;
  // three-product fp32 GEMM: the logical k runs over three stored segments
  a.seg_slices = pl.p.seg_map != 0 ? static_cast<int32_t>(pl.p.split_seg / slice_k(pl.eb)) : 0;
  a.p_seg = pl.p.seg_map;
  a.q_seg = pl.q.seg_map;
  ops.bias_on_i = P.swap_ab;  // a swapped problem computes C^T: C's columns are the kernel's rows
  a.ops = ops;
  e = tc_launch(pl.cfg, map_p, map_q, map_c, cmaps, a, P.grid, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  h->launches += 1;
  if (pl.c_staged) {  // the aligned copy's M x N elements into C
    const int c_elem = pl.c_type == kCF32 ? 4 : 2;
    e = unstage_c_launch(c_out, pl.c_ws_ld, C, ldc, pl.I, pl.J, c_elem, st);
    if (e != cudaSuccess) return cuda_fail(h, e);
    h->launches += 1;
  }
  return GEMM_OK;
}

gemm_status_t gemm_run(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N,
                       int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                       int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtype_t dtype,
                       void* stream) {
  return run_gemm(h, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, EpiOps(),
                  stream);
}

static gemm_status_t epi_ops(const gemm_epilogue_t* epi, EpiOps* out) {
  EpiOps ops;
  if (epi) {
    if (epi->activation < GEMM_ACT_NONE || epi->activation > GEMM_ACT_GELU) return GEMM_ERR_INVALID_ARG;
    if (!std::isfinite(epi->out_scale)) return GEMM_ERR_INVALID_ARG;
    if (epi->bias && reinterpret_cast<uintptr_t>(epi->bias) % sizeof(float) != 0) return GEMM_ERR_INVALID_ARG;
    ops.bias = epi->bias;
    ops.act = epi->activation;
    ops.out_scale = epi->out_scale;
  }
  *out = ops;
  return GEMM_OK;
}

gemm_status_t gemm_run_ex(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N,
                          int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                          int64_t ldb, float beta, void* C, int64_t ldc, gemm_dtype_t dtype,
                          const gemm_epilogue_t* epi, void* stream) {
  EpiOps ops;
  gemm_status_t s = epi_ops(epi, &ops);
  if (s != GEMM_OK) return s;
  return run_gemm(h, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, ops, stream);
}

gemm_status_t gemm_run_grouped(gemm_handle_t h, gemm_op_t transB, int64_t groups, const int64_t* m_sizes,
                               int64_t N, int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                               int64_t ldb, int64_t strideB, float beta, void* C, int64_t ldc,
                               gemm_dtype_t dtype, const gemm_epilogue_t* epi, void* stream) {
  EpiOps ops;
  gemm_status_t s = epi_ops(epi, &ops);
  if (s != GEMM_OK) return s;
  if (!h || groups < 0 || (groups > 0 && !m_sizes)) return GEMM_ERR_INVALID_ARG;
  if (groups == 0) return GEMM_OK;
  return run_gemm(h, GEMM_OP_N, transB, 0, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, ops, stream, 1, 0,
                  strideB, 0, groups, m_sizes);
}

gemm_status_t gemm_run_block_scaled(gemm_handle_t h, int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                                    int64_t lda, const void* SFA, int64_t ld_sfa, const void* B, int64_t ldb,
                                    const void* SFB, int64_t ld_sfb, float beta, void* C, int64_t ldc,
                                    gemm_dtype_t dtype, const gemm_epilogue_t* epi, void* stream) {
  EpiOps ops;
  gemm_status_t s = epi_ops(epi, &ops);
  if (s != GEMM_OK) return s;
  if (dtype_info(dtype).sc == 0) return GEMM_ERR_INVALID_ARG;
  BlockScale bs;
  bs.sfa = SFA;
  bs.ld_sfa = ld_sfa;
  bs.sfb = SFB;
  bs.ld_sfb = ld_sfb;
  return run_gemm(h, GEMM_OP_N, GEMM_OP_T, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, ops, stream, 1, 0,
                  0, 0, 0, nullptr, &bs);
}

gemm_status_t gemm_plan_block_scaled(gemm_handle_t h, int sm_count, int64_t M, int64_t N, int64_t K, const void* A,
                                     int64_t lda, const void* SFA, int64_t ld_sfa, const void* B, int64_t ldb,
                                     const void* SFB, int64_t ld_sfb, float beta, const void* C, int64_t ldc,
                                     gemm_dtype_t dtype, gemm_plan_t* plan) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  if (!h && sm_count <= 0) return GEMM_ERR_INVALID_ARG;
  if (dtype_info(dtype).sc == 0) return GEMM_ERR_INVALID_ARG;
  Options o = h ? h->opt : Options();
  const SlotTable slots = h ? h->slots : SlotTable::even(sm_count);
  BlockScale bs;
  bs.sfa = SFA;
  bs.ld_sfa = ld_sfa;
  bs.sfb = SFB;
  bs.ld_sfb = ld_sfb;
  Plan pl;
  gemm_status_t s = make_plan(o, slots, GEMM_OP_N, GEMM_OP_T, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl, 1,
                              0, 0, 0, 0, nullptr, &bs);
  if (s == GEMM_OK) *plan = pl.pub;
  return s;
}

// Grow one device staging buffer (synchronous: the old one may still be in use).
static cudaError_t host_stage_buffer(void** buf, size_t* have, size_t need) {
  if (need <= *have) return cudaSuccess;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  cudaFree(*buf);
  *buf = nullptr;
  *have = 0;
  const size_t want = round_up(need, size_t{1} << 20);
  e = cudaMalloc(buf, want);
  if (e == cudaSuccess) *have = want;
  return e;
}

gemm_status_t gemm_run_host(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N, int64_t K,
                            float alpha, const void* A, int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                            int64_t ldc, gemm_dtype_t dtype, void* stream) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  const DtypeInfo dt = dtype_info(dtype);
  if (!dt.valid) return GEMM_ERR_INVALID_ARG;
  if (dt.sc != 0) return GEMM_ERR_UNSUPPORTED;  // block-scaled inputs: device buffers only
  {  // the argument checks of gemm_run (host pointers stand in for the device copies)
    Plan pl;
    gemm_status_t s = make_plan(h->opt, h->slots, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl);
    if (s != GEMM_OK) return s;
    if (pl.pub.path == GEMM_PATH_NOOP) return GEMM_OK;
  }
  const int64_t ea = dt.eb;
  const int64_t ec = dt.c_type == kCF32 ? 4 : dt.c_type == kCE4M3 ? 1 : 2;
  const int64_t a_rows = transA == GEMM_OP_N ? M : K, a_cols = transA == GEMM_OP_N ? K : M;
  const int64_t b_rows = transB == GEMM_OP_T ? N : K, b_cols = transB == GEMM_OP_T ? K : N;
  const size_t a_bytes = K > 0 ? static_cast<size_t>(((a_rows - 1) * lda + a_cols) * ea) : 0;
  const size_t b_bytes = K > 0 ? static_cast<size_t>(((b_rows - 1) * ldb + b_cols) * ea) : 0;
  const size_t c_bytes = static_cast<size_t>(((M - 1) * ldc + N) * ec);
  DeviceGuard g(h->device);
  HostStage& hs = h->host;
  cudaError_t e = cudaSuccess;
  if (!hs.up) {
    e = cudaStreamCreateWithFlags(&hs.up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hs.down, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hs.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hs.end, cudaEventDisableTiming);
    for (int i = 0; i < kHostBlocks && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&hs.loaded[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hs.computed[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(h, e);
  }
  if ((e = host_stage_buffer(&hs.a, &hs.a_bytes, a_bytes)) != cudaSuccess ||
      (e = host_stage_buffer(&hs.b, &hs.b_bytes, b_bytes)) != cudaSuccess ||
      (e = host_stage_buffer(&hs.c, &hs.c_bytes, c_bytes)) != cudaSuccess) {
    cudaGetLastError();
    h->last_cuda_error = static_cast<int>(e);
    return GEMM_ERR_WORKSPACE;
  }
  // C in blocks of row chunks x column chunks (up to 4 x 4; one chunk along a
  // dimension shorter than 1024).  A's row chunks and B's column chunks go over
  // alternately (A0, B0, A1, B1, ...), and every block of C whose rows and
  // columns have both arrived is multiplied and copied back at once, so that
  // copies out start after an eighth of the inputs and overlap the rest of the
  // copies in.  (Row chunks alone, after all of B: 4096^3 took 0.624 ms; the
  // first row chunk in column blocks: 0.608 ms.)
  const int64_t rch = (M >= 1024 && K > 0) ? static_cast<int64_t>(round_up(static_cast<size_t>(cdiv(M, kHostChunks)), 256)) : M;
  const int64_t cch = (N >= 1024 && K > 0) ? static_cast<int64_t>(round_up(static_cast<size_t>(cdiv(N, kHostChunks)), 256)) : N;
  const int nr = static_cast<int>(cdiv(M, rch));
  const int nc = static_cast<int>(cdiv(N, cch));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ad = static_cast<char*>(hs.a);
  char* bd = static_cast<char*>(hs.b);
  char* cd = static_cast<char*>(hs.c);
  const char* ah = static_cast<const char*>(A);
  const char* bh = static_cast<const char*>(B);
  char* ch = static_cast<char*>(C);
  // A's rows of C r0 .. r0 + rows - 1 (rows of A stored M x K, else a column slice of each of its K rows)
  auto copy_a = [&](int64_t r0, int64_t rows) {
    if (a_bytes == 0) return cudaSuccess;
    if (transA == GEMM_OP_N)
      return cudaMemcpy2DAsync(ad + r0 * lda * ea, lda * ea, ah + r0 * lda * ea, lda * ea, K * ea, rows,
                               cudaMemcpyHostToDevice, hs.up);
    return cudaMemcpy2DAsync(ad + r0 * ea, lda * ea, ah + r0 * ea, lda * ea, rows * ea, K, cudaMemcpyHostToDevice,
                             hs.up);
  };
  // B's columns of C j0 .. j0 + cols - 1 (rows of B stored N x K, else a column slice of each of its K rows)
  auto copy_b = [&](int64_t j0, int64_t cols) {
    if (b_bytes == 0) return cudaSuccess;
    if (transB == GEMM_OP_T)
      return cudaMemcpy2DAsync(bd + j0 * ldb * ea, ldb * ea, bh + j0 * ldb * ea, ldb * ea, K * ea, cols,
                               cudaMemcpyHostToDevice, hs.up);
    return cudaMemcpy2DAsync(bd + j0 * ea, ldb * ea, bh + j0 * ea, ldb * ea, cols * ea, K, cudaMemcpyHostToDevice,
                             hs.up);
  };
  // block (i, j) of C: its old values in for the blend, the GEMM once everything
  // queued on the copy-in stream so far has landed, its values out
  int ev = 0;
  auto block = [&](int i, int j) -> gemm_status_t {
    const int64_t r0 = i * rch, rows = std::min(rch, M - r0);
    const int64_t j0 = j * cch, cols = std::min(cch, N - j0);
    char* cdb = cd + (r0 * ldc + j0) * ec;
    char* chb = ch + (r0 * ldc + j0) * ec;
    cudaError_t e2 = cudaSuccess;
    if (beta != 0.0f)
      e2 = cudaMemcpy2DAsync(cdb, ldc * ec, chb, ldc * ec, cols * ec, rows, cudaMemcpyHostToDevice, hs.up);
    if (e2 == cudaSuccess) e2 = cudaEventRecord(hs.loaded[ev], hs.up);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, hs.loaded[ev], 0);
    if (e2 != cudaSuccess) return cuda_fail(h, e2);
    const char* a_blk = transA == GEMM_OP_N ? ad + r0 * lda * ea : ad + r0 * ea;
    const char* b_blk = transB == GEMM_OP_T ? bd + j0 * ldb * ea : bd + j0 * ea;
    const gemm_status_t s2 = run_gemm(h, transA, transB, rows, cols, K, alpha, a_blk, lda, b_blk, ldb, beta, cdb, ldc,
                                      dtype, EpiOps(), st, 1, 0, 0, 0, 0, nullptr, nullptr, false);
    if (s2 != GEMM_OK) return s2;
    e2 = cudaEventRecord(hs.computed[ev], st);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(hs.down, hs.computed[ev], 0);
    if (e2 == cudaSuccess)
      e2 = cudaMemcpy2DAsync(chb, ldc * ec, cdb, ldc * ec, cols * ec, rows, cudaMemcpyDeviceToHost, hs.down);
    ++ev;
    return e2 == cudaSuccess ? GEMM_OK : cuda_fail(h, e2);
  };
  // the copy streams start after everything already queued on the caller's stream
  e = cudaEventRecord(hs.start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs.up, hs.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs.down, hs.start, 0);
  if (e != cudaSuccess) return cuda_fail(h, e);
  int ia = 0, ib = 0;  // row chunks of A and column chunks of B sent so far
  while (ia < nr || ib < nc) {
    if (ia < nr && (ia <= ib || ib == nc)) {  // A's next row chunk, then its blocks with the columns already there
      e = copy_a(ia * rch, std::min(rch, M - ia * rch));
      if (e != cudaSuccess) return cuda_fail(h, e);
      ++ia;
      for (int j = 0; j < ib; ++j) {
        const gemm_status_t s = block(ia - 1, j);
        if (s != GEMM_OK) return s;
      }
    } else {  // B's next column chunk, then its blocks with the rows already there
      e = copy_b(ib * cch, std::min(cch, N - ib * cch));
      if (e != cudaSuccess) return cuda_fail(h, e);
      ++ib;
      for (int i = 0; i < ia; ++i) {
        const gemm_status_t s = block(i, ib - 1);
        if (s != GEMM_OK) return s;
      }
    }
  }
  // the caller's stream continues once C is back on the host
  if (e == cudaSuccess) e = cudaEventRecord(hs.end, hs.down);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hs.end, 0);
  if (e != cudaSuccess) return cuda_fail(h, e);
  return GEMM_OK;
}

gemm_status_t gemm_plan_grouped(gemm_handle_t h, int sm_count, gemm_op_t transB, int64_t groups,
                                const int64_t* m_sizes, int64_t N, int64_t K, const void* A, int64_t lda,
                                const void* B, int64_t ldb, int64_t strideB, float beta, const void* C,
                                int64_t ldc, gemm_dtype_t dtype, gemm_plan_t* plan) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  if (!h && sm_count <= 0) return GEMM_ERR_INVALID_ARG;
  if (groups < 0 || (groups > 0 && !m_sizes)) return GEMM_ERR_INVALID_ARG;
  Options o = h ? h->opt : Options();
  const SlotTable slots = h ? h->slots : SlotTable::even(sm_count);
  Plan pl;
  gemm_status_t s = GEMM_OK;
  if (groups == 0)
    pl.pub.path = GEMM_PATH_NOOP;
  else
    s = make_plan(o, slots, GEMM_OP_N, transB, 0, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl, 1, 0, strideB,
                  0, groups, m_sizes);
  if (s == GEMM_OK) *plan = pl.pub;
  return s;
}

gemm_status_t gemm_run_strided_batched(gemm_handle_t h, gemm_op_t transA, gemm_op_t transB, int64_t M,
                                       int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                                       int64_t strideA, const void* B, int64_t ldb, int64_t strideB,
                                       float beta, void* C, int64_t ldc, int64_t strideC, int64_t batch,
                                       gemm_dtype_t dtype, const gemm_epilogue_t* epi, void* stream) {
  EpiOps ops;
  gemm_status_t s = epi_ops(epi, &ops);
  if (s != GEMM_OK) return s;
  return run_gemm(h, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, ops, stream, batch,
                  strideA, strideB, strideC);
}

gemm_status_t gemm_probe_tma_tile(gemm_handle_t h, const void* src, int64_t ld, int64_t cols, int64_t rows, void* dst,
                                  void* stream) {
  if (!h || !src || !dst || rows < 1 || rows > 256 || cols < 1 || ld < cols) return GEMM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(src) % 16 != 0 || (ld * 2) % 16 != 0) return GEMM_ERR_INVALID_ARG;
  auto fn = encode_fn();
  if (!fn) return GEMM_ERR_TENSORMAP;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2),
                           static_cast<cuuint64_t>(round_up(static_cast<size_t>(rows * ld * 2), 16))};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap map;
  CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(src), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return GEMM_ERR_TENSORMAP;
  DeviceGuard g(h->device);
  cudaError_t e = tma_tile_probe_launch(map, static_cast<int>(rows), static_cast<uint16_t*>(dst), h->d_status,
                                        static_cast<uint64_t>(h->opt.wait_limit_ns), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e);
  h->launches += 1;
  return GEMM_OK;
}

gemm_status_t gemm_get_status(gemm_handle_t h, void* stream, int32_t* detail) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e);
  int32_t word = 0;
  e = cudaMemcpy(&word, h->d_status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (detail) *detail = word;
  if (word == 0) return GEMM_OK;
  // A kernel gave up part-way: clear the status and any split-K counters it left behind.
  e = cudaMemset(h->d_status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->d_counters, 0, kCounterCap * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e);
  return GEMM_ERR_TIMEOUT;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gemm_run_noalloc: the same GEMM for callers that must not allocate device
// memory.  Its scratch (repacked operands, partial tiles of split tiles,
// arrival counters, the status word) lives in file-scope device arrays that
// every GPU loading the library holds until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t{16} << 20;  // 16 MiB
constexpr int kNoAllocCounters = 4096;
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  SlotTable slots;
  int sm_count = 0;
  uint8_t* scratch = nullptr;  // device addresses of the arrays below, for this device
  int32_t* counters = nullptr;
  int32_t* status = nullptr;
};

NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;
// Process-wide settings of the no-allocation path (gemm_noalloc_set_option):
// the barrier wait limit and the test hook that drops one load.
int64_t g_noalloc_wait_ns = kDefaultWaitNs;
int g_noalloc_drop_load = 0;

}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
static __device__ __align__(256) int32_t g_noalloc_counters[kNoAllocCounters];
static __device__ __align__(256) int32_t g_noalloc_status[64];

// Once per device, with that device current: look up the arrays' device
// addresses (in host code their names are only host-side stand-ins) and opt
// the kernels in to their shared memory.  Allocates nothing.
static gemm_status_t noalloc_setup(int device, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (device < 0 || device >= kNoAllocMaxDevices) return GEMM_ERR_NO_DEVICE;
  NoAllocDevice& d = g_noalloc_devices[device];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;
    d.sm_count = sms;
    if (measure_slots(sms, &d.slots) != cudaSuccess) return GEMM_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return GEMM_ERR_CUDA;
    d.scratch = static_cast<uint8_t*>(p);
    if (cudaGetSymbolAddress(&p, g_noalloc_counters) != cudaSuccess) return GEMM_ERR_CUDA;
    d.counters = static_cast<int32_t*>(p);
    if (cudaGetSymbolAddress(&p, g_noalloc_status) != cudaSuccess) return GEMM_ERR_CUDA;
    d.status = static_cast<int32_t*>(p);
    d.ready = true;
  }
  *out = &d;
  return GEMM_OK;
}

static int64_t counters_needed(const Sched& s, int cluster) {
  if (s.mode == kSchedStreamK)
    return (static_cast<int64_t>(s.tiles_i) * s.tiles_j - s.dp_tiles) * cluster;
  return s.split_k > 1 ? static_cast<int64_t>(s.tiles_i) * s.tiles_j * cluster : 0;
}

extern "C" gemm_status_t gemm_run_noalloc(gemm_op_t transA, gemm_op_t transB, int64_t M, int64_t N,
                                          int64_t K, float alpha, const void* A, int64_t lda,
                                          const void* B, int64_t ldb, float beta, void* C,
                                          int64_t ldc, gemm_dtype_t dtype, void* stream) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  NoAllocDevice* d = nullptr;
  gemm_status_t s = noalloc_setup(device, &d);
  if (s != GEMM_OK) return s;
  Options o;
  o.stage_c = false;  // no room for a copy of C in the fixed scratch
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    o.wait_limit_ns = g_noalloc_wait_ns;
    o.drop_load = g_noalloc_drop_load;
  }
  Plan pl;
  s = make_plan(o, d->slots, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl);
  if (s != GEMM_OK) return s;
  if (pl.pub.path >= GEMM_PATH_TC_1CTA &&
      (static_cast<size_t>(pl.pub.workspace_bytes) > kNoAllocScratchBytes ||
       counters_needed(pl.sched, pl.pub.cluster) > kNoAllocCounters)) {
    o.stream_k = 1;  // whole tiles need no partial sums: plan again without the stream-K tail
    s = make_plan(o, d->slots, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype, &pl);
    if (s != GEMM_OK) return s;
    if (static_cast<size_t>(pl.pub.workspace_bytes) > kNoAllocScratchBytes ||
        counters_needed(pl.sched, pl.pub.cluster) > kNoAllocCounters)
      return GEMM_ERR_WORKSPACE;  // needs more scratch than the fixed 16 MiB array holds
  }
  const int cg = pl.pub.path >= GEMM_PATH_TC_1CTA ? pl.pub.bm / kBM : 1;
  const gemm_plan_t& P = pl.pub;
  if (P.path == GEMM_PATH_NOOP) return GEMM_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (P.path == GEMM_PATH_SCALE_C) {
    e = scale_c_launch(C, pl.c_type, M, N, ldc, beta, EpiOps(), pl.batch, pl.c_sb, d->sm_count, st);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  // The arrays keep the previous call's contents: clear what must start at zero.
  e = cudaMemsetAsync(d->status, 0, sizeof(int32_t), st);
  const int64_t nctr = counters_needed(pl.sched, P.cluster);
  if (e == cudaSuccess && nctr > 0) e = cudaMemsetAsync(d->counters, 0, nctr * sizeof(int32_t), st);
  if (e != cudaSuccess) return GEMM_ERR_CUDA;

  const void* pbase;
  const void* qbase;
  int64_t pld, qld;
  e = prepare_operands(pl, d->scratch, d->sm_count, st, &pbase, &pld, &qbase, &qld, nullptr);
  if (e != cudaSuccess) return GEMM_ERR_CUDA;
  CUtensorMap map_p, map_q;
  s = encode_operand(&map_p, pl.p, pbase, pld, pl.p.repack ? pl.p.rows * pld : pl.p.bstride, pl.eb,
                     pl.in_dtype, kBM, nullptr);
  if (s != GEMM_OK) return s;
  s = encode_operand(&map_q, pl.q, qbase, qld, pl.q.repack ? pl.q.rows * qld : pl.q.bstride, pl.eb,
                     pl.in_dtype, P.bn / cg, nullptr);
  if (s != GEMM_OK) return s;
  CUtensorMap map_c;
  std::memset(&map_c, 0, sizeof(map_c));
  if (pl.tma_store == kBulkRows || pl.tma_store == kBulkTransposed) {
    // C as stored: I x J, or J x I for a swapped problem
    s = pl.tma_store == kBulkRows ? encode_c(&map_c, C, pl.I, pl.J, ldc, pl.c_type, false, pl.batch, pl.c_sb, nullptr)
                                  : encode_c(&map_c, C, pl.J, pl.I, ldc, pl.c_type, true, pl.batch, pl.c_sb, nullptr);
    if (s != GEMM_OK) return s;
  }
  CMaps cmaps;
  std::memset(&cmaps, 0, sizeof(cmaps));
  if (pl.c_classes > 0) {
    s = encode_c_classes(&cmaps, C, pl.I, pl.J, ldc, pl.c_classes, nullptr);
    if (s != GEMM_OK) return s;
  }
  TcArgs a;
  std::memset(&a, 0, sizeof(a));
  a.I = static_cast<int32_t>(pl.I);
  a.J = static_cast<int32_t>(pl.J);
  a.K = static_cast<int32_t>(pl.K);
  a.sched = pl.sched;
  a.p_kmajor = P.a_kmajor;
  a.q_kmajor = P.b_kmajor;
  a.stages = P.stages;
  a.kdepth = P.kdepth;
  a.idesc = make_idesc(pl.a_fmt, pl.b_fmt, !pl.p.kmajor, !pl.q.kmajor, kBM * cg, P.bn);
  a.alpha = alpha;
  a.beta = beta;
  a.c_classes = pl.c_classes;
  a.C = C;
  a.c_si = pl.c_si;
  a.c_sj = pl.c_sj;
  a.c_sb = pl.c_sb;
  a.p_bcast = pl.p.nb == 1 ? 1 : 0;
  a.q_bcast = pl.q.nb == 1 ? 1 : 0;
  a.c_type = pl.c_type;
  a.vec_store = P.vector_store;
  a.tma_store = pl.tma_store;
  a.partials = needs_partials(pl.sched) ? reinterpret_cast<float*>(d->scratch + pl.partial_offset) : nullptr;
  a.counters = d->counters;
  a.status = d->status;
  a.wait_limit_ns = static_cast<uint64_t>(o.wait_limit_ns);
  a.drop_load = o.drop_load;
  a.pdl = 0;  // (the no-allocation entry point clears its arrays first, with ordinary stream order)
  a.seg_slices = pl.p.seg_map != 0 ? static_cast<int32_t>(pl.p.split_seg / slice_k(pl.eb)) : 0;
  a.p_seg = pl.p.seg_map;
  a.q_seg = pl.q.seg_map;
  a.ops = EpiOps();  // no fused operations (the memset above zeroed out_scale)
  e = tc_launch(pl.cfg, map_p, map_q, map_c, cmaps, a, P.grid, st);
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// The status word of the no-allocation path: synchronise `stream`, then read
// the word of the current device's arrays and clear it.  Allocates nothing.
extern "C" gemm_status_t gemm_noalloc_get_status(void* stream, int32_t* detail) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  NoAllocDevice* d = nullptr;
  gemm_status_t s = noalloc_setup(device, &d);
  if (s != GEMM_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, d->status, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return GEMM_ERR_CUDA;
  if (detail) *detail = word;
  if (word == 0) return GEMM_OK;
  // A kernel gave up part-way: clear the word (each call clears the counters it uses).
  e = cudaMemsetAsync(d->status, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return GEMM_ERR_CUDA;
  return GEMM_ERR_TIMEOUT;
}

extern "C" gemm_status_t gemm_noalloc_set_option(gemm_option_t opt, int64_t value) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  switch (opt) {
    case GEMM_OPT_WAIT_LIMIT_NS:
      if (value < 1000000) return GEMM_ERR_INVALID_ARG;
      g_noalloc_wait_ns = value;
      return GEMM_OK;
    case GEMM_OPT_TEST_DROP_LOAD:
      if (value < 0 || value > (int64_t{1} << 30)) return GEMM_ERR_INVALID_ARG;
      g_noalloc_drop_load = static_cast<int>(value);
      return GEMM_OK;
    default:
      return GEMM_ERR_INVALID_ARG;
  }
}
