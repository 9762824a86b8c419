// tc_gemm.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   D (I x J) = P (I x K) * Q (K x J);   C[i*c_si + j*c_sj] = alpha * D[i][j] + beta * C[...]
//
// Design, and the page sections each part restates:
//  * A persistent grid: one CTA per SM walks a static list of work units in a
//    grouped (swizzled) raster order so that CTAs running together share rows
//    of P and columns of Q in L2 ("CUDA GEMM 矩阵乘法优化指南", 12.5 Persistent
//    Kernel; "GPU GEMM 优化完全拆解（三）", rasterization).
//  * Warp specialisation: warp 0 issues TMA copies into a multi-stage shared
//    memory ring guarded by full / empty mbarriers, warp 1 issues tcgen05.mma
//    from one thread, warps 2 .. 2 + EW - 1 run the epilogue (EW = 4, one per
//    32-lane quarter of tensor memory, or 8, two per quarter each storing half
//    of a tile's columns), and in DQ kernels kConvWarps more warps convert
//    block-scaled codes ("GPU GEMM 优化完全拆解（三）", warp specialization;
//    "CUDA GEMM 矩阵乘法优化指南", 12.4 and 13.2).
//  * Tiles arrive 128-byte swizzled ("[CUDA 优化实战] hgemm sm120", section 4:
//    the swizzle of 16-bit element (r, c) in a 64-wide row is c ^ ((r & 7) << 3)),
//    which is the layout the tensor core's shared-memory descriptor expects.
//  * CG == 2 runs one tile on a CTA pair (a cluster of two CTAs on neighbouring
//    SMs, "CUDA GEMM 矩阵乘法优化指南" 13.3-13.4): each CTA loads its 128 rows of P
//    and half of the tile's Q columns, and the leader CTA issues
//    tcgen05.mma.cta_group::2 with M = 256, which reads both CTAs' shared memory.
//    Per SM this halves the Q traffic from L2 for the same tile width.
//  * The fp32 accumulator lives in Tensor Memory, double-buffered so that the
//    epilogue of one tile overlaps the main loop of the next (the ping-pong idea
//    of "GPU GEMM 优化完全拆解（三）", Hopper 时代的三种 kernel 设计).
//  * Split-K and stream-K (schedule.h): a work unit may cover only a k-range
//    of a tile; its fp32 partial goes to a workspace and the last contribution
//    of the tile to arrive sums all partials in fixed k order, so the result is
//    deterministic ("GPU GEMM 优化完全拆解（三）", Split-K 与 Sliced-K;
//    "CUDA GEMM 矩阵乘法优化指南", 12.5).
//  * Every barrier wait is bounded by a wall-clock limit; a wait that runs out
//    records the role and barrier in the status word, raises a CTA-wide abort
//    flag, and every role then leaves its loop.  Before the CTA exits, the
//    producer waits for each of its copies in flight and the MMA thread for its
//    last MMAs, and Tensor Memory is always freed.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "epi_ops.cuh"
#include "gemm_internal.h"
#include "ptx.cuh"

namespace g10 {

template <int BN, int CG, bool DQ = false, int EW = 4>
struct TcConfig {
  static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
  static_assert(CG == 1 || CG == 2, "CTA group");
  // a CTA pair with BN == 64 loads 32-row halves of Q: K-major Q only (an
  // M/N-major swizzle atom is 64 elements wide); the planner enforces it
  static_assert(CG == 1 || BN >= 64, "a CTA pair needs at least 32-row halves of Q");
  static constexpr int kCluster = CG;           // CTAs per cluster
  static constexpr int kTileM = kBM * CG;        // rows of D per tile
  static constexpr int kQRows = BN / CG;         // rows of Q this CTA loads per k-block
  static constexpr int kABytes = kBM * kSliceBytes;  // this CTA's P tile: 128 rows x 128 bytes
  static constexpr int kBBytes = kQRows * kSliceBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // as many stages as fit in 227 KB beside the control block and alignment slack (at most 8)
  // epilogue staging: per epilogue warp two 32-row x 128-byte buffers for C (bulk stores
  // alternate between them; direct stores use the first)
  static_assert(EW == 4 || (EW == 8 && !DQ && BN >= 128), "epilogue warps");
  static constexpr int kEpiWarps = EW;
  static constexpr int kEpiCols = BN / (kEpiWarps / 4);  // columns of a tile one epilogue warp stores
  static constexpr int kStagingBytes = kEpiWarps * 2 * 32 * 128;
  static constexpr int kCtrlBytes = 256;
  static constexpr int kRingMax = 232448 - 1024 - kStagingBytes - 1024;  // 227 KB less the rest
  // DQ: the ring holds only P's converted 16-bit tiles (five stages: the
  // NVFP4 LM head took 63.7 us with three, 61.6 us with five); Q's tile, P's
  // block-scaled codes and a 16-byte box of their scale codes per row arrive
  // in a code ring filling the rest (its stage size and count depend on the
  // code format: TcArgs::code_stage_bytes, code_stages), which the MMA reads
  // Q from in place
  static constexpr int kStages = DQ ? 5 : kRingMax / kStageBytes > 8 ? 8 : kRingMax / kStageBytes;
  static constexpr int kRingBytes = DQ ? kStages * kABytes : kStages * kStageBytes;
  static constexpr int kCodeRingBytes = DQ ? kRingMax - kRingBytes : 0;
  static_assert(kCodeRingBytes % 1024 == 0, "code stages start on 1024-byte boundaries");
  // the last tile's epilogue stages C in the idle ring: 32 KB per epilogue warp
  // quarter (eight 4 KB buffers a warp, or four for each of two), one per
  // 32-column block of the tile
  static constexpr int kRingBufs = 32 / kEpiWarps;
  static constexpr bool kRingStagesC = kRingBytes >= 4 * 8 * 32 * 128;
  static_assert(DQ || kRingStagesC, "ring too small to stage a tile of C");
  static constexpr int kTmemCols = 2 * BN;       // two fp32 accumulators of BN columns
  // layout: [alignment slack][ring][code ring][control block, padded to 1 KB][staging]
  static constexpr size_t kSmemBytes = 1024 + kRingBytes + kCodeRingBytes + 1024 + kStagingBytes;
};

struct TcCtrl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint64_t c_full[8][2];  // per epilogue warp and staging buffer: a block of old C has landed
  uint64_t code_full[16];   // DQ: a code stage's Q tile, codes and scale codes have landed
  uint64_t code_empty[16];  // DQ: the MMA has read a code stage's Q tile (the converters its codes before)
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t last;
};
static_assert(sizeof(TcCtrl) <= 1024, "control block");

// Swizzle atoms of an MN-major operand: 64 elements along M or N (128 bytes)
// by 64 k-rows; atoms follow each other along M / N.
constexpr uint32_t kMnAtomBytes = 64 * 128;

__device__ __forceinline__ bool wait_bounded_raw(uint32_t bar, uint32_t parity, TcCtrl* ctrl, int32_t* status,
                                                 uint64_t limit_ns, int role, int which, bool honor_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  volatile uint32_t* abort_flag = &ctrl->abort;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      atomicCAS(status, 0, kStatusTimeout | (role << 8) | (which << 12));
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, TcCtrl* ctrl,
                                             const TcArgs& a, int role, int which,
                                             bool honor_abort) {
  return wait_bounded_raw(bar, parity, ctrl, a.status, a.wait_limit_ns, role, which, honor_abort);
}

// Lane 0 of a converged warp waits; the whole warp gets the outcome, so the
// warp's control flow stays uniform (the issuing roles run as whole warps and
// elect one lane to issue, which keeps their operands warp-uniform).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, TcCtrl* ctrl,
                                          const TcArgs& a, int role, int which, bool honor_abort) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, ctrl, a, role, which, honor_abort) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ------------------------------------------------------------------ epilogue --

// The epilogue's view of C, copied out of the kernel parameters into registers
// once per CTA.  (Reached through a pointer to the parameters instead, every
// field would be reloaded after each global store, which the compiler must
// assume may alias it: that made a warp's scalar store cost ~150 cycles.)
struct COut {
  void* C;
  int64_t si, sj;    // element strides of C along I and J
  int32_t I, J;
  int32_t type;      // CType
  float beta;
  bool vec;          // c_sj == 1 and rows 16-byte aligned: 16-byte stores
  int32_t tma;       // kBulkNone, kBulkRows or kBulkTransposed
  bool has_ops;      // any fused bias / activation / output scale
  bool blend_load;   // beta != 0 with bulk row stores: old C arrives by tensor loads
  EpiOps ops;
};

__device__ __forceinline__ COut make_cout(const TcArgs& a) {
  COut o;
  o.C = a.C;
  o.si = a.c_si;
  o.sj = a.c_sj;
  o.I = a.I;
  o.J = a.J;
  o.type = a.c_type;
  o.beta = a.beta;
  o.vec = a.vec_store != 0;
  o.tma = a.tma_store;
  o.ops = a.ops;
  o.has_ops = a.ops.any();
  o.blend_load = a.beta != 0.0f && a.tma_store == kBulkRows;
  return o;
}

__device__ __forceinline__ float load_c(const COut& c, int64_t off) {
  if (c.type == kCF32) return static_cast<const float*>(c.C)[off];
  if (c.type == kCBF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(c.C)[off]);
  if (c.type == kCE4M3) return from_e4m3(static_cast<const uint8_t*>(c.C)[off]);
  return __half2float(static_cast<const __half*>(c.C)[off]);
}

__device__ __forceinline__ void store_c(const COut& c, int64_t off, float v) {
  if (c.type == kCF32)
    static_cast<float*>(c.C)[off] = v;
  else if (c.type == kCBF16)
    static_cast<__nv_bfloat16*>(c.C)[off] = __float2bfloat16_rn(v);
  else if (c.type == kCE4M3)
    static_cast<uint8_t*>(c.C)[off] = to_e4m3(v);
  else
    static_cast<__half*>(c.C)[off] = __float2half_rn(v);
}

__device__ __forceinline__ uint32_t pack2(int32_t type, float lo, float hi) {
  if (type == kCBF16) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
  }
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ float2 unpack2(int32_t type, uint32_t bits) {
  if (type == kCBF16) return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&bits));
  return __half22float2(*reinterpret_cast<__half2*>(&bits));
}

// Write ops(v + beta * C) for row i, columns j0 .. j0 + 31 of D (v already
// holds alpha * D).
__device__ __forceinline__ void store_chunk(const COut& c, int i, int j0, const float (&v)[32]) {
  if (i >= c.I) return;
  const bool blend = c.beta != 0.0f;
  if (c.vec && j0 + 32 <= c.J) {
    const int64_t base = static_cast<int64_t>(i) * c.si + j0;
    if (c.type == kCE4M3) {  // written only (beta == 0): 32 bytes as two 16-byte stores
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t b = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float z = c.has_ops ? apply_ops(c.ops, v[4 * q + t], i, j0 + 4 * q + t) : v[4 * q + t];
          b |= static_cast<uint32_t>(to_e4m3(z)) << (8 * t);
        }
        w[q] = b;
      }
      uint4* p = reinterpret_cast<uint4*>(static_cast<uint8_t*>(c.C) + base);
      p[0] = make_uint4(w[0], w[1], w[2], w[3]);
      p[1] = make_uint4(w[4], w[5], w[6], w[7]);
      return;
    }
    if (c.type == kCF32) {
      float4* p = reinterpret_cast<float4*>(static_cast<float*>(c.C) + base);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 o = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        if (blend) {
          const float4 x = p[q];
          o.x += c.beta * x.x; o.y += c.beta * x.y; o.z += c.beta * x.z; o.w += c.beta * x.w;
        }
        if (c.has_ops) {
          const int j = j0 + 4 * q;
          o.x = apply_ops(c.ops, o.x, i, j);
          o.y = apply_ops(c.ops, o.y, i, j + 1);
          o.z = apply_ops(c.ops, o.z, i, j + 2);
          o.w = apply_ops(c.ops, o.w, i, j + 3);
        }
        p[q] = o;
      }
    } else {
      uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(c.C) + base);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) o[t] = v[8 * q + t];
        if (blend) {
          const uint4 x = p[q];
          const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float2 f = unpack2(c.type, xw[t]);
            o[2 * t] += c.beta * f.x;
            o[2 * t + 1] += c.beta * f.y;
          }
        }
        if (c.has_ops) {
#pragma unroll
          for (int t = 0; t < 8; ++t) o[t] = apply_ops(c.ops, o[t], i, j0 + 8 * q + t);
        }
        p[q] = make_uint4(pack2(c.type, o[0], o[1]), pack2(c.type, o[2], o[3]), pack2(c.type, o[4], o[5]),
                          pack2(c.type, o[6], o[7]));
      }
    }
    return;
  }
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const int j = j0 + t;
    if (j < c.J) {
      const int64_t off = static_cast<int64_t>(i) * c.si + static_cast<int64_t>(j) * c.sj;
      float o = v[t];
      if (blend) o += c.beta * load_c(c, off);
      if (c.has_ops) o = apply_ops(c.ops, o, i, j);
      store_c(c, off, o);
    }
  }
}

// The fused operations on a row piece v[0..31] = columns j0 .. j0 + 31 of row i
// (nvalid of them inside C).  Each operation is its own loop behind a branch
// that is uniform across the warp, and everything stays in registers: local
// memory or extra L1 traffic would compete with the shared-memory port that
// feeds the tensor core.  The bias along J comes in as one coalesced load per
// warp (lane t holds bias[j0 + t]) and is broadcast by shuffles.
__device__ __forceinline__ void apply_ops32(const EpiOps& ops, float (&v)[32], int lane, int64_t i, int64_t j0,
                                            int nvalid) {
  if (ops.bias) {
    if (ops.bias_on_i) {
      const float b = __ldg(ops.bias + i);
#pragma unroll
      for (int t = 0; t < 32; ++t) v[t] += b;
    } else {
      const float mine = lane < nvalid ? __ldg(ops.bias + j0 + lane) : 0.0f;
#pragma unroll
      for (int t = 0; t < 32; ++t) v[t] += __shfl_sync(0xffffffffu, mine, t);
    }
  }
  if (ops.act == kActRelu) {
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = v[t] > 0.0f ? v[t] : 0.0f;
  } else if (ops.act == kActGelu) {
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = 0.5f * v[t] * (1.0f + erff(v[t] * 0.70710678118654752f));
  }
  if (ops.out_scale != 1.0f) {
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] *= ops.out_scale;
  }
}

// One epilogue warp's output path.  The warp owns 32 rows of the tile (I) and
// produces them 32 columns (J) at a time.
//  * kBulkRows: each thread's 32 values go into its row of a 128-byte-swizzled
//    32 x 128-byte staging buffer, which leaves as one bulk tensor store.
//  * kBulkTransposed (swapped problems, where C is J x I in memory): the warp's
//    32 x 32 block is written transposed, one value per thread per memory row,
//    so that the store's box is 32 rows of C by 32 contiguous elements.
//  * kBulkNone: store_chunk writes the values directly.
// Staging buffers are 4 KB.  A warp normally alternates between two, waiting
// before reuse until the store that last read a buffer has read it; for a
// CTA's last tile (use_ring) the idle operand ring provides eight per warp, so
// every store of the tile is in flight at once.
constexpr uint32_t kStagingBuf = 32 * 128;

struct EpiOut {
  COut c;
  const CUtensorMap* map_c;
  uint32_t staging;  // this warp's buffers (shared address, 1024-byte aligned)
  int lane;
  int y0;            // first row of the warp's 32 rows (I)
  int z;             // batch of the current tile (bulk stores)
  void* c0;          // C of batch 0; c.C points at the current tile's batch
  int nstore;        // bulk stores issued from the current buffers
  bool ring;         // buffers in the operand ring: no reuse, no waits
  // beta != 0 with bulk stores: the old C of each 32-row block is loaded by the
  // copy engine into the staging buffer it will leave from, one block ahead
  uint32_t cbar;     // this warp's two mbarriers (buffer 0, buffer 1: 8 bytes apart)
  uint32_t cphase;   // bit b: parity of buffer b's next load
  uint32_t pending;  // bit b: a load into buffer b not yet waited for
  int jstart;        // first column of the current tile
  int jend;          // first column past the current tile
  TcCtrl* ctrl;
  int32_t* status;
  uint64_t wait_ns;
  // fp32 C whose rows start off 16-byte boundaries, in row classes
  const CMaps* cmaps;
  int classes;       // P (0: per-row copies instead)
  float cy[4];       // this thread's row: the previous block's last four values

  __device__ __forceinline__ void use_ring(uint32_t base) {
    staging = base;
    nstore = 0;
    ring = true;
  }

  __device__ __forceinline__ uint32_t buffer(bool fresh) {
    const uint32_t buf = staging + static_cast<uint32_t>((ring ? nstore : (nstore & 1)) * kStagingBuf);
    if (fresh && !ring) {
      if (lane == 0) bulk_wait_group_read<1>();  // the store that last read this buffer is done
      __syncwarp();
    }
    return buf;
  }

  __device__ __forceinline__ void issue(uint32_t buf, int x, int y) {  // at batch z
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(map_c, buf, x, y, z);
      bulk_commit_group();
    }
    __syncwarp();
    ++nstore;
  }

  // Stage the warp's 32 x 32 block, row `lane` from this thread, in `buf`:
  // fp32, 128-byte rows whose 16-byte pieces are swizzled by row (piece k of
  // row r at k ^ (r & 7)), so that neither these row writes nor the reads of
  // one piece from 8 consecutive rows meet bank conflicts.
  __device__ __forceinline__ void stage(uint32_t buf, const float (&v)[32]) {
    const uint32_t row = buf + static_cast<uint32_t>(lane * 128);
    const uint32_t sw = static_cast<uint32_t>(lane & 7);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      st_shared_v4(row + ((k ^ sw) << 4), __float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]),
                   __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
    __syncwarp();
  }

  // Old C for the blend: the copy engine loads the block at column x of the
  // warp's 32 rows into staging buffer `slot` (the block's own bulk store will
  // leave from it), once the store that last read that buffer is done.
  __device__ __forceinline__ void load_block(int slot, int x) {
    if (lane == 0) {
      bulk_wait_group_read<0>();
      const uint32_t bar = cbar + static_cast<uint32_t>(slot * 8);
      mbar_arrive_expect_tx(bar, kStagingBuf);
      tma_load_3d(staging + static_cast<uint32_t>(slot * kStagingBuf), map_c, bar, x, y0, z);
    }
    pending |= 1u << slot;
    __syncwarp();
  }

  // Wait (bounded) until buffer `slot`'s load has landed.
  __device__ __forceinline__ void wait_block(int slot, bool honor_abort) {
    int ok = 1;
    if (lane == 0)
      ok = wait_bounded_raw(cbar + static_cast<uint32_t>(slot * 8), (cphase >> slot) & 1u, ctrl, status, wait_ns,
                            kRoleEpilogue, kBarCLoad, honor_abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {  // a load that gave up may still land: its phase is not consumed
      cphase ^= 1u << slot;
      pending &= ~(1u << slot);
    }
  }

  // A tile whose columns run from jt to jend (exclusive) begins: with beta !=
  // 0 and bulk stores, its first block of old C starts loading.
  __device__ __forceinline__ void begin_tile(int jt, int jend_) {
    jstart = jt;
    jend = jend_;
    if (c.blend_load) load_block(nstore & 1, jt);
  }

  // fp32 C whose rows start off 16-byte boundaries, in P row classes (CMaps):
  // the rows of class r start s_r values past a boundary, so the block's 32
  // columns j .. j + 31 of such a row, shifted right by s_r behind the s_r last
  // values of the previous block, fill whole 16-byte pieces from column j -
  // s_r.  Each thread writes that shifted row into its class's part of a
  // 128-byte-swizzled staging buffer, and one tensor store per class writes
  // the block (P stores where per-row copies took 32).  A tile's first block
  // cannot write the piece it shares with the tile to its left: its store
  // starts one piece later (28-column boxes, unswizzled 112-byte rows) and the
  // first 4 - s_r values go out by plain stores, as do the values after a
  // tile's last block.  The classes' tensors end at their last whole 16-byte
  // piece before column N (a store would write a partial last piece whole);
  // the few values past it go out by plain stores too.
  __device__ __forceinline__ void put_row_class(int i, int j, const float (&v)[32]) {
    const int jv = c.J < jend ? c.J : jend;  // first column past the tile's columns inside C
    if (j >= jv) return;                     // (the same for the whole warp)
    const int ncols = jv - j < 32 ? jv - j : 32;
    const bool first = j == jstart;
    const bool last = j + 32 >= jv;
    const int P = classes;
    const int rows = 32 / P;                 // a class's rows in the warp's 32
    const int cls = lane % P;
    const int br = lane / P;                 // this thread's row in its class's part of the buffer
    char* rowp = static_cast<char*>(c.C) + (static_cast<int64_t>(i) * c.si + j) * 4;
    const int sh = static_cast<int>((reinterpret_cast<uintptr_t>(rowp) & 15u) >> 2);
    const uint32_t buf = buffer(true);
    const uint32_t sub = buf + static_cast<uint32_t>(cls * rows * 128);  // 1024-byte aligned (P <= 4)
    // The P threads of one 8-thread store phase that share a buffer row index
    // (one per class) write their pieces in an order rotated by their class,
    // so that they reach different banks: piece (k + cls) mod n at step k.
    if (first) {
      // v[4 - sh .. 31 - sh]: columns j + 4 - sh .. j + 31 - sh, from the block's second piece on
      const uint32_t row = sub + static_cast<uint32_t>(br * 112);
      float o[7][4];
#pragma unroll
      for (int k = 0; k < 7; ++k)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = 4 * k + u;
          float x = v[e + 4];
#pragma unroll
          for (int t = 1; t < 4; ++t)
            if (t == sh) x = v[e + 4 - t];
          o[k][u] = x;
        }
      float t1[7][4], t2[7][4];  // rotated left by cls (mod 7): by 1, then by 2
#pragma unroll
      for (int k = 0; k < 7; ++k)
#pragma unroll
        for (int u = 0; u < 4; ++u) t1[k][u] = (cls & 1) ? o[(k + 1) % 7][u] : o[k][u];
#pragma unroll
      for (int k = 0; k < 7; ++k)
#pragma unroll
        for (int u = 0; u < 4; ++u) t2[k][u] = (cls & 2) ? t1[(k + 2) % 7][u] : t1[k][u];
#pragma unroll
      for (int k = 0; k < 7; ++k) {
        const int q = (k + cls) % 7;
        st_shared_v4(row + static_cast<uint32_t>(q * 16), __float_as_uint(t2[k][0]), __float_as_uint(t2[k][1]),
                     __float_as_uint(t2[k][2]), __float_as_uint(t2[k][3]));
      }
    } else {
      // [the previous block's last sh values | v[0 .. 31 - sh]]: columns j - sh .. j + 31 - sh
      const uint32_t row = sub + static_cast<uint32_t>(br * 128);
      const uint32_t sw = static_cast<uint32_t>(br & 7);
      float o[8][4];
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = 4 * k + u;
          float x = v[e];
#pragma unroll
          for (int t = 1; t < 4; ++t)
            if (t == sh) x = e < t ? cy[4 - t + (e < t ? e : 0)] : v[e - t < 0 ? 0 : e - t];
          o[k][u] = x;
        }
      float t1[8][4], t2[8][4];  // rotated left by cls (mod 8): by 1, then by 2
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int u = 0; u < 4; ++u) t1[k][u] = (cls & 1) ? o[(k + 1) & 7][u] : o[k][u];
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int u = 0; u < 4; ++u) t2[k][u] = (cls & 2) ? t1[(k + 2) & 7][u] : t1[k][u];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t q = static_cast<uint32_t>((k + cls) & 7);
        st_shared_v4(row + ((q ^ sw) << 4), __float_as_uint(t2[k][0]), __float_as_uint(t2[k][1]),
                     __float_as_uint(t2[k][2]), __float_as_uint(t2[k][3]));
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) cy[t] = v[28 + t];
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      for (int r = 0; r < P; ++r)
        tma_store_3d(&cmaps->m[first ? 4 + r : r], buf + static_cast<uint32_t>(r * rows * 128), first ? j + 4 : j,
                     y0 / P, 0);
      bulk_commit_group();
    }
    __syncwarp();
    ++nstore;
    // plain stores: the first block's values before its box, after the tile's
    // last block the values past its box, and the values past the class
    // tensor's last whole 16-byte piece (columns jcut and on)
    // (jcut >= J - 3: an interior block with no values from column J - 3 on stores nothing)
    if ((first || last || j + 32 > c.J - 3) && i < c.I) {
      const int jcut = ((c.J + sh) & ~3) - sh;
      const int64_t off = static_cast<int64_t>(i) * c.si + j;
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if (t < ncols && ((first && t < 4 - sh) || j + t >= jcut || (last && t >= 32 - sh)))
          static_cast<float*>(c.C)[off + t] = v[t];
    }
  }

  // Rows of C that bulk tensor stores cannot write (not 16-byte aligned, or
  // ending inside a 16-byte piece): each thread writes its own row of the
  // block.  Its 32 values go into a slot of shared memory shifted by the row's
  // misalignment (sh elements), so that the slot's first byte stands for the
  // 16-byte boundary at or before the row's first value; one 1-D bulk copy
  // then writes the row's whole 16-byte pieces.  The piece that the block's
  // last values share with the next block of the same row stays in the slot's
  // last piece and leaves with the next block's copy.  At the tile's first and
  // last columns, whose neighbouring values belong to other tiles, the values
  // of the partial pieces are written by plain stores.  Slots of 144 (fp32)
  // or 80 (16-bit) bytes put the 16-byte stores of eight consecutive threads
  // on distinct banks.  Nothing outside the tile's columns inside C is written.
  template <int ESZ>
  __device__ __forceinline__ void put_row_copy(int i, int j, const float (&v)[32]) {
    constexpr int kPer = 16 / ESZ;              // values per 16-byte piece
    constexpr int kPieces = 32 / kPer + 1;      // the block's pieces and the one it may share
    constexpr uint32_t kSlot = kPieces * 16;
    const int jv = c.J < jend ? c.J : jend;     // first column past the tile's columns inside C
    if (j >= jv || i >= c.I) return;
    const int ncols = jv - j < 32 ? jv - j : 32;
    char* rowp = static_cast<char*>(c.C) + (static_cast<int64_t>(i) * c.si + j) * ESZ;
    const int mbytes = static_cast<int>(reinterpret_cast<uintptr_t>(rowp) & 15u);
    const int sh = mbytes / ESZ;
    const bool first = j == jstart;
    const bool last = j + 32 >= jv;
    const uint32_t slot = staging + static_cast<uint32_t>(lane) * kSlot;
    bulk_wait_group_read<0>();  // this thread's previous copy has read the slot
    float carry[kPer];          // the values the previous block left in the shared piece
    {
      const float4 q = ld_shared_v4_f32(slot + (kPieces - 1) * 16);
      if constexpr (ESZ == 4) {
        carry[0] = q.x; carry[1] = q.y; carry[2] = q.z; carry[3] = q.w;
      } else {
        const uint32_t w[4] = {__float_as_uint(q.x), __float_as_uint(q.y), __float_as_uint(q.z), __float_as_uint(q.w)};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = unpack2(c.type, w[t]);
          carry[2 * t] = f.x;
          carry[2 * t + 1] = f.y;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPieces; ++k) {
      float o[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = k * kPer + u;  // slot position: carry[e] before the shift, v[e - sh] after it
        float x = 0.0f;
#pragma unroll
        for (int t = 0; t < kPer; ++t)
          if (t == sh) x = e < t ? carry[e < kPer ? e : 0] : (e - t < 32 ? v[e - t < 32 ? e - t : 0] : 0.0f);
        o[u] = x;
      }
      if constexpr (ESZ == 4)
        st_shared_v4(slot + k * 16, __float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                     __float_as_uint(o[3]));
      else
        st_shared_v4(slot + k * 16, pack2(c.type, o[0], o[1]), pack2(c.type, o[2], o[3]), pack2(c.type, o[4], o[5]),
                     pack2(c.type, o[6], o[7]));
    }
    fence_proxy_async_smem();
    char* base = rowp - mbytes;  // the slot's first byte stands here
    char* lo = base + ((first && sh > 0) ? 16 : 0);
    char* hi = reinterpret_cast<char*>(reinterpret_cast<uintptr_t>(rowp + ncols * ESZ) & ~uintptr_t{15});
    if (hi > lo) {
      bulk_copy_s2g(lo, slot + static_cast<uint32_t>(lo - base), static_cast<uint32_t>(hi - lo));
      bulk_commit_group();
    }
    // plain stores: the values before the copy in the tile's first block, and
    // after the tile's last block the values past the copy
    const int head = (first && sh > 0) ? (kPer - sh < ncols ? kPer - sh : ncols) : 0;
    const int past = static_cast<int>((hi - rowp) / ESZ);
    const int tail = past > head ? past : head;
    const int64_t off = static_cast<int64_t>(i) * c.si + j;
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (t < head || (last && t >= tail && t < ncols)) store_c(c, off + t, v[t]);
  }

  // No load may still be writing shared memory when the warp leaves.
  __device__ __forceinline__ void drain_loads() {
    for (int b = 0; b < 2; ++b)
      if (pending & (1u << b)) wait_block(b, false);
  }

  // Bulk row stores with beta != 0: this block's old C is in its staging
  // buffer (loaded one block ahead); each thread reads its row's values, adds
  // beta times them to its own, applies the fused operations and writes the
  // row back in place, and the block leaves through one bulk tensor store.
  // Every byte of C crosses the shared-memory port four times (load, read,
  // write, store), against two plus a global load and store through L1 when
  // the blend read and wrote C directly.
  __device__ __forceinline__ void put_blend(int i, int j, const float (&vin)[32], int half) {
    const bool wide = c.type == kCF32;
    const int slot = nstore & 1;
    const uint32_t buf = staging + static_cast<uint32_t>(slot * kStagingBuf);
    if (wide || half == 0) {
      const int jn = j + (wide ? 32 : 64);
      if (jn < jend) load_block(slot ^ 1, jn);
      wait_block(slot, false);
    }
    float v[32];
    const uint32_t row = buf + static_cast<uint32_t>(lane * 128);
    const uint32_t sw = static_cast<uint32_t>(lane & 7);  // 128-byte swizzle of 16-byte pieces
    if (wide) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 o = ld_shared_v4_f32(row + ((k ^ sw) << 4));
        v[4 * k] = vin[4 * k] + c.beta * o.x;
        v[4 * k + 1] = vin[4 * k + 1] + c.beta * o.y;
        v[4 * k + 2] = vin[4 * k + 2] + c.beta * o.z;
        v[4 * k + 3] = vin[4 * k + 3] + c.beta * o.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 o = ld_shared_v4_f32(row + (((4 * half + k) ^ sw) << 4));
        const uint32_t w[4] = {__float_as_uint(o.x), __float_as_uint(o.y), __float_as_uint(o.z), __float_as_uint(o.w)};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = unpack2(c.type, w[t]);
          v[8 * k + 2 * t] = vin[8 * k + 2 * t] + c.beta * f.x;
          v[8 * k + 2 * t + 1] = vin[8 * k + 2 * t + 1] + c.beta * f.y;
        }
      }
    }
    // (the whole warp: the bias shuffle needs every lane; rows past I compute
    // values the clipped store drops)
    if (c.has_ops) apply_ops32(c.ops, v, lane, i < c.I ? i : c.I - 1, j, c.J - j < 32 ? c.J - j : 32);
    if (wide) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_shared_v4(row + ((k ^ sw) << 4), __float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]),
                     __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_shared_v4(row + (((4 * half + k) ^ sw) << 4), pack2(c.type, v[8 * k], v[8 * k + 1]),
                     pack2(c.type, v[8 * k + 2], v[8 * k + 3]), pack2(c.type, v[8 * k + 4], v[8 * k + 5]),
                     pack2(c.type, v[8 * k + 6], v[8 * k + 7]));
    }
    if (wide || half == 1) issue(buf, wide ? j : j - 32, y0);
  }

  // Direct stores when the rows of C are contiguous (unswapped problems): the
  // warp's block goes through its staging buffer and comes back out along the
  // rows of C, so that each global access of the warp covers whole row pieces:
  // 16 bytes per lane where rows are 16-byte aligned and the block is whole in
  // J, else one element per lane (32 consecutive elements of one row).  The
  // old values for beta * C are read the same way, all of a block's loads
  // issued (after the block is staged) before its first store.  (Written from each thread's own row, a
  // warp's accesses fell into 32 rows and every load of C waited for the store
  // before it: 4096^3 took 1.6 times as long with beta != 0.)
  __device__ __forceinline__ void put_rows(int j, const float (&v)[32]) {
    const uint32_t buf = staging;
    const int ncols = c.J - j < 32 ? c.J - j : 32;
    const bool whole = ncols == 32 && c.vec;
    const bool blend = c.beta != 0.0f;
    if (whole && c.type == kCF32) {
      const int g = lane & 7;  // columns 4g .. 4g + 3 of rows 4p + lane / 8
      stage(buf, v);
      float4 x[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const int i = y0 + 4 * p + (lane >> 3);
        x[p] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (blend && i < c.I)
          x[p] = *reinterpret_cast<const float4*>(static_cast<const float*>(c.C) + static_cast<int64_t>(i) * c.si +
                                                  j + 4 * g);
      }
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const int r = 4 * p + (lane >> 3);
        const int i = y0 + r;
        if (i < c.I) {
          float4 o = ld_shared_v4_f32(buf + static_cast<uint32_t>(r * 128 + ((g ^ (r & 7)) << 4)));
          if (blend) {
            o.x += c.beta * x[p].x; o.y += c.beta * x[p].y; o.z += c.beta * x[p].z; o.w += c.beta * x[p].w;
          }
          if (c.has_ops) {
            const int jj = j + 4 * g;
            o.x = apply_ops(c.ops, o.x, i, jj);
            o.y = apply_ops(c.ops, o.y, i, jj + 1);
            o.z = apply_ops(c.ops, o.z, i, jj + 2);
            o.w = apply_ops(c.ops, o.w, i, jj + 3);
          }
          *reinterpret_cast<float4*>(static_cast<float*>(c.C) + static_cast<int64_t>(i) * c.si + j + 4 * g) = o;
        }
      }
    } else if (whole && c.type != kCE4M3) {  // 16-bit C
      const int g = lane & 3;  // columns 8g .. 8g + 7 (staged pieces 2g, 2g + 1) of rows 8p + lane / 4
      stage(buf, v);
      uint4 x[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int i = y0 + 8 * p + (lane >> 2);
        x[p] = make_uint4(0u, 0u, 0u, 0u);
        if (blend && i < c.I)
          x[p] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(c.C) + static_cast<int64_t>(i) * c.si +
                                                 j + 8 * g);
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int r = 8 * p + (lane >> 2);
        const int i = y0 + r;
        if (i < c.I) {
          const float4 a0 = ld_shared_v4_f32(buf + static_cast<uint32_t>(r * 128 + (((2 * g) ^ (r & 7)) << 4)));
          const float4 a1 = ld_shared_v4_f32(buf + static_cast<uint32_t>(r * 128 + (((2 * g + 1) ^ (r & 7)) << 4)));
          float o[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          if (blend) {
            const uint32_t xw[4] = {x[p].x, x[p].y, x[p].z, x[p].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float2 f = unpack2(c.type, xw[t]);
              o[2 * t] += c.beta * f.x;
              o[2 * t + 1] += c.beta * f.y;
            }
          }
          if (c.has_ops) {
#pragma unroll
            for (int t = 0; t < 8; ++t) o[t] = apply_ops(c.ops, o[t], i, j + 8 * g + t);
          }
          *reinterpret_cast<uint4*>(static_cast<uint16_t*>(c.C) + static_cast<int64_t>(i) * c.si + j + 8 * g) =
              make_uint4(pack2(c.type, o[0], o[1]), pack2(c.type, o[2], o[3]), pack2(c.type, o[4], o[5]),
                         pack2(c.type, o[6], o[7]));
        }
      }
    } else if (whole) {  // 8-bit C (written only: beta == 0)
      const int g = lane & 1;  // columns 16g .. 16g + 15 (staged pieces 4g .. 4g + 3) of rows 16p + lane / 2
      stage(buf, v);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int r = 16 * p + (lane >> 1);
        const int i = y0 + r;
        if (i < c.I) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 f = ld_shared_v4_f32(buf + static_cast<uint32_t>(r * 128 + (((4 * g + k) ^ (r & 7)) << 4)));
            float o[4] = {f.x, f.y, f.z, f.w};
            uint32_t b = 0;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float z = c.has_ops ? apply_ops(c.ops, o[t], i, j + 16 * g + 4 * k + t) : o[t];
              b |= static_cast<uint32_t>(to_e4m3(z)) << (8 * t);
            }
            w[k] = b;
          }
          *reinterpret_cast<uint4*>(static_cast<uint8_t*>(c.C) + static_cast<int64_t>(i) * c.si + j + 16 * g) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    } else {  // misaligned rows, or the block's last columns lie past J
      // (eight rows at a time: the old values of eight rows in flight together)
      stage(buf, v);
#pragma unroll 1
      for (int r0 = 0; r0 < 32; r0 += 8) {
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int i = y0 + r0 + t;
          x[t] = 0.0f;
          if (blend && i < c.I && lane < ncols) x[t] = load_c(c, static_cast<int64_t>(i) * c.si + j + lane);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int r = r0 + t;
          const int i = y0 + r;
          if (i < c.I && lane < ncols) {
            float o = ld_shared_f32(buf + static_cast<uint32_t>(r * 128 + ((((lane >> 2) ^ (r & 7)) << 4) |
                                                                            ((lane & 3) << 2))));
            if (blend) o += c.beta * x[t];
            if (c.has_ops) o = apply_ops(c.ops, o, i, j + lane);
            store_c(c, static_cast<int64_t>(i) * c.si + j + lane, o);
          }
        }
      }
    }
    __syncwarp();  // every lane has read the block before the next one is staged
  }

  __device__ __forceinline__ void put(int i, int j, const float (&vin)[32], int half) {
    if (c.tma == kBulkNone) {
      if (c.sj == 1)
        put_rows(j, vin);
      else  // swapped problems: consecutive lanes already hold consecutive elements of C
        store_chunk(c, i, j, vin);
      return;
    }
    if (c.blend_load) {
      put_blend(i, j, vin, half);
      return;
    }
    // the other bulk paths run with beta == 0: the fused operations apply to
    // alpha * D, inside C only (the bias holds no value for the clipped edge of a tile)
    float v[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) v[t] = vin[t];
    // (the whole warp enters: the bias shuffle needs every lane; rows past I
    // compute values the clipped store drops)
    if (c.has_ops) apply_ops32(c.ops, v, lane, i < c.I ? i : c.I - 1, j, c.J - j < 32 ? c.J - j : 32);
    if (c.tma == kBulkRowCopies) {
      if (classes > 0)
        put_row_class(i, j, v);
      else if (c.type == kCF32)
        put_row_copy<4>(i, j, v);
      else
        put_row_copy<2>(i, j, v);
      return;
    }
    if (c.tma == kBulkTransposed) {
      const uint32_t buf = buffer(true);
      if (c.type == kCF32) {
        // memory row t holds 32 fp32 of I: 16-byte piece (lane / 4) sits at (lane / 4) ^ (t & 7)
#pragma unroll
        for (int t = 0; t < 32; ++t)
          st_shared_b32(buf + static_cast<uint32_t>(t * 128 + ((((lane >> 2) ^ (t & 7)) << 4) | ((lane & 3) << 2))),
                        __float_as_uint(v[t]));
      } else {
        // 16-bit: unswizzled 64-byte rows
#pragma unroll
        for (int t = 0; t < 32; ++t)
          st_shared_b16(buf + static_cast<uint32_t>(t * 64 + lane * 2),
                        static_cast<uint16_t>(pack2(c.type, v[t], 0.0f) & 0xFFFFu));
      }
      issue(buf, y0, j);
      return;
    }
    // 16-bit C: two 32-column pieces fill one 128-byte row (half 0, then half 1)
    const bool wide = c.type == kCF32;
    const uint32_t buf = buffer(wide || half == 0);
    const uint32_t row = buf + static_cast<uint32_t>(lane * 128);
    const uint32_t sw = static_cast<uint32_t>(lane & 7);  // 128-byte swizzle of 16-byte pieces
    if (wide) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_shared_v4(row + ((k ^ sw) << 4), __float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]),
                     __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_shared_v4(row + (((4 * half + k) ^ sw) << 4), pack2(c.type, v[8 * k], v[8 * k + 1]),
                     pack2(c.type, v[8 * k + 2], v[8 * k + 3]), pack2(c.type, v[8 * k + 4], v[8 * k + 5]),
                     pack2(c.type, v[8 * k + 6], v[8 * k + 7]));
    }
    if (wide || half == 1) issue(buf, wide ? j : j - 32, y0);
  }

  // Before the CTA exits, every bulk store must have read its staging buffer;
  // the global writes complete with the grid, like any other store.
  __device__ __forceinline__ void finish() {
    drain_loads();
    if (c.tma == kBulkRowCopies && classes == 0) {
      bulk_wait_group_read<0>();  // every thread issued copies of its own row
    } else if (c.tma != kBulkNone) {
      if (lane == 0) bulk_wait_group_read<0>();
    }
    __syncwarp();
  }
};

// ----------------------------------------------------------------- the roles --

template <int BN, int CG, int EB, int KD, bool DQ, int EW>
__device__ __forceinline__ void producer_role(const CUtensorMap* map_p, const CUtensorMap* map_q,
                                              const CUtensorMap* map_sf, const TcArgs& a, uint8_t* ring_a,
                                              uint8_t* ring_b, uint8_t* code_ring, TcCtrl* ctrl, uint32_t rank,
                                              int first, int stride) {
  using Cfg = TcConfig<BN, CG, DQ, EW>;
  const int q = static_cast<int>(rank);  // rank inside the CTA pair (0: the leader)
  constexpr int kSliceK = slice_k(EB);  // k elements of one 128-byte slice
  // 8- and 32-bit operands are always K-major (the planner admits no other layout)
  const bool p_kmajor = EB != 2 || a.p_kmajor != 0;
  const bool q_kmajor = EB != 2 || a.q_kmajor != 0;
  const int kslices = (a.K + kSliceK - 1) / kSliceK;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t pending = 0, pending_parity = 0;  // copies in flight, per stage
  int nload = 0;
  bool ok = true;
  WorkIter work(a.sched, first, stride);
  Unit w;
  while (ok && work.next(w)) {
    // (grouped GEMMs: the group's rows start further down P)
    const int i0 = (a.sched.groups > 0 ? static_cast<int>(a.group_row[w.tb]) : 0) + w.ti * Cfg::kTileM + q * kBM;
    const int j0 = w.tj * BN + q * Cfg::kQRows;
    const int zp = a.p_bcast ? 0 : w.tb;  // batch coordinate (0 for an operand shared by all batches)
    const int zq = a.q_bcast ? 0 : w.tb;
    // (three-product fp32 GEMM: segment and k-slice within it of the unit's first k-slice)
    int seg_s = 0, seg_in = 0;
    if constexpr (EB == 4) {
      if (a.seg_slices > 0) {
        seg_s = (w.kb0 * KD) / a.seg_slices;
        seg_in = w.kb0 * KD - seg_s * a.seg_slices;
      }
    }
    for (int kb = w.kb0; kb < w.kb1; ++kb) {  // one stage: k-slices kb * kdepth .. + kdepth - 1
      if constexpr (DQ) {
        // The code ring, one k-slice a stage: Q's 16-bit tile (which the MMA
        // reads in place), P's codes and a 16-byte box of their scale codes
        // per row, all counted on code_full; the converter warps fill the ring
        // with P's values.
        if (!warp_wait(smem_u32(&ctrl->code_empty[stage]), phase ^ 1u, ctrl, a, kRoleProducer, kBarEmpty, true)) {
          ok = false;
          break;
        }
        ++nload;
        if (a.drop_load != 0 && blockIdx.x == 0 && nload == a.drop_load) {
          pending &= ~(1u << stage);  // test hook: this stage's barrier is never completed
        } else {
          const uint32_t cbar = smem_u32(&ctrl->code_full[stage]);
          if (elect_one()) {
            mbar_arrive_expect_tx(cbar, Cfg::kBBytes + kBM * a.code_bytes + kBM * 16);
            const uint32_t cs = smem_u32(code_ring + stage * a.code_stage_bytes);
            tma_load_3d(cs, map_q, cbar, kb * slice_k(EB), j0, zq);
            tma_load_3d(cs + Cfg::kBBytes, map_p, cbar, kb * a.code_bytes, i0, 0);
            tma_load_3d(cs + Cfg::kBBytes + kBM * a.code_bytes, map_sf, cbar, (kb * a.spk) & ~15, i0, 0);
          }
          __syncwarp();
          pending |= 1u << stage;
          pending_parity = (pending_parity & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == a.code_stages) {
          stage = 0;
          phase ^= 1u;
        }
        continue;
      }
      if (!warp_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, ctrl, a, kRoleProducer, kBarEmpty,
                     true)) {
        ok = false;
        break;
      }
      ++nload;
      const uint32_t full_local = smem_u32(&ctrl->full[stage]);
      // A pair credits both CTAs' bytes to the leader's barrier, which the MMA waits on.
      const uint32_t full = CG == 2 ? mapa_shared(full_local, 0) : full_local;
      if (a.drop_load != 0 && blockIdx.x == 0 && nload == a.drop_load) {
        pending &= ~(1u << stage);  // test hook: this stage's barrier is never completed
      } else {
        // k-slices of this stage inside K (a ragged K leaves fewer in the last stage)
        const int ks0 = kb * KD;
        const int nks = KD == 1 ? 1 : min(KD, kslices - ks0);
        if (elect_one()) {
          if (q == 0) mbar_arrive_expect_tx(full_local, CG * nks * Cfg::kStageBytes);
          auto load = [&](uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z) {
            if constexpr (CG == 2)
              tma_load_3d_pair(dst, map, full, x, y, z);
            else
              tma_load_3d(dst, map, full, x, y, z);
          };
#pragma unroll
          for (int t = 0; t < KD; ++t) {
            if (t == nks) break;
            const int slot = stage * KD + t;  // ring slot of one k-slice
            const uint32_t sa = smem_u32(ring_a + slot * Cfg::kABytes);
            const uint32_t sb = smem_u32(ring_b + slot * Cfg::kBBytes);
            int k0 = (ks0 + t) * kSliceK;
            int kq = k0;
            if constexpr (EB == 4) {
              // fp32 from three TF32 products: each operand is stored as two
              // segments of seg_slices k-slices, and logical segment s of the
              // GEMM over 3 segments reads stored segment bit s of p_seg / q_seg
              if (a.seg_slices > 0) {
                k0 = (((a.p_seg >> seg_s) & 1) * a.seg_slices + seg_in) * kSliceK;
                kq = (((a.q_seg >> seg_s) & 1) * a.seg_slices + seg_in) * kSliceK;
                if (++seg_in == a.seg_slices) {
                  seg_in = 0;
                  ++seg_s;
                }
              }
            }
            if (p_kmajor) {
              load(sa, map_p, k0, i0, zp);
            } else {
              load(sa, map_p, i0, k0, zp);
              load(sa + kMnAtomBytes, map_p, i0 + 64, k0, zp);
            }
            if (q_kmajor) {
              load(sb, map_q, kq, j0, zq);
            } else {
#pragma unroll
              for (int c = 0; c < Cfg::kQRows / 64; ++c)
                load(sb + c * kMnAtomBytes, map_q, j0 + 64 * c, kq, zq);
            }
          }
        }
        __syncwarp();
        pending |= 1u << stage;
        pending_parity = (pending_parity & ~(1u << stage)) | (phase << stage);
      }
      if (++stage == a.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  // No copy may still be writing shared memory when the CTA exits.  The leader's
  // barrier counts both CTAs' bytes, so the leader's wait covers the pair; a
  // peer CTA is held at the final cluster barrier until the leader has waited.
  if (q == 0 && (threadIdx.x & 31) == 0) {
    const int nstages = DQ ? a.code_stages : Cfg::kStages;
    for (int s = 0; s < nstages; ++s)
      if (pending & (1u << s))
        wait_bounded(smem_u32(DQ ? &ctrl->code_full[s] : &ctrl->full[s]), (pending_parity >> s) & 1u, ctrl, a,
                     kRoleProducer, kBarDrain, false);
  }
  __syncwarp();
}

// DQ kernels: kConvWarps converter warps turn P's block-scaled codes into the
// 16-bit values the MMA reads, stage by stage (the producer's order: the same
// work units and k-blocks, one k-slice a stage).  Warp cw converts rows
// 16 cw .. 16 cw + 15 of the 128-row P tile, two threads a row, each half of
// the row's 64 values, into the ring's 128-byte-swizzled K-major layout
// (16-byte piece p of row r at p ^ (r & 7)), then completes the stage's full
// barrier with one arrival per warp.  (Two warps on each of the SM's four
// schedulers halve each warp's share of a stage: four warps with a whole row
// per thread left the conversion on the critical path, about 20 us of the
// LM head's 65.)
//  * E2M1 codes (two a byte, the even k in the low four bits) with unsigned
//    E4M3 scales per 16 values -> fp16: code and scale as fp16, one fp16
//    product, exact (at most 6 significant bits, inside fp16's range).
//  * E4M3 / E5M2 codes with E8M0 scales (2^(s - 127)) per 32 values -> bf16:
//    code as fp16, then fp32 times the scale, rounded to bf16 (exact inside
//    bf16's range; the dequantising copy kernel rounds the same way).
// Products past K, or past P's rows, come from zero codes the copy engine
// filled in, so they are 0.
template <int BN, int CG>
__device__ __forceinline__ void converter_role(const TcArgs& a, uint8_t* ring_a, uint8_t* code_ring, TcCtrl* ctrl,
                                               int cw, int lane, int first, int stride) {
  using Cfg = TcConfig<BN, CG, true>;
  static_assert(kBM == 16 * kConvWarps, "two threads a row");
  const int r = cw * 16 + (lane >> 1);
  const int h = lane & 1;  // values 32 h .. 32 h + 31 of the row's 64
  const uint32_t sw = static_cast<uint32_t>(r & 7);
  int stage = 0, cstage = 0;  // the P ring and the code ring
  uint32_t phase = 0, cphase = 0;
  bool ok = true;
  WorkIter work(a.sched, first, stride);
  Unit w;
  while (ok && work.next(w)) {
    for (int kb = w.kb0; kb < w.kb1; ++kb) {
      if (!warp_wait(smem_u32(&ctrl->code_full[cstage]), cphase, ctrl, a, kRoleConvert, kBarCodeFull, true) ||
          !warp_wait(smem_u32(&ctrl->empty[stage]), phase ^ 1u, ctrl, a, kRoleConvert, kBarEmpty, true)) {
        ok = false;
        break;
      }
      const uint8_t* cst = code_ring + cstage * a.code_stage_bytes + Cfg::kBBytes;  // past the Q tile
      const uint32_t codes = smem_u32(cst) + static_cast<uint32_t>(r * a.code_bytes + h * (a.code_bytes / 2));
      const uint32_t scales =
          smem_u32(cst + kBM * a.code_bytes) + static_cast<uint32_t>(r * 16 + ((kb * a.spk) & 15));
      const uint32_t dst = smem_u32(ring_a + stage * Cfg::kABytes) + static_cast<uint32_t>(r * 128);
      if (a.dq_fmt == 1) {
        uint32_t wd[4];
        {
          const float4 c0 = ld_shared_v4_f32(codes);
          wd[0] = __float_as_uint(c0.x); wd[1] = __float_as_uint(c0.y); wd[2] = __float_as_uint(c0.z);
          wd[3] = __float_as_uint(c0.w);
        }
        // this half's two unsigned E4M3 scales as fp16 pairs (sign bits cleared)
        const uint32_t sc = ld_shared_u16(scales + 2 * h) & 0x7F7Fu;
        const uint32_t s01 = e4m3x2_to_f16x2(sc);
        const uint32_t sf[2] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232)};
#pragma unroll
        for (int p = 0; p < 4; ++p) {  // values 32 h + 8p .. + 7, scale p / 2 of the half
          const __half2 s2 = *reinterpret_cast<const __half2*>(&sf[p >> 1]);
          uint32_t o[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t hv = e2m1x2_to_f16x2((wd[p] >> (8 * b)) & 0xFFu);
            const __half2 prod = __hmul2(*reinterpret_cast<const __half2*>(&hv), s2);
            o[b] = *reinterpret_cast<const uint32_t*>(&prod);
          }
          st_shared_v4(dst + ((static_cast<uint32_t>(4 * h + p) ^ sw) << 4), o[0], o[1], o[2], o[3]);
        }
      } else {
        const bool e5m2 = a.dq_fmt == 3;
        const uint32_t s = (ld_shared_u16(scales) >> (8 * h)) & 0xFFu;  // the half's one scale
        const float f = s == 255u ? __int_as_float(0x7FC00000)
                                  : s == 0u ? __int_as_float(0x00400000) : __int_as_float(static_cast<int>(s << 23));
        const float4 c0 = ld_shared_v4_f32(codes), c1 = ld_shared_v4_f32(codes + 16);
        const uint32_t wd[8] = {__float_as_uint(c0.x), __float_as_uint(c0.y), __float_as_uint(c0.z),
                                __float_as_uint(c0.w), __float_as_uint(c1.x), __float_as_uint(c1.y),
                                __float_as_uint(c1.z), __float_as_uint(c1.w)};
#pragma unroll
        for (int p = 0; p < 4; ++p) {  // piece 4h + p: words 2p, 2p + 1
          uint32_t o[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t pair = (wd[2 * p + (b >> 1)] >> (16 * (b & 1))) & 0xFFFFu;
            const uint32_t hv = e5m2 ? e5m2x2_to_f16x2(pair) : e4m3x2_to_f16x2(pair);
            const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&hv));
            const __nv_bfloat162 y = __floats2bfloat162_rn(x.x * f, x.y * f);
            o[b] = *reinterpret_cast<const uint32_t*>(&y);
          }
          st_shared_v4(dst + ((static_cast<uint32_t>(4 * h + p) ^ sw) << 4), o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();  // the MMA reads these values through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl->full[stage]));
      if (++stage == a.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++cstage == a.code_stages) {
        cstage = 0;
        cphase ^= 1u;
      }
    }
  }
}

template <int BN, int CG, int EB, int KD, bool DQ, int EW>
__device__ __forceinline__ void mma_role(const TcArgs& a, uint8_t* ring_a, uint8_t* ring_b, uint8_t* code_ring,
                                         TcCtrl* ctrl, uint32_t tmem_base, uint32_t rank, int first,
                                         int stride) {
  using Cfg = TcConfig<BN, CG, DQ, EW>;
  int cstage = 0;  // DQ: the code ring stage holding the k-slice's Q tile
  constexpr int kSliceK = slice_k(EB);  // k elements of one 128-byte slice
  // 8- and 32-bit operands are always K-major (the planner admits no other layout)
  const bool p_kmajor = EB != 2 || a.p_kmajor != 0;
  const bool q_kmajor = EB != 2 || a.q_kmajor != 0;
  const int kslices = (a.K + kSliceK - 1) / kSliceK;
  int stage = 0;
  uint32_t phase = 0;
  int it = 0;
  bool ok = true;
  // A stage is freed, and the accumulator handed to the epilogues, in both
  // CTAs of a pair (each CTA's copies land in its own shared memory and each
  // CTA's epilogue reads its own rows of the accumulator).
  auto commit_both = [&](uint32_t bar) {
    if constexpr (CG == 2)
      mma_commit_pair(bar, 0x3);
    else
      mma_commit<1>(bar);
  };
  WorkIter work(a.sched, first, stride);
  Unit w;
  for (; ok && work.next(w); ++it) {
    const int buf = it & 1;
    const uint32_t acc_parity = (it >> 1) & 1;
    if (!warp_wait(smem_u32(&ctrl->acc_empty[buf]), acc_parity ^ 1u, ctrl, a, kRoleMma,
                   kBarAccEmpty, true))
      break;
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
    for (int kb = w.kb0; kb < w.kb1; ++kb) {
      if (!warp_wait(smem_u32(&ctrl->full[stage]), phase, ctrl, a, kRoleMma, kBarFull, true)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int ks0 = kb * KD;
      const int nks = KD == 1 ? 1 : min(KD, kslices - ks0);
      // K-major: the 16-wide k-slice starts 32 bytes further along each swizzled
      // 128-byte row; 8-row groups are 1024 bytes apart.
      // MN-major: the k-slice is 16 rows of 128 bytes further on; 8-row groups are
      // 1024 bytes apart and swizzle atoms along M / N are kMnAtomBytes apart.
      const uint32_t a_step = p_kmajor ? 32u : 2048u;
      const uint32_t b_step = q_kmajor ? 32u : 2048u;
      if (elect_one()) {
#pragma unroll
        for (int t = 0; t < KD; ++t) {
          if (t == nks) break;
          const int slot = stage * KD + t;
          const uint64_t ad0 =
              smem_desc_sw128(smem_u32(ring_a + slot * Cfg::kABytes), p_kmajor ? 16u : kMnAtomBytes, 1024);
          const uint8_t* qtile = DQ ? code_ring + cstage * a.code_stage_bytes : ring_b + slot * Cfg::kBBytes;
          const uint64_t bd0 = smem_desc_sw128(smem_u32(qtile), q_kmajor ? 16u : kMnAtomBytes, 1024);
#pragma unroll
          for (int k = 0; k < kSliceBytes / 32; ++k)  // the start address sits in the descriptor's low bits
            mma_ss<CG, EB>(d_tmem, ad0 + ((a_step * k) >> 4), bd0 + ((b_step * k) >> 4), a.idesc,
                           (kb > w.kb0 || t > 0 || k > 0) ? 1u : 0u);
        }
        commit_both(smem_u32(&ctrl->empty[stage]));  // frees the stage once these MMAs have read it
        if constexpr (DQ) mma_commit<1>(smem_u32(&ctrl->code_empty[cstage]));  // and the code stage's Q tile
      }
      __syncwarp();
      if (++stage == a.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if constexpr (DQ) {
        if (++cstage == a.code_stages) cstage = 0;
      }
    }
    if (!ok) break;
    if (elect_one()) commit_both(smem_u32(&ctrl->acc_full[buf]));  // accumulator ready for the epilogues
    __syncwarp();
  }
  // Tensor Memory is freed only after every MMA issued here has finished.  The
  // elected lane is the one that issued them, so its commit tracks them all.
  if (elect_one()) {
    mma_commit<CG>(smem_u32(&ctrl->mma_done));
    wait_bounded(smem_u32(&ctrl->mma_done), 0, ctrl, a, kRoleMma, kBarDrain, false);
  }
  __syncwarp();
}

template <int BN, int CG, int EB, bool DQ, int EW>
__device__ __forceinline__ void epilogue_role(const TcArgs& a, const CUtensorMap* map_c, const CMaps* cmaps,
                                              uint8_t* staging, uint8_t* ring, TcCtrl* ctrl,
                                              uint32_t tmem_base,
                                              int warp, int lane, uint32_t rank, int first,
                                              int stride) {
  using Cfg = TcConfig<BN, CG, DQ, EW>;
  constexpr int kEpiThreads = 32 * Cfg::kEpiWarps;
  const int q = static_cast<int>(rank);  // rank inside the CTA pair (0: the leader)
  const int ew = warp - 2;       // epilogue warp
  const int quarter = warp & 3;  // a warp may only read TMEM lanes 32*(warp%4) .. +31
  const int row = quarter * 32 + lane;
  // the tile's columns cb .. cb + kEpiCols - 1 are this warp's (with eight
  // epilogue warps, two to a quarter of the rows, each takes half)
  const int cb = (ew / 4) * Cfg::kEpiCols;
  constexpr int kCols = Cfg::kEpiCols;
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  const float alpha = a.alpha;
  EpiOut out;
  out.c = make_cout(a);
  out.c0 = a.C;
  out.z = 0;
  out.map_c = map_c;
  out.staging = smem_u32(staging + ew * 2 * kStagingBuf);
  out.lane = lane;
  out.nstore = 0;
  out.ring = false;
  out.cbar = smem_u32(&ctrl->c_full[ew][0]);
  out.cphase = 0;
  out.pending = 0;
  out.jstart = 0;
  out.jend = 0;
  out.ctrl = ctrl;
  out.status = a.status;
  out.wait_ns = a.wait_limit_ns;
  out.cmaps = cmaps;
  out.classes = a.c_classes;
#pragma unroll
  for (int t = 0; t < 4; ++t) out.cy[t] = 0.0f;
  const int64_t esize = a.c_type == kCF32 ? 4 : a.c_type == kCE4M3 ? 1 : 2;
  int it = 0;
  WorkIter work(a.sched, first, stride);
  Unit w;
  for (; work.next(w); ++it) {
    const int buf = it & 1;
    const uint32_t acc_parity = (it >> 1) & 1;
    const int i = w.ti * Cfg::kTileM + q * kBM + row;
    const int jt = w.tj * BN;  // first column of the tile
    out.y0 = w.ti * Cfg::kTileM + q * kBM + quarter * 32;
    out.z = w.tb;
    // beta != 0 with bulk stores: the tile's first block of old C loads while
    // the accumulator is still being computed
    if (!w.partial) out.begin_tile(jt + cb, jt + cb + kCols);
    const bool ok = wait_bounded(smem_u32(&ctrl->acc_full[buf]), acc_parity, ctrl, a,
                                 kRoleEpilogue, kBarAccFull, true);
    if (bar_any(1, kEpiThreads, !ok)) break;  // all epilogue warps leave together
    tc_fence_after_sync();
    if (Cfg::kRingStagesC && (out.c.tma == kBulkRows || out.c.tma == kBulkTransposed) && !out.ring &&
        !out.c.blend_load) {
      WorkIter peek = work;
      Unit next_unit;
      // This CTA's last unit: its copies have landed and its MMAs (the pair's)
      // have read the ring for the last time, so the ring can stage C.
      if (!peek.next(next_unit)) out.use_ring(smem_u32(ring + ew * Cfg::kRingBufs * kStagingBuf));
    }
    const uint32_t taddr = lane_base + static_cast<uint32_t>(buf * BN);
    // the MMA (leader CTA) waits until every epilogue thread of the pair has read the buffer
    const uint32_t acc_empty_local = smem_u32(&ctrl->acc_empty[buf]);
    const uint32_t acc_empty = CG == 2 ? mapa_shared(acc_empty_local, 0) : acc_empty_local;
    auto release = [&]() {
      tc_fence_before_sync();
      if constexpr (CG == 2)
        mbar_arrive_cluster(acc_empty);
      else
        mbar_arrive(acc_empty);
    };
    {
      if (a.sched.groups > 0) {  // the group's rows of C; rows past its count are not stored
        out.c.C = static_cast<char*>(out.c0) + a.group_row[w.tb] * a.c_si * esize;
        out.c.I = a.group_m[w.tb];
      } else {
        out.c.C = static_cast<char*>(out.c0) + static_cast<int64_t>(w.tb) * a.c_sb * esize;
      }
    }
    if (!w.partial && EB == 1) {
      // 8-bit inputs: one 32-column read at a time (reading ahead, below,
      // measured 2% slower on the 4096^3 E4M3 GEMM, whose tiles are half as long)
#pragma unroll 1
      for (int c = cb; c < cb + kCols; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c, r);
        tmem_ld_wait(r);
        if (c + 32 == cb + kCols) release();  // last read of this accumulator: hand it back
        float v[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = alpha * __uint_as_float(r[t]);
        out.put(i, jt + c, v, (c >> 5) & 1);
      }
    } else if (!w.partial) {
      // Two register buffers: the next 32 columns are read from TMEM while the
      // current ones are converted and stored (5% faster at K = 1024, where the
      // epilogue of one tile outlasts the next tile's main loop).
      uint32_t ra[32], rb[32];
      tmem_ld_32x32b_x32(taddr + cb, ra);
#pragma unroll 1
      for (int c = cb; c < cb + kCols; c += 64) {
        tmem_ld_wait(ra);
        tmem_ld_32x32b_x32(taddr + c + 32, rb);
        {
          float v[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) v[t] = alpha * __uint_as_float(ra[t]);
          out.put(i, jt + c, v, 0);
        }
        tmem_ld_wait(rb);
        if (c + 64 < cb + kCols)
          tmem_ld_32x32b_x32(taddr + c + 64, ra);
        else
          release();  // last read of this accumulator: hand it back
        {
          float v[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) v[t] = alpha * __uint_as_float(rb[t]);
          out.put(i, jt + c + 32, v, 1);
        }
      }
    } else {
      // Partial of this k-range, in groups of four columns: the float4 of row r,
      // columns 4g .. 4g + 3 sits at index g * kBM + r, so that a warp's 32 rows
      // are 512 contiguous bytes and every access moves 16 bytes per lane.
      const int slot = w.pslot * Cfg::kCluster + static_cast<int>(rank);
      const int ctr = w.ctr * Cfg::kCluster + static_cast<int>(rank);
      float4* part = reinterpret_cast<float4*>(a.partials + static_cast<size_t>(slot) * BN * kBM);
#pragma unroll 1
      for (int c = cb; c < cb + kCols; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c, r);
        tmem_ld_wait(r);
        if (c + 32 == cb + kCols) release();
#pragma unroll
        for (int g = 0; g < 8; ++g)
          __stcg(part + static_cast<size_t>((c >> 2) + g) * kBM + row,
                 make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                             __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])));
      }
      // One GPU-scope fence by the arriving thread, after the barrier that orders
      // every epilogue thread's partial stores before it, publishes the whole
      // partial (fences are cumulative); a fence in each epilogue thread would
      // stall every one of them on its own stores.
      bar_sync(1, kEpiThreads);
      if (threadIdx.x == 64) {
        __threadfence();
        const int old = atomicAdd(&a.counters[ctr], 1);
        const uint32_t last = (old == w.ncontrib - 1) ? 1u : 0u;
        if (last) {
          atomicExch(&a.counters[ctr], 0);  // clean for the next call
          __threadfence();                  // the other contributions, before anyone reads them
        }
        *reinterpret_cast<volatile uint32_t*>(&ctrl->last) = last;
      }
      bar_sync(1, kEpiThreads);
      if (*reinterpret_cast<volatile uint32_t*>(&ctrl->last)) {
        out.begin_tile(jt + cb, jt + cb + kCols);
        // 64 columns per round: 16 independent 16-byte loads per contribution in
        // flight (the sum is latency-bound, one L2 round trip per round); 32 in
        // kernels of more than 320 threads, whose threads hold fewer registers.
        constexpr int kRound = threads_of(EW, DQ) > 320 ? 32 : 64;
        constexpr int kG = kRound / 4;
#pragma unroll 1
        for (int c = cb; c < cb + kCols; c += kRound) {
          float4 acc[kG];
#pragma unroll
          for (int g = 0; g < kG; ++g) acc[g] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
          for (int k = 0; k < w.ncontrib; ++k) {  // fixed k order: the sum does not depend on timing
            const int ks = contrib_slot(a.sched, w, k) * Cfg::kCluster + static_cast<int>(rank);
            const float4* ps = reinterpret_cast<const float4*>(a.partials + static_cast<size_t>(ks) * BN * kBM);
            float4 x[kG];
#pragma unroll
            for (int g = 0; g < kG; ++g) x[g] = __ldcg(ps + static_cast<size_t>((c >> 2) + g) * kBM + row);
#pragma unroll
            for (int g = 0; g < kG; ++g) {
              acc[g].x += x[g].x;
              acc[g].y += x[g].y;
              acc[g].z += x[g].z;
              acc[g].w += x[g].w;
            }
          }
#pragma unroll
          for (int h = 0; h < kRound / 32; ++h) {
            float v[32];
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              v[4 * g] = alpha * acc[8 * h + g].x;
              v[4 * g + 1] = alpha * acc[8 * h + g].y;
              v[4 * g + 2] = alpha * acc[8 * h + g].z;
              v[4 * g + 3] = alpha * acc[8 * h + g].w;
            }
            out.put(i, jt + c + 32 * h, v, ((c + 32 * h) >> 5) & 1);
          }
        }
      }
    }
  }
  out.finish();  // every bulk store has read its staging buffer before the CTA can exit
}

template <int BN, int CG, int EB, bool DQ, int EW>
__global__ void __launch_bounds__(threads_of(EW, DQ), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_p,
                   const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CMaps cmaps,
                   const TcArgs args) {
  using Cfg = TcConfig<BN, CG, DQ, EW>;
  // The roles take the arguments by reference; a local copy whose address never
  // leaves this kernel lets the compiler keep the fields in registers across
  // the global stores and "memory"-clobbering asm of the loops, instead of
  // reloading them from the parameter space after each one.
  const TcArgs a = args;
  // The next kernel of the stream may be scheduled now: its CTAs take SMs as
  // this grid's leave and run their set-up while this grid finishes.
  grid_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms need 1024-byte aligned tiles.
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* ring_a = smem;
  uint8_t* ring_b = smem + Cfg::kStages * Cfg::kABytes;
  uint8_t* code_ring = smem + Cfg::kRingBytes;  // (DQ kernels)
  TcCtrl* ctrl = reinterpret_cast<TcCtrl*>(smem + Cfg::kRingBytes + Cfg::kCodeRingBytes);
  uint8_t* staging = smem + Cfg::kRingBytes + Cfg::kCodeRingBytes + 1024;  // 1024-byte aligned

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A CTA pair shares each tile; its rank-0 CTA is the leader that issues the MMAs.
  // A cluster (a pair, or one CTA) walks the schedule as one slot.
  constexpr int kCl = Cfg::kCluster;
  const uint32_t rank = kCl > 1 ? cluster_ctarank() : 0u;
  const int first = static_cast<int>(blockIdx.x) / kCl;
  const int stride = static_cast<int>(gridDim.x) / kCl;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), DQ ? kConvWarps : 1);  // (DQ: one arrival per converter warp)
      mbar_init(smem_u32(&ctrl->empty[s]), 1);  // released by the pair's MMA commit
    }
    if (DQ)
      for (int s = 0; s < a.code_stages; ++s) {
        mbar_init(smem_u32(&ctrl->code_full[s]), 1);
        mbar_init(smem_u32(&ctrl->code_empty[s]), 1);
      }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl->acc_full[b]), 1);
      mbar_init(smem_u32(&ctrl->acc_empty[b]), 32 * Cfg::kEpiWarps * CG);
    }
    mbar_init(smem_u32(&ctrl->mma_done), 1);
    for (int w = 0; w < Cfg::kEpiWarps; ++w)
      for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&ctrl->c_full[w][b]), 1);
    ctrl->abort = 0;
    ctrl->last = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_p);
    prefetch_tensormap(&map_q);
    if (DQ) prefetch_tensormap(&cmaps.m[0]);
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(&ctrl->tmem_base), Cfg::kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kCl > 1) cluster_sync();  // every CTA's barriers exist before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem_base = ctrl->tmem_base;
  // Set-up done (barriers, tensor memory, tensor maps); no global memory has
  // been touched.  From here on operands, C, partials and counters may be those
  // of the previous kernel of the stream: wait until it has finished.
  grid_dependency_wait();

  if (warp == 0) {
    // k-slices per stage are a template argument of the issuing roles, so that
    // the one-slice loop compiles to the same straight-line issue code as
    // before two-slice stages existed (a runtime trip count cost ~12% at 4096^3)
    // (DQ kernels: one k-slice a stage, the planner's choice)
    if (!DQ && a.kdepth == 2)
      producer_role<BN, CG, EB, 2, DQ, EW>(&map_p, &map_q, &cmaps.m[0], a, ring_a, ring_b, code_ring, ctrl, rank, first,
                                       stride);
    else
      producer_role<BN, CG, EB, 1, DQ, EW>(&map_p, &map_q, &cmaps.m[0], a, ring_a, ring_b, code_ring, ctrl, rank, first,
                                       stride);
  } else if (warp == 1) {
    if (rank % CG == 0) {
      if (!DQ && a.kdepth == 2)
        mma_role<BN, CG, EB, 2, DQ, EW>(a, ring_a, ring_b, code_ring, ctrl, tmem_base, rank, first, stride);
      else
        mma_role<BN, CG, EB, 1, DQ, EW>(a, ring_a, ring_b, code_ring, ctrl, tmem_base, rank, first, stride);
    }
  } else if (warp < 2 + Cfg::kEpiWarps) {
    epilogue_role<BN, CG, EB, DQ, EW>(a, &map_c, &cmaps, staging, ring_a, ctrl, tmem_base, warp, lane, rank, first,
                                  stride);
  } else if constexpr (DQ) {
    converter_role<BN, CG>(a, ring_a, code_ring, ctrl, warp - 6, lane, first, stride);
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kCl > 1) {
    // After an abort, give copies the leader could not account for time to land.
    if (*reinterpret_cast<volatile uint32_t*>(&ctrl->abort)) {
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 100000) {
      }
    }
    cluster_sync();  // neither CTA leaves while the pair's MMAs may still touch it
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace g10
