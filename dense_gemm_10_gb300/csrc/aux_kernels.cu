// aux_kernels.cu -- the non-tensor-core kernels of the library:
//  * repack: copies an operand whose rows are not 16-byte aligned into
//    an aligned buffer, because the tensor-memory-accelerator copy engine only
//    reads rows whose pitch is a multiple of 16 bytes;
//  * unstage_c: the other way for C: the aligned copy that bulk stores wrote
//    goes into C's own rows;
//  * split_tf32: writes an fp32 operand K-major as TF32 values for the TF32
//    tensor-core kind ("GPU GEMM 优化完全拆解（三）", 数值精度).  One part: the
//    value cut to TF32 (sign, 8-bit exponent, top 10 fraction bits), as the
//    tensor core reads an fp32 operand.  Several parts (the fp32 GEMM from
//    three TF32 products): hi = TF32(x) and lo = TF32(x - hi), both rounded to
//    nearest, laid out in segments chosen by a bit pattern; the GEMM reads
//    the segments in the order that sums the chosen products;
//  * dequant_block_scaled: writes a block-scaled operand (MXFP8 or NVFP4 codes
//    with one scale code per block of k, "CUDA GEMM 矩阵乘法优化指南", 13.2) as
//    bf16 values code x scale, K-major, for the bf16 tensor-core GEMM.  Each
//    such value has at most 6 significant bits (E2M1 x E4M3, E4M3 x 2^e,
//    E5M2 x 2^e), so bf16 holds it exactly inside its exponent range;
//  * scale_c: C = ops(beta * C), the whole GEMM when K == 0 ("CUDA GEMM
//    矩阵乘法优化指南", section 2.1, with an empty sum), with the fused epilogue
//    operations of epi_ops.cuh.
// All are HBM-bound.  repack and unstage_c give each thread one 16-byte
// piece of four rows, with every load of the four rows issued before the
// first store; scale_c is a grid-stride loop over a grid sized to the SM count.
#include <algorithm>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "epi_ops.cuh"

namespace g10 {

// Bytes sh .. sh + 15 of the 32 bytes (lo, hi), sh in 0 .. 15.
__device__ __forceinline__ uint4 bytes_at(const uint4& lo, const uint4& hi, int sh) {
  uint32_t w0, w1, w2, w3, w4;  // the five words the result's bytes fall in
  switch (sh >> 2) {
    case 0: w0 = lo.x; w1 = lo.y; w2 = lo.z; w3 = lo.w; w4 = hi.x; break;
    case 1: w0 = lo.y; w1 = lo.z; w2 = lo.w; w3 = hi.x; w4 = hi.y; break;
    case 2: w0 = lo.z; w1 = lo.w; w2 = hi.x; w3 = hi.y; w4 = hi.z; break;
    default: w0 = lo.w; w1 = hi.x; w2 = hi.y; w3 = hi.z; w4 = hi.w; break;
  }
  const uint32_t r = static_cast<uint32_t>(sh & 3) * 8;
  return make_uint4(__funnelshift_r(w0, w1, r), __funnelshift_r(w1, w2, r), __funnelshift_r(w2, w3, r),
                    __funnelshift_r(w3, w4, r));
}

// One thread per 16-byte piece of the aligned copy, four rows at a time.  A
// source row may start anywhere, so the piece's bytes are read as the one or
// two aligned 16-byte pieces of the source they fall in (each holds at least
// one byte of the row, so it lies in memory the row's allocation maps) and
// shifted into place: two loads per piece where an element at a time took
// eight (bf16 B of 1000 x 4097: 8.2 us that way).  All loads of the four
// rows are issued before the first store.  The copy's rows are padded to
// whole pieces; the padding receives zeros (the tensor maps stop at `cols`, so
// it is never read).  The kernel lets the next kernel of the stream (a GEMM
// launched as a programmatic dependent) start its set-up on SMs this grid has
// left; that GEMM waits for this grid's completion before reading the copy.
template <typename T>
__global__ void __launch_bounds__(256) repack_kernel(const T* __restrict__ src, int64_t lds, int64_t sbs,
                                                     T* __restrict__ dst, int64_t ldd, int64_t dbs, int64_t rows,
                                                     int64_t cols, int64_t nb) {
  constexpr int kV = 16 / sizeof(T);
  constexpr int kRows = 4;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kV;
  if (c >= cols) return;
  const int nbytes = static_cast<int>(cols - c < kV ? cols - c : kV) * static_cast<int>(sizeof(T));
  for (int64_t b = blockIdx.z; b < nb; b += gridDim.z)
  for (int64_t r0 = static_cast<int64_t>(blockIdx.y) * kRows; r0 < rows; r0 += static_cast<int64_t>(gridDim.y) * kRows) {
    const int nr = rows - r0 < kRows ? static_cast<int>(rows - r0) : kRows;
    uint4 lo[kRows], hi[kRows];
    int sh[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      lo[u] = hi[u] = make_uint4(0u, 0u, 0u, 0u);
      sh[u] = 0;
      if (u < nr) {
        const uintptr_t s = reinterpret_cast<uintptr_t>(src + b * sbs + (r0 + u) * lds + c);
        const uint4* a = reinterpret_cast<const uint4*>(s & ~uintptr_t{15});
        sh[u] = static_cast<int>(s & 15u);
        lo[u] = __ldg(a);
        if (sh[u] + nbytes > 16) hi[u] = __ldg(a + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      if (u < nr) {
        uint4 x = bytes_at(lo[u], hi[u], sh[u]);
        if (nbytes < 16) {  // the row's last, partial piece: zeros past the row
          uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int keep = nbytes - 4 * j;
            w[j] = keep >= 4 ? w[j] : keep <= 0 ? 0u : (w[j] & ((1u << (8 * keep)) - 1u));
          }
        }
        *reinterpret_cast<uint4*>(dst + b * dbs + (r0 + u) * ldd + c) = x;
      }
    }
  }
}

__global__ void scale_c_kernel(void* C, int32_t c_type, int64_t M, int64_t N, int64_t ldc,
                               float beta, EpiOps ops, int64_t batch, int64_t sbc) {
  const bool any = ops.any();
  for (int64_t b = blockIdx.z; b < batch; b += gridDim.z)
  for (int64_t r = blockIdx.y; r < M; r += gridDim.y) {
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < N;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int64_t off = b * sbc + r * ldc + c;
      if (c_type == kCF32) {
        float* p = static_cast<float*>(C) + off;
        float z = beta == 0.0f ? 0.0f : beta * *p;
        *p = any ? apply_ops(ops, z, r, c) : z;
      } else if (c_type == kCBF16) {
        __nv_bfloat16* p = static_cast<__nv_bfloat16*>(C) + off;
        float z = beta == 0.0f ? 0.0f : beta * __bfloat162float(*p);
        *p = __float2bfloat16_rn(any ? apply_ops(ops, z, r, c) : z);
      } else if (c_type == kCF16) {
        __half* p = static_cast<__half*>(C) + off;
        float z = beta == 0.0f ? 0.0f : beta * __half2float(*p);
        *p = __float2half_rn(any ? apply_ops(ops, z, r, c) : z);
      } else {  // E4M3 output is written only (beta == 0)
        static_cast<uint8_t*>(C)[off] = to_e4m3(any ? apply_ops(ops, 0.0f, r, c) : 0.0f);
      }
    }
  }
}

// fp32 -> TF32 (10 fraction bits), round to nearest, ties away from zero.
__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// fp32 -> TF32 by dropping the 13 low fraction bits (NaN stays NaN).
__device__ __forceinline__ float cut_tf32(float x) {
  return x != x ? x : __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// Element (r, k) of one source matrix: src[k * lds + r] (kTrans) or src[r * lds + k].
// Output row r: parts segments of seg (>= K) values at dst[r * ldd], values
// K .. seg - 1 zero; parts == 1: the cut value; else segment s holds the low
// part when bit s of pattern is set, the high part otherwise.  Transposed
// sources go through a 32 x 32 shared-memory tile so that reads and writes are
// both coalesced.
template <bool kTrans>
__global__ void split_tf32_kernel(const float* __restrict__ src, int64_t lds, int64_t sbs, float* __restrict__ dst,
                                  int64_t ldd, int64_t dbs, int64_t rows, int64_t K, int64_t seg, int64_t nb,
                                  int parts, int pattern) {
  __shared__ float tile[32][33];
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8 threads
  const int64_t tiles_r = (rows + 31) / 32, tiles_k = (seg + 31) / 32;
  for (int64_t b = blockIdx.z; b < nb; b += gridDim.z) {
    const float* S = src + b * sbs;
    float* D = dst + b * dbs;
    for (int64_t t = blockIdx.x; t < tiles_r * tiles_k; t += gridDim.x) {
      const int64_t r0 = (t / tiles_k) * 32, k0 = (t % tiles_k) * 32;
      __syncthreads();
      for (int i = ty; i < 32; i += 8) {  // tile[k - k0][r - r0]
        if (kTrans) {
          const int64_t k = k0 + i, r = r0 + tx;
          tile[i][tx] = (k < K && r < rows) ? S[k * lds + r] : 0.0f;
        } else {
          const int64_t r = r0 + i, k = k0 + tx;
          tile[tx][i] = (k < K && r < rows) ? S[r * lds + k] : 0.0f;
        }
      }
      __syncthreads();
      for (int i = ty; i < 32; i += 8) {
        const int64_t r = r0 + i, k = k0 + tx;
        if (r >= rows || k >= seg) continue;
        const float x = tile[tx][i];  // (0 past K)
        float* row = D + r * ldd;
        if (parts == 1) {
          row[k] = cut_tf32(x);
          continue;
        }
        float hi = to_tf32(x);
        if (isinf(hi) && !isinf(x)) hi = cut_tf32(x);  // rounded past the largest value
        const float lo = isfinite(x) ? to_tf32(x - hi) : 0.0f;
        for (int s = 0; s < parts; ++s) row[s * seg + k] = ((pattern >> s) & 1) ? lo : hi;
      }
    }
  }
}

// Code values.  E4M3 / E5M2 through CUDA's FP8 conversions; E2M1 (sign, two
// exponent bits with bias 1, one fraction bit) from its eight magnitudes.
__device__ __forceinline__ float fp8_value(uint8_t c, bool e5m2) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), e5m2 ? __NV_E5M2 : __NV_E4M3);
  return __half2float(__half(h));
}
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const float mag = (c & 6u) == 0 ? 0.5f * static_cast<float>(c & 1u)
                                  : static_cast<float>(2u + (c & 1u)) * __int_as_float((125 + ((c >> 1) & 3)) << 23);  // (2 + m) 2^(e - 2)
  return (c & 8u) ? -mag : mag;
}
// Scale codes: E8M0 = 2^(s - 127) (255 is NaN); unsigned E4M3 = E4M3 without its sign.
__device__ __forceinline__ float scale_value(uint8_t s, bool e8m0) {
  if (!e8m0) return fp8_value(static_cast<uint8_t>(s & 0x7F), false);
  if (s == 255) return __int_as_float(0x7FC00000);
  return s == 0 ? __int_as_float(0x00400000) /* 2^-127, a subnormal */ : __int_as_float(static_cast<int>(s) << 23);
}

// One thread per 16 consecutive values of a row: dst[r * ldd + k] for k0 <= k <
// k0 + 16 (values past K written as 0; ldd a multiple of 16).  fmt: 0 E4M3, 1
// E5M2, 2 E2M1 (two a byte, even k in the low four bits); lds in values.  16
// divides the block, so one scale code covers the 16 values.  `vec`: rows
// start 16-byte (FP8) / 8-byte (FP4) aligned, so whole pieces load as one
// vector; the tail of a row (k0 + 16 > K) is read byte by byte.
// Raw code words of one 16-value piece: FP8 w[0..3] (byte t of the piece at bits
// 8 (t % 4) of w[t / 4]), FP4 w[0..1] (value t at bits 4 (t % 8) of w[t / 8]).
__device__ __forceinline__ void load_piece(const uint8_t* __restrict__ src, int64_t lds, int fmt, int vec, int64_t r,
                                           int64_t k0, int64_t K, uint32_t (&w)[4]) {
  w[0] = w[1] = w[2] = w[3] = 0u;
  if (k0 >= K) return;
  const bool whole = vec != 0 && k0 + 16 <= K;
  if (fmt == 2) {
    const uint8_t* row = src + r * (lds / 2);
    if (whole) {
      const uint2 q = *reinterpret_cast<const uint2*>(row + k0 / 2);
      w[0] = q.x;
      w[1] = q.y;
    } else {
      for (int t = 0; t < 16 && k0 + t < K; t += 2)
        w[t >> 3] |= static_cast<uint32_t>(row[(k0 + t) / 2]) << (4 * (t & 7));
    }
  } else {
    const uint8_t* row = src + r * lds;
    if (whole) {
      const uint4 q = *reinterpret_cast<const uint4*>(row + k0);
      w[0] = q.x;
      w[1] = q.y;
      w[2] = q.z;
      w[3] = q.w;
    } else {
      for (int t = 0; t < 16 && k0 + t < K; ++t) w[t >> 2] |= static_cast<uint32_t>(row[k0 + t]) << (8 * (t & 3));
    }
  }
}

// Thread x of the grid's x dimension takes the 16-value piece k0 = 16 x of rows
// blockIdx.y, blockIdx.y + gridDim.y, ... and writes dst[r * ldd + k] for its
// 16 values (values past K written as 0; ldd a multiple of 16).  fmt: 0 E4M3,
// 1 E5M2, 2 E2M1 (two a byte, even k in the low four bits); lds in values.  16
// divides the block, so one scale code covers a piece.  `vec`: rows start
// 16-byte (FP8) / 8-byte (FP4) aligned, so whole pieces load as one vector; the
// tail of a row (k0 + 16 > K) is read byte by byte.
template <bool kF16>
__global__ void dequant_kernel(const uint8_t* __restrict__ src, int64_t lds, const uint8_t* __restrict__ sf,
                               int64_t ld_sf, int fmt, int e8m0, int block, int vec, uint16_t* __restrict__ dst,
                               int64_t ldd, int64_t rows, int64_t K) {
  const int64_t k0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 16;
  if (k0 >= ldd) return;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    uint32_t w[4];
    load_piece(src, lds, fmt, vec, r, k0, K, w);
    const float scale = k0 < K ? scale_value(sf[r * ld_sf + k0 / block], e8m0 != 0) : 0.0f;
    uint32_t packed[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      float x0, x1;
      if (fmt == 2) {
        x0 = e2m1_value((w[(2 * t) >> 3] >> (4 * ((2 * t) & 7))) & 0xFu);
        x1 = e2m1_value((w[(2 * t + 1) >> 3] >> (4 * ((2 * t + 1) & 7))) & 0xFu);
      } else {
        x0 = fp8_value(static_cast<uint8_t>(w[(2 * t) >> 2] >> (8 * ((2 * t) & 3))), fmt == 1);
        x1 = fp8_value(static_cast<uint8_t>(w[(2 * t + 1) >> 2] >> (8 * ((2 * t + 1) & 3))), fmt == 1);
      }
      // values past K (the high half of a last, half-used FP4 byte too) are 0
      if (k0 + 2 * t >= K) x0 = 0.0f;
      if (k0 + 2 * t + 1 >= K) x1 = 0.0f;
      if constexpr (kF16) {  // (NVFP4 values: at most 6 significant bits, inside fp16's range)
        const __half2 pr = __floats2half2_rn(x0 * scale, x1 * scale);
        packed[t] = *reinterpret_cast<const uint32_t*>(&pr);
      } else {
        const __nv_bfloat162 pr = __floats2bfloat162_rn(x0 * scale, x1 * scale);
        packed[t] = *reinterpret_cast<const uint32_t*>(&pr);
      }
    }
    uint4* out = reinterpret_cast<uint4*>(dst + r * ldd + k0);
    out[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    out[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
}

static dim3 grid_3d(int64_t rows, int64_t cols, int64_t nb, int sm_count) {
  const int64_t bx = (cols + 255) / 256 < 16 ? (cols + 255) / 256 : 16;
  int64_t by = (static_cast<int64_t>(sm_count) * 8 + bx - 1) / bx;
  if (by > rows) by = rows;
  if (by > 65535) by = 65535;
  int64_t bz = nb < 65535 ? nb : 65535;
  if (bz * by > 4 * 65535) bz = (4 * 65535) / (by > 0 ? by : 1);
  return dim3(static_cast<unsigned>(bx > 0 ? bx : 1), static_cast<unsigned>(by > 0 ? by : 1),
              static_cast<unsigned>(bz > 0 ? bz : 1));
}

cudaError_t repack_launch(const void* src, int64_t lds, int64_t sbs, void* dst, int64_t ldd, int64_t dbs,
                          int64_t rows, int64_t cols, int64_t nb, int esize, int sm_count,
                          cudaStream_t stream) {
  (void)sm_count;
  if (rows <= 0 || cols <= 0 || nb <= 0) return cudaSuccess;
  // the aligned copy: 16-byte aligned base, rows and batches of whole 16-byte pieces
  if ((reinterpret_cast<uintptr_t>(dst) % 16) != 0 || (ldd * esize) % 16 != 0 || (nb > 1 && (dbs * esize) % 16 != 0) ||
      ldd * esize < (cols * esize + 15) / 16 * 16)
    return cudaErrorInvalidValue;
  const int64_t pieces = (cols * esize + 15) / 16;
  const int64_t gx = (pieces + 255) / 256;
  if (gx > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(gx), static_cast<unsigned>(std::min<int64_t>((rows + 3) / 4, 65535)),
               static_cast<unsigned>(std::min<int64_t>(nb, 65535)));
  if (esize == 1)
    repack_kernel<uint8_t><<<g, 256, 0, stream>>>(static_cast<const uint8_t*>(src), lds, sbs,
                                                  static_cast<uint8_t*>(dst), ldd, dbs, rows, cols, nb);
  else
    repack_kernel<uint16_t><<<g, 256, 0, stream>>>(static_cast<const uint16_t*>(src), lds, sbs,
                                                   static_cast<uint16_t*>(dst), ldd, dbs, rows, cols, nb);
  return cudaGetLastError();
}

// The aligned copy of C (rows of lds elements, 16-byte aligned) into C: one
// thread per 16-byte piece of four rows, the four pieces loaded before any
// element is stored (a thread that moved one element at a time kept one load
// in flight and ran at a third of the HBM bandwidth); the elements go out one
// by one, since C's rows may start anywhere.  Pieces past `cols` are read (the
// aligned rows hold them) but not written.
template <typename T>
__global__ void __launch_bounds__(256) unstage_c_kernel(const T* __restrict__ src, int64_t lds, T* __restrict__ dst,
                                                        int64_t ldd, int64_t rows, int64_t cols) {
  constexpr int kV = 16 / sizeof(T);
  constexpr int kRows = 4;
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kV;
  if (c >= cols) return;
  const int nv = cols - c < kV ? static_cast<int>(cols - c) : kV;
  for (int64_t r0 = static_cast<int64_t>(blockIdx.y) * kRows; r0 < rows; r0 += static_cast<int64_t>(gridDim.y) * kRows) {
    const int nr = rows - r0 < kRows ? static_cast<int>(rows - r0) : kRows;
    uint4 x[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u)
      if (u < nr) x[u] = *reinterpret_cast<const uint4*>(src + (r0 + u) * lds + c);
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      if (u < nr) {
        const T* e = reinterpret_cast<const T*>(&x[u]);
        T* d = dst + (r0 + u) * ldd + c;
#pragma unroll
        for (int t = 0; t < kV; ++t)
          if (t < nv) d[t] = e[t];
      }
    }
  }
}

cudaError_t unstage_c_launch(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                             int esize, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(src) % 16) != 0 || (lds * esize) % 16 != 0) return cudaErrorInvalidValue;
  const int64_t pieces = (cols * esize + 15) / 16;
  const int64_t gx = (pieces + 255) / 256;
  int64_t gy = (rows + 3) / 4;
  if (gy > 65535) gy = 65535;
  if (gx > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
  if (esize == 4)
    unstage_c_kernel<uint32_t><<<g, 256, 0, stream>>>(static_cast<const uint32_t*>(src), lds,
                                                      static_cast<uint32_t*>(dst), ldd, rows, cols);
  else if (esize == 2)
    unstage_c_kernel<uint16_t><<<g, 256, 0, stream>>>(static_cast<const uint16_t*>(src), lds,
                                                      static_cast<uint16_t*>(dst), ldd, rows, cols);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t split_tf32_launch(const float* src, int64_t lds, int64_t sbs, bool transposed, float* dst,
                              int64_t ldd, int64_t dbs, int64_t rows, int64_t K, int64_t seg, int64_t nb, int parts,
                              int pattern, int sm_count, cudaStream_t stream) {
  if (seg < K || ldd < parts * seg) return cudaErrorInvalidValue;
  const int64_t tiles = ((rows + 31) / 32) * ((seg + 31) / 32);
  int64_t gx = static_cast<int64_t>(sm_count) * 8;
  if (gx > tiles) gx = tiles;
  int64_t gz = nb < 65535 ? nb : 65535;
  const dim3 grid(static_cast<unsigned>(gx > 0 ? gx : 1), 1, static_cast<unsigned>(gz > 0 ? gz : 1));
  if (transposed)
    split_tf32_kernel<true><<<grid, dim3(32, 8), 0, stream>>>(src, lds, sbs, dst, ldd, dbs, rows, K, seg, nb,
                                                              parts, pattern);
  else
    split_tf32_kernel<false><<<grid, dim3(32, 8), 0, stream>>>(src, lds, sbs, dst, ldd, dbs, rows, K, seg, nb,
                                                               parts, pattern);
  return cudaGetLastError();
}

cudaError_t dequant_launch(const void* src, int64_t lds, const void* sf, int64_t ld_sf, int fmt, bool e8m0,
                           int block, void* dst, int64_t ldd, int64_t rows, int64_t K, bool f16_out, int sm_count,
                           cudaStream_t stream) {
  if (ldd % 16 != 0) return cudaErrorInvalidValue;
  const int64_t pieces = ldd / 16;  // per row
  const unsigned gx = static_cast<unsigned>((pieces + 127) / 128);
  // rows per pass: about 16 blocks of 128 threads per SM in all
  int64_t gy = static_cast<int64_t>(sm_count) * 16 / gx;
  if (gy > rows) gy = rows;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const uintptr_t base = reinterpret_cast<uintptr_t>(src);
  const int vec = fmt == 2 ? (base % 8 == 0 && (lds / 2) % 8 == 0) : (base % 16 == 0 && lds % 16 == 0);
  const dim3 grid(gx, static_cast<unsigned>(gy), 1);
  if (f16_out)
    dequant_kernel<true><<<grid, 128, 0, stream>>>(static_cast<const uint8_t*>(src), lds,
                                                   static_cast<const uint8_t*>(sf), ld_sf, fmt, e8m0 ? 1 : 0, block,
                                                   vec, static_cast<uint16_t*>(dst), ldd, rows, K);
  else
    dequant_kernel<false><<<grid, 128, 0, stream>>>(static_cast<const uint8_t*>(src), lds,
                                                    static_cast<const uint8_t*>(sf), ld_sf, fmt, e8m0 ? 1 : 0, block,
                                                    vec, static_cast<uint16_t*>(dst), ldd, rows, K);
  return cudaGetLastError();
}

cudaError_t scale_c_launch(void* C, int32_t c_type, int64_t M, int64_t N, int64_t ldc, float beta,
                           const EpiOps& ops, int64_t batch, int64_t sbc, int sm_count,
                           cudaStream_t stream) {
  scale_c_kernel<<<grid_3d(M, N, batch, sm_count), 256, 0, stream>>>(C, c_type, M, N, ldc, beta, ops, batch,
                                                                       sbc);
  return cudaGetLastError();
}

}  // namespace g10
