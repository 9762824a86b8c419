// aux_kernels.cu -- the two non-tensor-core kernels of the library:
//  * repack: copies an operand whose rows are not 16-byte aligned into
//    an aligned buffer, because the tensor-memory-accelerator copy engine only
//    reads rows whose pitch is a multiple of 16 bytes;
//  * scale_c: C = ops(beta * C), the whole GEMM when K == 0 ("CUDA GEMM
//    矩阵乘法优化指南", section 2.1, with an empty sum), with the fused epilogue
//    operations of epi_ops.cuh.
// Both are HBM-bound grid-stride copies over a grid sized to the SM count.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epi_ops.cuh"

namespace g10 {

template <typename T>
__global__ void repack_kernel(const T* __restrict__ src, int64_t lds, int64_t sbs, T* __restrict__ dst,
                              int64_t ldd, int64_t dbs, int64_t rows, int64_t cols, int64_t nb) {
  for (int64_t b = blockIdx.z; b < nb; b += gridDim.z)
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const T* s = src + b * sbs + r * lds;
    T* d = dst + b * dbs + r * ldd;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < cols;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x)
      d[c] = s[c];
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
  const dim3 g = grid_3d(rows, cols, nb, sm_count);
  if (esize == 1)
    repack_kernel<uint8_t><<<g, 256, 0, stream>>>(static_cast<const uint8_t*>(src), lds, sbs,
                                                  static_cast<uint8_t*>(dst), ldd, dbs, rows, cols, nb);
  else
    repack_kernel<uint16_t><<<g, 256, 0, stream>>>(static_cast<const uint16_t*>(src), lds, sbs,
                                                   static_cast<uint16_t*>(dst), ldd, dbs, rows, cols, nb);
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
