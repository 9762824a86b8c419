// epi_ops.cuh -- the elementwise operations fused into a GEMM's store of C and
// the conversions to C's element types, shared by the tcgen05 kernel's
// epilogue and the K == 0 kernel.
//
// The operations are the ones "第4章：经典算子实现 —— GEMM" (section 7.2: GEMM
// + bias + activation) and "GPU GEMM 优化完全拆解（三）" (mainloop 与 epilogue:
// ReLU and quantisation scaling done before write-back) fuse into the
// epilogue: z += bias, z = act(z) with ReLU max(z, 0) or GELU z * Phi(z) =
// z * (1 + erf(z / sqrt 2)) / 2, then z *= out_scale.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "gemm_internal.h"

namespace g10 {

__device__ __forceinline__ float apply_ops(const EpiOps& o, float z, int64_t i, int64_t j) {
  if (o.bias) z += __ldg(o.bias + (o.bias_on_i ? i : j));
  if (o.act == kActRelu) z = z > 0.0f ? z : 0.0f;
  else if (o.act == kActGelu) z = 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
  return z * o.out_scale;
}

// fp32 -> E4M3 with round-to-nearest-even, saturating at +-448 (quantised output).
__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float from_e4m3(uint8_t b) {
  __nv_fp8_e4m3 x;
  x.__x = b;
  return static_cast<float>(x);
}

}  // namespace g10
