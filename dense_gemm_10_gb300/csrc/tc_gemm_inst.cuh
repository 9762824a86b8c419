// tc_gemm_inst.cuh -- one instantiation of the tcgen05 GEMM kernel per
// translation unit (TC_BN set by the including file), so the three tile
// widths compile in parallel.
#include "tc_gemm.cuh"

#define TC_CAT2(a, b) a##b
#define TC_CAT(a, b) TC_CAT2(a, b)

namespace g10 {

cudaError_t TC_CAT(tc_prepare_bn, TC_BN)() {
  return cudaFuncSetAttribute(tc_gemm_kernel<TC_BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(TcConfig<TC_BN>::kSmemBytes));
}

cudaError_t TC_CAT(tc_launch_bn, TC_BN)(const CUtensorMap& map_p, const CUtensorMap& map_q,
                                        const TcArgs& args, int grid, cudaStream_t stream) {
  tc_gemm_kernel<TC_BN><<<grid, kThreads, TcConfig<TC_BN>::kSmemBytes, stream>>>(map_p, map_q, args);
  return cudaGetLastError();
}

}  // namespace g10
