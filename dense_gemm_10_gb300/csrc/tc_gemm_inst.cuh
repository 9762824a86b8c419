// tc_gemm_inst.cuh -- one instantiation of the tcgen05 GEMM kernel per
// translation unit (TC_BN and TC_CG set by the including file), so the tile
// configurations compile in parallel.
#include "tc_gemm.cuh"

#define TC_CAT4(a, b, c, d) a##b##c##d
#define TC_NAME(a, b, c, d) TC_CAT4(a, b, c, d)

namespace g10 {

cudaError_t TC_NAME(tc_prepare_bn, TC_BN, _cg, TC_CG)(int* max_clusters) {
  using Cfg = TcConfig<TC_BN, TC_CG>;
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<TC_BN, TC_CG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg::kSmemBytes));
  if (e != cudaSuccess || TC_CG == 1) return e;
  // How many CTA pairs can be resident at once (clusters must sit inside one GPC).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = TC_CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(TC_CG, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, tc_gemm_kernel<TC_BN, TC_CG>, &cfg);
}

cudaError_t TC_NAME(tc_launch_bn, TC_BN, _cg, TC_CG)(const CUtensorMap& map_p,
                                                     const CUtensorMap& map_q, const TcArgs& args,
                                                     int grid, cudaStream_t stream) {
  using Cfg = TcConfig<TC_BN, TC_CG>;
  if (TC_CG == 1) {
    tc_gemm_kernel<TC_BN, TC_CG><<<grid, kThreads, Cfg::kSmemBytes, stream>>>(map_p, map_q, args);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = TC_CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<TC_BN, TC_CG>, map_p, map_q, args);
}

}  // namespace g10
