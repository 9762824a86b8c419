// tc_gemm_inst.cuh -- one instantiation of the tcgen05 GEMM kernel per
// translation unit (TC_BN, TC_CG, TC_EB and, for kernels that convert
// block-scaled codes, TC_DQ, for eight epilogue warps TC_EW, set by the
// including file), so the tile configurations compile in parallel.
#include "tc_gemm.cuh"

#ifndef TC_DQ
#define TC_DQ 0
#endif
#ifndef TC_EW
#define TC_EW 4
#endif
#define TC_CAT10(a, b, c, d, e, f, g, h, i, j) a##b##c##d##e##f##g##h##i##j
#define TC_NAME(a, b, c, d, e, f, g, h, i, j) TC_CAT10(a, b, c, d, e, f, g, h, i, j)
#define TC_KERNEL tc_gemm_kernel<TC_BN, TC_CG, TC_EB, TC_DQ != 0, TC_EW>

namespace g10 {

cudaError_t TC_NAME(tc_prepare_bn, TC_BN, _cg, TC_CG, _eb, TC_EB, _dq, TC_DQ, _ew, TC_EW)(int* max_clusters) {
  using Cfg = TcConfig<TC_BN, TC_CG, TC_DQ != 0, TC_EW>;
  cudaError_t e = cudaFuncSetAttribute(TC_KERNEL,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg::kSmemBytes));
  if (e != cudaSuccess || TC_CG == 1) return e;
  // How many CTA pairs can be resident at once (a cluster must sit inside one GPC).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = TC_CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(TC_CG, 1, 1);
  cfg.blockDim = dim3(threads_of(TC_EW, TC_DQ != 0), 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, TC_KERNEL, &cfg);
}

cudaError_t TC_NAME(tc_launch_bn, TC_BN, _cg, TC_CG, _eb, TC_EB, _dq, TC_DQ, _ew, TC_EW)(
    const CUtensorMap& map_p, const CUtensorMap& map_q, const CUtensorMap& map_c, const CMaps& cmaps,
    const TcArgs& args, int grid, cudaStream_t stream) {
  using Cfg = TcConfig<TC_BN, TC_CG, TC_DQ != 0, TC_EW>;
  const size_t smem = Cfg::kSmemBytes;  // every epilogue stages C (bulk or direct stores)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (TC_CG > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = TC_CG;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (args.pdl) {  // may start while the previous kernel of the stream finishes (griddepcontrol)
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads_of(TC_EW, TC_DQ != 0), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, TC_KERNEL, map_p, map_q, map_c, cmaps, args);
}

}  // namespace g10
