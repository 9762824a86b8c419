// tc_dispatch.cu -- the kernel instantiation for a tile configuration.
#include "tc_gemm.cuh"

namespace g10 {

#define TC_DECLARE(BN, CG, MC)                                                                     \
  cudaError_t tc_prepare_bn##BN##_cg##CG##_mc##MC(int* max_clusters);                             \
  cudaError_t tc_launch_bn##BN##_cg##CG##_mc##MC(const CUtensorMap&, const CUtensorMap&,            \
                                                 const CUtensorMap&, const TcArgs&, int,            \
                                                 cudaStream_t);
TC_DECLARE(64, 1, 1)
TC_DECLARE(128, 1, 1)
TC_DECLARE(256, 1, 1)
TC_DECLARE(128, 2, 1)
TC_DECLARE(256, 2, 1)
TC_DECLARE(256, 2, 2)
TC_DECLARE(64, 2, 1)

const TileConfig kTileConfigs[kNumTileConfigs] = {
    {64, 1, 1}, {128, 1, 1}, {256, 1, 1}, {128, 2, 1}, {256, 2, 1}, {256, 2, 2}, {64, 2, 1}};

int tc_config_index(int bn, int cg, int mc) {
  for (int i = 0; i < kNumTileConfigs; ++i)
    if (kTileConfigs[i].bn == bn && kTileConfigs[i].cg == cg && kTileConfigs[i].mc == mc) return i;
  return -1;
}

int tc_stages(int bn, int cg, int mc) {
  switch (tc_config_index(bn, cg, mc)) {
    case 0: return TcConfig<64, 1, 1>::kStages;
    case 1: return TcConfig<128, 1, 1>::kStages;
    case 2: return TcConfig<256, 1, 1>::kStages;
    case 3: return TcConfig<128, 2, 1>::kStages;
    case 4: return TcConfig<256, 2, 1>::kStages;
    case 5: return TcConfig<256, 2, 2>::kStages;
    case 6: return TcConfig<64, 2, 1>::kStages;
  }
  return 0;
}

cudaError_t tc_prepare(int bn, int cg, int mc, int* max_clusters) {
  *max_clusters = 0;
  switch (tc_config_index(bn, cg, mc)) {
    case 0: return tc_prepare_bn64_cg1_mc1(max_clusters);
    case 1: return tc_prepare_bn128_cg1_mc1(max_clusters);
    case 2: return tc_prepare_bn256_cg1_mc1(max_clusters);
    case 3: return tc_prepare_bn128_cg2_mc1(max_clusters);
    case 4: return tc_prepare_bn256_cg2_mc1(max_clusters);
    case 5: return tc_prepare_bn256_cg2_mc2(max_clusters);
    case 6: return tc_prepare_bn64_cg2_mc1(max_clusters);
  }
  return cudaErrorInvalidValue;
}

cudaError_t tc_launch(int bn, int cg, int mc, const CUtensorMap& map_p, const CUtensorMap& map_q,
                      const CUtensorMap& map_c, const TcArgs& args, int grid, cudaStream_t stream) {
  switch (tc_config_index(bn, cg, mc)) {
    case 0: return tc_launch_bn64_cg1_mc1(map_p, map_q, map_c, args, grid, stream);
    case 1: return tc_launch_bn128_cg1_mc1(map_p, map_q, map_c, args, grid, stream);
    case 2: return tc_launch_bn256_cg1_mc1(map_p, map_q, map_c, args, grid, stream);
    case 3: return tc_launch_bn128_cg2_mc1(map_p, map_q, map_c, args, grid, stream);
    case 4: return tc_launch_bn256_cg2_mc1(map_p, map_q, map_c, args, grid, stream);
    case 5: return tc_launch_bn256_cg2_mc2(map_p, map_q, map_c, args, grid, stream);
    case 6: return tc_launch_bn64_cg2_mc1(map_p, map_q, map_c, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace g10
