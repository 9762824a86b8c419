// tc_dispatch.cu -- choose the kernel instantiation for a tile width and CTA group.
#include "tc_gemm.cuh"

namespace g10 {

#define TC_DECLARE(BN, CG)                                                                  \
  cudaError_t tc_prepare_bn##BN##_cg##CG(int* max_clusters);                                \
  cudaError_t tc_launch_bn##BN##_cg##CG(const CUtensorMap&, const CUtensorMap&, const TcArgs&, \
                                        int, cudaStream_t);
TC_DECLARE(64, 1)
TC_DECLARE(128, 1)
TC_DECLARE(256, 1)
TC_DECLARE(128, 2)
TC_DECLARE(256, 2)

bool tc_supported(int bn, int cg) {
  return (cg == 1 && (bn == 64 || bn == 128 || bn == 256)) || (cg == 2 && (bn == 128 || bn == 256));
}

int tc_stages(int bn, int cg) {
  if (cg == 2) return bn == 256 ? TcConfig<256, 2>::kStages : TcConfig<128, 2>::kStages;
  return bn == 256 ? TcConfig<256, 1>::kStages
                   : bn == 128 ? TcConfig<128, 1>::kStages : TcConfig<64, 1>::kStages;
}

cudaError_t tc_prepare(int bn, int cg, int* max_clusters) {
  *max_clusters = 0;
  if (cg == 1 && bn == 64) return tc_prepare_bn64_cg1(max_clusters);
  if (cg == 1 && bn == 128) return tc_prepare_bn128_cg1(max_clusters);
  if (cg == 1 && bn == 256) return tc_prepare_bn256_cg1(max_clusters);
  if (cg == 2 && bn == 128) return tc_prepare_bn128_cg2(max_clusters);
  if (cg == 2 && bn == 256) return tc_prepare_bn256_cg2(max_clusters);
  return cudaErrorInvalidValue;
}

cudaError_t tc_launch(int bn, int cg, const CUtensorMap& map_p, const CUtensorMap& map_q,
                      const TcArgs& args, int grid, cudaStream_t stream) {
  if (cg == 1 && bn == 64) return tc_launch_bn64_cg1(map_p, map_q, args, grid, stream);
  if (cg == 1 && bn == 128) return tc_launch_bn128_cg1(map_p, map_q, args, grid, stream);
  if (cg == 1 && bn == 256) return tc_launch_bn256_cg1(map_p, map_q, args, grid, stream);
  if (cg == 2 && bn == 128) return tc_launch_bn128_cg2(map_p, map_q, args, grid, stream);
  if (cg == 2 && bn == 256) return tc_launch_bn256_cg2(map_p, map_q, args, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace g10
