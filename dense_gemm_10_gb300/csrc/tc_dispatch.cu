// tc_dispatch.cu -- choose the kernel instantiation for a tile width.
#include "tc_gemm.cuh"

namespace g10 {

cudaError_t tc_prepare_bn64();
cudaError_t tc_prepare_bn128();
cudaError_t tc_prepare_bn256();
cudaError_t tc_launch_bn64(const CUtensorMap&, const CUtensorMap&, const TcArgs&, int, cudaStream_t);
cudaError_t tc_launch_bn128(const CUtensorMap&, const CUtensorMap&, const TcArgs&, int, cudaStream_t);
cudaError_t tc_launch_bn256(const CUtensorMap&, const CUtensorMap&, const TcArgs&, int, cudaStream_t);

int tc_stages(int bn) {
  return bn == 256 ? TcConfig<256>::kStages : bn == 128 ? TcConfig<128>::kStages : TcConfig<64>::kStages;
}

size_t tc_smem_bytes(int bn) {
  return bn == 256 ? TcConfig<256>::kSmemBytes
                   : bn == 128 ? TcConfig<128>::kSmemBytes : TcConfig<64>::kSmemBytes;
}

cudaError_t tc_prepare(int bn) {
  if (bn == 256) return tc_prepare_bn256();
  if (bn == 128) return tc_prepare_bn128();
  if (bn == 64) return tc_prepare_bn64();
  return cudaErrorInvalidValue;
}

cudaError_t tc_launch(int bn, const CUtensorMap& map_p, const CUtensorMap& map_q,
                      const TcArgs& args, int grid, cudaStream_t stream) {
  if (bn == 256) return tc_launch_bn256(map_p, map_q, args, grid, stream);
  if (bn == 128) return tc_launch_bn128(map_p, map_q, args, grid, stream);
  if (bn == 64) return tc_launch_bn64(map_p, map_q, args, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace g10
