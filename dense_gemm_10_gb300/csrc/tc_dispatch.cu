// tc_dispatch.cu -- the table of kernel instantiations, one per tile
// configuration (each compiled in its own translation unit).
#include "tc_gemm.cuh"

namespace g10 {

using PrepareFn = cudaError_t (*)(int*);
using LaunchFn = cudaError_t (*)(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CMaps&,
                                 const TcArgs&, int, cudaStream_t);

#define TC_DECLARE(BN, CG, EB, DQ)                                                                \
  cudaError_t tc_prepare_bn##BN##_cg##CG##_eb##EB##_dq##DQ(int* max_clusters);                    \
  cudaError_t tc_launch_bn##BN##_cg##CG##_eb##EB##_dq##DQ(const CUtensorMap&, const CUtensorMap&,   \
                                                          const CUtensorMap&, const CMaps&,          \
                                                          const TcArgs&, int, cudaStream_t);
#define TC_ENTRY(BN, CG, EB, DQ)                                                                  \
  {{BN, CG, EB, DQ}, TcConfig<BN, CG, DQ != 0>::kStages, TcConfig<BN, CG, DQ != 0>::kCodeRingBytes,      \
   tc_prepare_bn##BN##_cg##CG##_eb##EB##_dq##DQ, tc_launch_bn##BN##_cg##CG##_eb##EB##_dq##DQ}

TC_DECLARE(64, 1, 2, 0)
TC_DECLARE(128, 1, 2, 0)
TC_DECLARE(256, 1, 2, 0)
TC_DECLARE(128, 2, 2, 0)
TC_DECLARE(256, 2, 2, 0)
TC_DECLARE(64, 2, 2, 0)
TC_DECLARE(64, 1, 1, 0)
TC_DECLARE(128, 1, 1, 0)
TC_DECLARE(128, 2, 1, 0)
TC_DECLARE(256, 2, 1, 0)
TC_DECLARE(64, 1, 4, 0)
TC_DECLARE(128, 1, 4, 0)
TC_DECLARE(256, 2, 4, 0)
TC_DECLARE(64, 1, 2, 1)

namespace {
struct Entry {
  TileConfig cfg;
  int stages;
  int code_ring_bytes;
  PrepareFn prepare;
  LaunchFn launch;
};
const Entry kEntries[kNumTileConfigs] = {
    TC_ENTRY(64, 1, 2, 0),  TC_ENTRY(128, 1, 2, 0), TC_ENTRY(256, 1, 2, 0), TC_ENTRY(128, 2, 2, 0),
    TC_ENTRY(256, 2, 2, 0), TC_ENTRY(64, 2, 2, 0),  TC_ENTRY(64, 1, 1, 0),  TC_ENTRY(128, 1, 1, 0),
    TC_ENTRY(128, 2, 1, 0), TC_ENTRY(256, 2, 1, 0), TC_ENTRY(64, 1, 4, 0),  TC_ENTRY(128, 1, 4, 0),
    TC_ENTRY(256, 2, 4, 0), TC_ENTRY(64, 1, 2, 1)};
}  // namespace

// (the last: 64-wide tiles whose P arrives as block-scaled codes, converted in the kernel)
const TileConfig kTileConfigs[kNumTileConfigs] = {
    {64, 1, 2, 0},  {128, 1, 2, 0}, {256, 1, 2, 0}, {128, 2, 2, 0}, {256, 2, 2, 0}, {64, 2, 2, 0}, {64, 1, 1, 0},
    {128, 1, 1, 0}, {128, 2, 1, 0}, {256, 2, 1, 0}, {64, 1, 4, 0},  {128, 1, 4, 0}, {256, 2, 4, 0}, {64, 1, 2, 1}};

int tc_stages(int cfg) { return cfg >= 0 && cfg < kNumTileConfigs ? kEntries[cfg].stages : 0; }

int tc_code_ring_bytes(int cfg) { return cfg >= 0 && cfg < kNumTileConfigs ? kEntries[cfg].code_ring_bytes : 0; }

cudaError_t tc_prepare(int cfg, int* max_clusters) {
  *max_clusters = 0;
  if (cfg < 0 || cfg >= kNumTileConfigs) return cudaErrorInvalidValue;
  return kEntries[cfg].prepare(max_clusters);
}

cudaError_t tc_launch(int cfg, const CUtensorMap& map_p, const CUtensorMap& map_q,
                      const CUtensorMap& map_c, const CMaps& cmaps, const TcArgs& args, int grid,
                      cudaStream_t stream) {
  if (cfg < 0 || cfg >= kNumTileConfigs) return cudaErrorInvalidValue;
  return kEntries[cfg].launch(map_p, map_q, map_c, cmaps, args, grid, stream);
}

}  // namespace g10
