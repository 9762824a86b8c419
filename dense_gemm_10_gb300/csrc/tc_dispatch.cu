// tc_dispatch.cu -- the table of kernel instantiations, one per tile
// configuration (each compiled in its own translation unit).
#include "tc_gemm.cuh"

namespace g10 {

using PrepareFn = cudaError_t (*)(int*);
using LaunchFn = cudaError_t (*)(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CMaps&,
                                 const TcArgs&, int, cudaStream_t);

#define TC_DECLARE(BN, CG, EB, DQ, EW)                                                              \
  cudaError_t tc_prepare_bn##BN##_cg##CG##_eb##EB##_dq##DQ##_ew##EW(int* max_clusters);                \
  cudaError_t tc_launch_bn##BN##_cg##CG##_eb##EB##_dq##DQ##_ew##EW(const CUtensorMap&, const CUtensorMap&, \
                                                                 const CUtensorMap&, const CMaps&,       \
                                                                 const TcArgs&, int, cudaStream_t);
#define TC_ENTRY(BN, CG, EB, DQ, EW)                                                                \
  {{BN, CG, EB, DQ, EW}, TcConfig<BN, CG, DQ != 0, EW>::kStages, TcConfig<BN, CG, DQ != 0, EW>::kCodeRingBytes, \
   tc_prepare_bn##BN##_cg##CG##_eb##EB##_dq##DQ##_ew##EW, tc_launch_bn##BN##_cg##CG##_eb##EB##_dq##DQ##_ew##EW}

TC_DECLARE(64, 1, 2, 0, 4)
TC_DECLARE(128, 1, 2, 0, 4)
TC_DECLARE(256, 1, 2, 0, 4)
TC_DECLARE(128, 2, 2, 0, 4)
TC_DECLARE(256, 2, 2, 0, 4)
TC_DECLARE(64, 2, 2, 0, 4)
TC_DECLARE(64, 1, 1, 0, 4)
TC_DECLARE(128, 1, 1, 0, 4)
TC_DECLARE(128, 2, 1, 0, 4)
TC_DECLARE(256, 2, 1, 0, 4)
TC_DECLARE(64, 1, 4, 0, 4)
TC_DECLARE(128, 1, 4, 0, 4)
TC_DECLARE(256, 2, 4, 0, 4)
TC_DECLARE(64, 1, 2, 1, 4)
TC_DECLARE(256, 2, 2, 0, 8)

namespace {
struct Entry {
  TileConfig cfg;
  int stages;
  int code_ring_bytes;
  PrepareFn prepare;
  LaunchFn launch;
};
const Entry kEntries[kNumTileConfigs] = {
    TC_ENTRY(64, 1, 2, 0, 4),
    TC_ENTRY(128, 1, 2, 0, 4),
    TC_ENTRY(256, 1, 2, 0, 4),
    TC_ENTRY(128, 2, 2, 0, 4),
    TC_ENTRY(256, 2, 2, 0, 4),
    TC_ENTRY(64, 2, 2, 0, 4),
    TC_ENTRY(64, 1, 1, 0, 4),
    TC_ENTRY(128, 1, 1, 0, 4),
    TC_ENTRY(128, 2, 1, 0, 4),
    TC_ENTRY(256, 2, 1, 0, 4),
    TC_ENTRY(64, 1, 4, 0, 4),
    TC_ENTRY(128, 1, 4, 0, 4),
    TC_ENTRY(256, 2, 4, 0, 4),
    TC_ENTRY(64, 1, 2, 1, 4),
    TC_ENTRY(256, 2, 2, 0, 8)};
}  // namespace

// (entry 13: 64-wide tiles whose P arrives as block-scaled codes, converted in
// the kernel; entry 14: the 256-wide CTA-pair 16-bit tile with eight epilogue
// warps, taken for C that bulk tensor stores cannot write whole)
const TileConfig kTileConfigs[kNumTileConfigs] = {
    {64, 1, 2, 0, 4},
    {128, 1, 2, 0, 4},
    {256, 1, 2, 0, 4},
    {128, 2, 2, 0, 4},
    {256, 2, 2, 0, 4},
    {64, 2, 2, 0, 4},
    {64, 1, 1, 0, 4},
    {128, 1, 1, 0, 4},
    {128, 2, 1, 0, 4},
    {256, 2, 1, 0, 4},
    {64, 1, 4, 0, 4},
    {128, 1, 4, 0, 4},
    {256, 2, 4, 0, 4},
    {64, 1, 2, 1, 4},
    {256, 2, 2, 0, 8}};

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
