// Tile width 256, a CTA pair per tile (cta_group::2); 16-bit inputs (tcgen05.mma
// kind::f16); eight epilogue warps, two per tensor-memory lane quarter, each
// storing half of the tile's columns (for C whose rows bulk tensor stores
// cannot write whole, where the epilogue's per-block work is the longer part).
#define TC_BN 256
#define TC_CG 2
#define TC_EB 2
#define TC_EW 8
#include "tc_gemm_inst.cuh"
