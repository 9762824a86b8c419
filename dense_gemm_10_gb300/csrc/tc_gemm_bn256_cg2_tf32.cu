// Tile width 256, a CTA pair per tile (cta_group::2); TF32 inputs (tcgen05.mma kind::tf32), for the fp32 GEMMs.
#define TC_BN 256
#define TC_CG 2
#define TC_EB 4
#include "tc_gemm_inst.cuh"
