// Tile width 128, one CTA per tile; TF32 inputs (tcgen05.mma kind::tf32), for the fp32 GEMMs.
#define TC_BN 128
#define TC_CG 1
#define TC_EB 4
#include "tc_gemm_inst.cuh"
