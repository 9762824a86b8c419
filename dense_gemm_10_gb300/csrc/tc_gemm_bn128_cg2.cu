// Tile width 128, CTA group 2 of the persistent tcgen05 GEMM kernel.
#define TC_BN 128
#define TC_CG 2
#include "tc_gemm_inst.cuh"
