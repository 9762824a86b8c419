// Tile width 256, CTA group 2 of the persistent tcgen05 GEMM kernel.
#define TC_BN 256
#define TC_CG 2
#include "tc_gemm_inst.cuh"
