// Tile width 256, CTA group 1 of the persistent tcgen05 GEMM kernel.
#define TC_BN 256
#define TC_CG 1
#include "tc_gemm_inst.cuh"
