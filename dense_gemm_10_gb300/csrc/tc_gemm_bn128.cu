// Tile width 128 of the persistent tcgen05 GEMM kernel.
#define TC_BN 128
#include "tc_gemm_inst.cuh"
