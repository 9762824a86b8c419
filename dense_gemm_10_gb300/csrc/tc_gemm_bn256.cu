// Tile width 256 of the persistent tcgen05 GEMM kernel.
#define TC_BN 256
#include "tc_gemm_inst.cuh"
