// Tile width 64 of the persistent tcgen05 GEMM kernel.
#define TC_BN 64
#include "tc_gemm_inst.cuh"
