// Tile width 128, one CTA per tile; 16-bit inputs (tcgen05.mma kind::f16).
#define TC_BN 128
#define TC_CG 1
#define TC_EB 2
#include "tc_gemm_inst.cuh"
