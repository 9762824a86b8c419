// Tile width 128, CTA group 2, 1 CTA pair(s) sharing P by multicast.
#define TC_BN 128
#define TC_CG 2
#define TC_MC 1
#include "tc_gemm_inst.cuh"
