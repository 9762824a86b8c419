// Tile width 64, CTA group 2, 1 CTA pair(s) sharing P by multicast.
#define TC_BN 64
#define TC_CG 2
#define TC_MC 1
#include "tc_gemm_inst.cuh"
