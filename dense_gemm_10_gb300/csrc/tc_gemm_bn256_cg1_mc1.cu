// Tile width 256, CTA group 1, 1 CTA pair(s) sharing P by multicast.
#define TC_BN 256
#define TC_CG 1
#define TC_MC 1
#include "tc_gemm_inst.cuh"
