// Tile width 256, CTA group 2, 2 CTA pair(s) per cluster sharing P by multicast;
// 16-bit inputs (tcgen05.mma kind::f16).
#define TC_BN 256
#define TC_CG 2
#define TC_MC 2
#define TC_EB 2
#include "tc_gemm_inst.cuh"
