// Tile width 128, a CTA pair per tile (cta_group::2); 8-bit float inputs (tcgen05.mma kind::f8f6f4).
#define TC_BN 128
#define TC_CG 2
#define TC_EB 1
#include "tc_gemm_inst.cuh"
