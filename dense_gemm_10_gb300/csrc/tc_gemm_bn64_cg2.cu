// Tile width 64, a CTA pair per tile (cta_group::2); 16-bit inputs (tcgen05.mma kind::f16).
#define TC_BN 64
#define TC_CG 2
#define TC_EB 2
#include "tc_gemm_inst.cuh"
