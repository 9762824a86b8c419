// Tile width 64, CTA group 1, TF32 inputs (tcgen05.mma kind::tf32), for the
// fp32 GEMM emulated with split TF32 operands.
#define TC_BN 64
#define TC_CG 1
#define TC_MC 1
#define TC_EB 4
#include "tc_gemm_inst.cuh"
