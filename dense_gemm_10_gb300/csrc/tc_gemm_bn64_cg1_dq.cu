// Tile width 64, one CTA per tile; 16-bit MMA inputs (tcgen05.mma kind::f16)
// whose P operand arrives as block-scaled codes (NVFP4, MXFP8) and is
// converted in the kernel by four more warps.
#define TC_BN 64
#define TC_CG 1
#define TC_EB 2
#define TC_DQ 1
#include "tc_gemm_inst.cuh"
