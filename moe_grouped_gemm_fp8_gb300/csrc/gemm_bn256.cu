// FP8 GEMM kernels with 256-column output tiles (4-stage pipeline).
#include "gemm_kernel.cuh"

DG_DEFINE_GEMM_BN(256, 4)
