// FP8 GEMM kernels with 128-column output tiles (6-stage pipeline).
#include "gemm_kernel.cuh"

DG_DEFINE_GEMM_BN(128, 6)
