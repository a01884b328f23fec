// FP8 GEMM kernels with 192-column output tiles (5-stage pipeline).
#include "gemm_kernel.cuh"

DG_DEFINE_GEMM_BN(192, 5)
