// FP8 GEMM kernels with 192-column output tiles (4-stage pipeline).
#include "gemm_kernel.cuh"

DG_DEFINE_GEMM_BN(192, 4)
