// FP8 GEMM kernels on CTA pairs, 256 x 192 output tiles (6-stage pipeline).
#include "gemm2_kernel.cuh"

DG_DEFINE_GEMM2_BN(192, 6)
