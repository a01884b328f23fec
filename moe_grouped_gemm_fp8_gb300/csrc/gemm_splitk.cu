// Dense FP8 GEMM with split-K over a cluster of 2 or 4 CTAs (128-column
// tiles): for problems with fewer output tiles than SMs, such as decode-sized
// M.  The partial sums are reduced through distributed shared memory.
#include "gemm_kernel.cuh"

namespace dg {

cudaError_t gemm_splitk_launch(int ksplit, const CUtensorMap& a, const CUtensorMap& b,
                               const CUtensorMap& sfa, const CUtensorMap& sfb,
                               const CUtensorMap& d, GemmArgs args, int clusters,
                               cudaStream_t stream) {
  if (clusters <= 0) return cudaErrorInvalidValue;
  if (ksplit == 2)
    return gemm_launch_impl<128, 5, kDense, 2>(a, b, sfa, sfb, d, args, 2 * clusters, stream);
  if (ksplit == 4)
    return gemm_launch_impl<128, 4, kDense, 4>(a, b, sfa, sfb, d, args, 4 * clusters, stream);
  return cudaErrorInvalidValue;
}

int gemm_splitk_max_clusters(int ksplit) {
  static int cache[64][2];
  static bool filled[64][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int i = ksplit == 2 ? 0 : 1;
  if (!filled[dev][i]) {
    cache[dev][i] = ksplit == 2 ? gemm_splitk_max_clusters_impl<128, 5, 2>()
                                : gemm_splitk_max_clusters_impl<128, 4, 4>();
    filled[dev][i] = true;
  }
  return cache[dev][i];
}

}  // namespace dg
