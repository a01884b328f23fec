// Dense FP8 GEMM with split-K over a cluster of 2 or 4 CTAs (128-column
// tiles): for problems with fewer output tiles than SMs, such as decode-sized
// M.  The partial sums are reduced through distributed shared memory.
#include <atomic>

#include "gemm_kernel.cuh"

namespace dg {

// short_a: M <= 64, so the A slot of a stage holds 64 rows (8 KB instead of
// 16) and two more stages fit.
constexpr int kSplit2Stages = 5, kSplit4Stages = 4, kSplit2ShortStages = 7, kSplit4ShortStages = 6;
int gemm_splitk_stages(int ksplit, bool short_a) {
  if (ksplit == 2) return short_a ? kSplit2ShortStages : kSplit2Stages;
  if (ksplit == 4) return short_a ? kSplit4ShortStages : kSplit4Stages;
  return 0;
}

cudaError_t gemm_splitk_launch(int ksplit, bool short_a, const CUtensorMap& a, const CUtensorMap& b,
                               const CUtensorMap& sfa, const CUtensorMap& sfb,
                               const CUtensorMap& d, GemmArgs args, int clusters,
                               cudaStream_t stream) {
  if (clusters <= 0) return cudaErrorInvalidValue;
  unsigned long long* err = nullptr;
  cudaError_t e = error_word_address(&err);
  if (e != cudaSuccess) return e;
  args.err = err;
  constexpr int kShort = kBlockM / 2;
  if (ksplit == 2)
    return short_a ? gemm_launch_impl<128, kSplit2ShortStages, kDense, 2, kShort>(a, b, sfa, sfb, d, args, 2 * clusters, stream)
                   : gemm_launch_impl<128, kSplit2Stages, kDense, 2>(a, b, sfa, sfb, d, args, 2 * clusters, stream);
  if (ksplit == 4)
    return short_a ? gemm_launch_impl<128, kSplit4ShortStages, kDense, 4, kShort>(a, b, sfa, sfb, d, args, 4 * clusters, stream)
                   : gemm_launch_impl<128, kSplit4Stages, kDense, 4>(a, b, sfa, sfb, d, args, 4 * clusters, stream);
  return cudaErrorInvalidValue;
}

int gemm_splitk_max_clusters(int ksplit) {
  // cached per (device, factor) as count + 1 (0: not yet queried); racing
  // callers store the same value
  static std::atomic<int> cache[64][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int i = ksplit == 2 ? 0 : 1;
  int c = cache[dev][i].load(std::memory_order_relaxed);
  if (c == 0) {
    c = 1 + (ksplit == 2 ? gemm_splitk_max_clusters_impl<128, kSplit2Stages, 2>()
                         : gemm_splitk_max_clusters_impl<128, kSplit4Stages, 4>());
    cache[dev][i].store(c, std::memory_order_relaxed);
  }
  return c - 1;
}

}  // namespace dg
