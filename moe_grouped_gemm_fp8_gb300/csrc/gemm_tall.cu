// FP8 GEMM kernels with 256-row output tiles for the dense NT and the
// M-grouped contiguous forms: two 128-row MMAs per K step share the B tile,
// so each K block moves 32 KB of A and BN x 128 bytes of B for twice the work
// of a 128-row tile (3-stage pipeline, one TMEM accumulator of 2 x BN
// columns).  Contiguous tiles pair two 128-row blocks of one group.  Dense
// tiles walked tile by tile run in clusters of two CTAs on adjacent 256-row
// blocks that share each B tile through TMA multicast.
#include "gemm_kernel.cuh"

namespace dg {

int gemm_tall_stages(int block_n) { return (block_n == 192 || block_n == 224) ? 3 : 0; }

// Dense NT with a single M block of at most 64 rows (decode): 64-row A slots,
// so 8 (BN = 128) or 6 (BN = 192) stages instead of 6 and 4.
constexpr int kShortStages128 = 8, kShortStages192 = 6;
int gemm_short_stages(int block_n) {
  return block_n == 128 ? kShortStages128 : block_n == 192 ? kShortStages192 : 0;
}
bool gemm_short_supported(int block_n) { return gemm_short_stages(block_n) > 0; }

cudaError_t gemm_short_launch_impl(int block_n, const CUtensorMap& a, const CUtensorMap& b,
                                   const CUtensorMap& sfa, const CUtensorMap& sfb,
                                   const CUtensorMap& d, const GemmArgs& args, int grid,
                                   cudaStream_t stream) {
  constexpr int BM = kBlockM / 2;
  switch (block_n) {
    case 128: return gemm_launch_impl<128, kShortStages128, kDense, 1, BM>(a, b, sfa, sfb, d, args, grid, stream);
    case 192: return gemm_launch_impl<192, kShortStages192, kDense, 1, BM>(a, b, sfa, sfb, d, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t gemm_tall_launch_impl(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                                  const CUtensorMap& sfa, const CUtensorMap& sfb,
                                  const CUtensorMap& d, const GemmArgs& args, int grid,
                                  cudaStream_t stream) {
  constexpr int BM = 2 * kBlockM;
  if (mode == kDense && args.sk_units > 0) {
    switch (block_n) {
      case 192: return gemm_launch_impl<192, 3, kDense, 1, BM, true, true>(a, b, sfa, sfb, d, args, grid, stream);
      case 224: return gemm_launch_impl<224, 3, kDense, 1, BM, true, true>(a, b, sfa, sfb, d, args, grid, stream);
    }
  } else if (mode == kDense && args.epi8 && args.mc) {
    switch (block_n) {
      case 192: return gemm_launch_impl<192, 3, kDense, 1, BM, true, false, true>(a, b, sfa, sfb, d, args, grid, stream);
      case 224: return gemm_launch_impl<224, 3, kDense, 1, BM, true, false, true>(a, b, sfa, sfb, d, args, grid, stream);
    }
  } else if (mode == kDense && args.epi8) {
    switch (block_n) {
      case 192: return gemm_launch_impl<192, 3, kDense, 1, BM, true>(a, b, sfa, sfb, d, args, grid, stream);
      case 224: return gemm_launch_impl<224, 3, kDense, 1, BM, true>(a, b, sfa, sfb, d, args, grid, stream);
    }
  } else if (mode == kDense) {
    switch (block_n) {
      case 192: return gemm_launch_impl<192, 3, kDense, 1, BM>(a, b, sfa, sfb, d, args, grid, stream);
      case 224: return gemm_launch_impl<224, 3, kDense, 1, BM>(a, b, sfa, sfb, d, args, grid, stream);
    }
  } else if (mode == kContiguous) {
    switch (block_n) {
      case 192: return gemm_launch_impl<192, 3, kContiguous, 1, BM>(a, b, sfa, sfb, d, args, grid, stream);
      case 224: return gemm_launch_impl<224, 3, kContiguous, 1, BM>(a, b, sfa, sfb, d, args, grid, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
