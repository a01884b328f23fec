// K-grouped FP8 GEMM (MoE weight gradients, FP32 output) on 128 x 256 tiles
// with eight epilogue warps: each drains 128 columns of one TMEM lane quarter
// into registers, so the tile's single accumulator goes back to the MMA after
// four TMEM loads per warp instead of after half of the FP32 stores.
#include "gemm_kernel.cuh"

namespace dg {

cudaError_t gemm_kgrouped_epi8_launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                                      const CUtensorMap& sfb, const CUtensorMap& d, const GemmArgs& args,
                                      int grid, cudaStream_t stream) {
  if (args.mc) return gemm_launch_impl<256, 4, kKGrouped, 1, kBlockM, true, false, true>(a, b, sfa, sfb, d, args, grid, stream);
  return gemm_launch_impl<256, 4, kKGrouped, 1, kBlockM, true>(a, b, sfa, sfb, d, args, grid, stream);
}

}  // namespace dg
