// Tile-width dispatch and the device error word of the GEMM kernels.
#include <cuda_runtime.h>

#include "dg_internal.h"

namespace dg {

__device__ unsigned long long g_gemm_err = 0ull;

int gemm_stages(int block_n) {
  switch (block_n) {
    case 128: return gemm_stages_bn128();
    case 192: return gemm_stages_bn192();
    case 224: return gemm_stages_bn224();
    case 256: return gemm_stages_bn256();
  }
  return 0;
}

bool gemm_block_n_supported(int block_n) { return gemm_stages(block_n) > 0; }

cudaError_t gemm_launch(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                        GemmArgs args, int grid, cudaStream_t stream) {
  // Host code must pass the device address of the error word, not the
  // host-side shadow the symbol name denotes here.
  void* err = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&err, g_gemm_err);
  if (e != cudaSuccess) return e;
  args.err = static_cast<unsigned long long*>(err);
  switch (block_n) {
    case 128: return gemm_launch_bn128(mode, a, b, sfa, sfb, d, args, grid, stream);
    case 192: return gemm_launch_bn192(mode, a, b, sfa, sfb, d, args, grid, stream);
    case 224: return gemm_launch_bn224(mode, a, b, sfa, sfb, d, args, grid, stream);
    case 256: return gemm_launch_bn256(mode, a, b, sfa, sfb, d, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t gemm_fetch_error(unsigned long long* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_gemm_err, sizeof(*word));
  if (e != cudaSuccess) return e;
  const unsigned long long zero = 0ull;
  return cudaMemcpyToSymbol(g_gemm_err, &zero, sizeof(zero));
}

}  // namespace dg
