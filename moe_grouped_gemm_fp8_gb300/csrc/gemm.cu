// Tile-width dispatch and the device error word of the GEMM kernels.
#include <cuda_runtime.h>

#include <atomic>

#include "dg_internal.h"

namespace dg {

__device__ unsigned long long g_gemm_err = 0ull;

// Device address of the error word on the current device.  Host code must
// pass this address, not the host-side shadow the symbol name denotes here;
// looked up once per device.
cudaError_t error_word_address(unsigned long long** out) {
  // host threads may call concurrently: the cache is atomic (a lookup that
  // races another stores the same address)
  static std::atomic<unsigned long long*> addr[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  unsigned long long* a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gemm_err);
    if (e != cudaSuccess) return e;
    a = static_cast<unsigned long long*>(p);
    addr[dev].store(a, std::memory_order_release);
  }
  *out = a;
  return cudaSuccess;
}

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
  unsigned long long* err = nullptr;
  cudaError_t e = error_word_address(&err);
  if (e != cudaSuccess) return e;
  args.err = err;
  if (mode == kKGrouped && block_n == 256 && args.epi8)
    return gemm_kgrouped_epi8_launch(a, b, sfa, sfb, d, args, grid, stream);
  switch (block_n) {
    case 128: return gemm_launch_bn128(mode, a, b, sfa, sfb, d, args, grid, stream);
    case 192: return gemm_launch_bn192(mode, a, b, sfa, sfb, d, args, grid, stream);
    case 224: return gemm_launch_bn224(mode, a, b, sfa, sfb, d, args, grid, stream);
    case 256: return gemm_launch_bn256(mode, a, b, sfa, sfb, d, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t gemm_tall_launch(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                             const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                             GemmArgs args, int grid, cudaStream_t stream) {
  unsigned long long* err = nullptr;
  cudaError_t e = error_word_address(&err);
  if (e != cudaSuccess) return e;
  args.err = err;
  return gemm_tall_launch_impl(mode, block_n, a, b, sfa, sfb, d, args, grid, stream);
}

cudaError_t gemm_short_launch(int block_n, const CUtensorMap& a, const CUtensorMap& b,
                              const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                              GemmArgs args, int grid, cudaStream_t stream) {
  unsigned long long* err = nullptr;
  cudaError_t e = error_word_address(&err);
  if (e != cudaSuccess) return e;
  args.err = err;
  return gemm_short_launch_impl(block_n, a, b, sfa, sfb, d, args, grid, stream);
}

bool gemm2_block_n_supported(int block_n) {
  return block_n == 192 || block_n == 224 || block_n == 256;
}

int gemm2_max_clusters(int mode, int block_n) {
  // cached per (device, mode, width) as count + 1 (0: not yet queried); the
  // occupancy query is host-side only, and racing callers store the same value
  static std::atomic<int> cache[64][3][3];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int wi = block_n == 192 ? 0 : (block_n == 224 ? 1 : 2);
  int c = cache[dev][mode][wi].load(std::memory_order_relaxed);
  if (c == 0) {
    int n = 0;
    switch (block_n) {
      case 192: n = gemm2_max_clusters_bn192(mode); break;
      case 224: n = gemm2_max_clusters_bn224(mode); break;
      case 256: n = gemm2_max_clusters_bn256(mode); break;
    }
    c = n + 1;
    cache[dev][mode][wi].store(c, std::memory_order_relaxed);
  }
  return c - 1;
}

cudaError_t gemm2_launch(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                         const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                         GemmArgs args, int clusters, cudaStream_t stream) {
  unsigned long long* err = nullptr;
  cudaError_t e = error_word_address(&err);
  if (e != cudaSuccess) return e;
  args.err = err;
  switch (block_n) {
    case 192: return gemm2_launch_bn192(mode, a, b, sfa, sfb, d, args, clusters, stream);
    case 224: return gemm2_launch_bn224(mode, a, b, sfa, sfb, d, args, clusters, stream);
    case 256: return gemm2_launch_bn256(mode, a, b, sfa, sfb, d, args, clusters, stream);
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
