// A measurement aid, not part of the GEMM library: the per-launch time of a
// plain streaming read of a buffer from HBM, the floor that any kernel which
// reads those bytes once cannot beat (launch, ramp-up and drain included).
// The benchmark reports it next to the memory-bound GEMMs.  Every thread
// keeps eight 16-byte non-caching loads in flight; the result is folded into
// a value that is stored only in a case that does not occur, so the loads
// cannot be removed.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void hbm_read_kernel(const uint4* __restrict__ p, size_t n16, unsigned* sink) {
  unsigned acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = ld_stream(p + i + j * stride);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u && sink) *sink = acc;
}

}  // namespace

// Reads bytes / 16 16-byte words from p (16-byte aligned device memory) on
// `stream` with grid x 512 threads.  sink: one device word (may be written).
// Returns the CUDA error of the launch (0 = success).
extern "C" int dg_hbm_read_floor(const void* p, size_t bytes, unsigned* sink, int grid, void* stream) {
  if (!p || grid <= 0 || (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return (int)cudaErrorInvalidValue;
  hbm_read_kernel<<<grid, 512, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(p), bytes / 16,
                                                                         sink);
  return (int)cudaGetLastError();
}
