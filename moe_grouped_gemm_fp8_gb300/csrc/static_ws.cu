// dg_fp8_gemm_nt_static_ws: the stream-K dense GEMM for callers that cannot
// allocate device memory.  Its workspace is a file-scope device array that
// exists from the moment the library is loaded; nothing is allocated or freed
// here, by this library or by any other.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "dg_internal.h"

namespace dg {
namespace {

// Scratch of dg_fp8_gemm_nt_static_ws: 32 KiB of stream-K flags, then one
// FP32 partial-sum slot of 256 x block_n values per SM.  32 MiB holds the
// 192-column tiles' slots for up to 165 SMs (the 224-column ones for up to
// 145).  Zero-initialised when the module is loaded; held by every device
// that loads the library until the process exits.
constexpr uint64_t kStaticWsBytes = (uint64_t)32 << 20;
constexpr uint64_t kStaticWsFlagBytes = (uint64_t)32 << 10;  // the flags that must start at zero
__device__ __align__(256) static unsigned char g_static_ws[kStaticWsBytes];

// Device address of g_static_ws on the current device.  In host code the
// symbol names a host-side stand-in, never a device address, so the address
// is looked up with cudaGetSymbolAddress, once per device, with that device
// current.
cudaError_t static_ws_address(void** out) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* p = addr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return e;
    addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace dg

extern "C" {

dg_status dg_fp8_gemm_nt_static_ws(const void* a, const int32_t* sfa, const void* b,
                                   const int32_t* sfb, const void* c, void* d, int64_t m,
                                   int64_t n, int64_t k, int64_t lda, int64_t ldb, int64_t ldc,
                                   int64_t ldd, void* stream) {
  // Scratch this problem needs on the SMs the call will use (0: the
  // tile-by-tile walk, which needs none).  Shape errors are reported here.
  uint64_t need = 0;
  const int32_t sms = dg_get_num_sms();
  if (sms < 1) return DG_ERR_CUDA;
  dg_status s = dg_fp8_gemm_nt_workspace_size(m, n, k, c != nullptr, sms, &need);
  if (s != DG_OK) return s;
  if (need > dg::kStaticWsBytes) return DG_ERR_TOO_LARGE;
  if (m == 0 || n == 0) return DG_OK;
  void* ws = nullptr;
  if (dg::static_ws_address(&ws) != cudaSuccess) return DG_ERR_CUDA;
  // The flags must be zero when a launch starts.  Every launch leaves them
  // zero, but one that ran out of time may not have, so they are cleared
  // (stream-ordered) before each call.
  if (need > 0 &&
      cudaMemsetAsync(ws, 0, dg::kStaticWsFlagBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DG_ERR_CUDA;
  return dg_fp8_gemm_nt_ws(a, sfa, b, sfb, c, d, m, n, k, lda, ldb, ldc, ldd, ws,
                           dg::kStaticWsBytes, stream);
}

}  // extern "C"
