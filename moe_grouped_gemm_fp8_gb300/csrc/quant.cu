// FP32 -> E4M3 quantisation with power-of-two fine-grained scales, and the
// FP32 -> packed UE8M0 scale transform.  Memory-bound kernels: every input
// byte is read once with 16-byte coalesced loads and every output byte is
// written once.
//
// Scale rule and layouts: "DeepGEMM: kernels GEMM FP8 limpos e eficientes por
// meio de scaling granular", section "Interface GEMM e restrições de layout"
// (fine-grained scaling; SM100 packed UE8M0, four per 32-bit word, MN-major
// and TMA-aligned) and section "Utilitários e variáveis de ambiente"
// (transform_sf_into_required_layout).
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_device.cuh"

namespace dg {

__device__ unsigned long long g_quant_err = 0ull;

__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float abs_max4(const float4& v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

__device__ __forceinline__ uint32_t quant4(const float4& v, int e) {
  const uint32_t lo = cvt_e4m3x2(scale_down(v.x, e), scale_down(v.y, e));
  const uint32_t hi = cvt_e4m3x2(scale_down(v.z, e), scale_down(v.w, e));
  return lo | (hi << 16);
}

// 1x128 groups.  One warp per (group, row, 512-column pack); lane l handles
// columns 4l .. 4l+3 of each 128-column block.  Warps are ordered row-fastest
// so the packed scale words of consecutive warps are adjacent in memory.
template <bool kPacked>
__global__ void __launch_bounds__(256) quant_rows_kernel(const float* __restrict__ x,
                                                         uint8_t* __restrict__ q,
                                                         void* __restrict__ sf, int64_t groups,
                                                         int64_t rows, int64_t rows_out,
                                                         int64_t cols, int kblocks, int kpacks) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t w = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (w >= groups * rows_out * kpacks) return;
  const int64_t r = w % rows_out;
  const int64_t j = (w / rows_out) % kpacks;
  const int64_t g = w / (rows_out * kpacks);
  uint32_t word = 0;
  if (r < rows) {
    const int64_t row = g * rows + r;
    const float* xr = x + row * cols;
    uint8_t* qr = q + row * cols;
    float4 v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int kb = (int)(4 * j) + t;
      if (kb < kblocks) v[t] = ld_stream_f4(xr + (int64_t)kb * 128 + lane * 4);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int kb = (int)(4 * j) + t;
      if (kb >= kblocks) break;
      const int e = scale_exponent(warp_max(abs_max4(v[t])));
      *reinterpret_cast<uint32_t*>(qr + (int64_t)kb * 128 + lane * 4) = quant4(v[t], e);
      word |= (uint32_t)(e + 127) << (8 * t);
      if (!kPacked && lane == 0) reinterpret_cast<float*>(sf)[row * kblocks + kb] = pow2f(e);
    }
  }
  if (kPacked && lane == 0) reinterpret_cast<int32_t*>(sf)[(g * kpacks + j) * rows_out + r] = (int32_t)word;
}

// 128x128 blocks.  One 256-thread CTA per (group, 128-row block, 512-column
// pack); warp w covers rows w, w+8, ..., lane l columns 4l .. 4l+3.
template <bool kPacked>
__global__ void __launch_bounds__(256) quant_blocks_kernel(const float* __restrict__ x,
                                                           uint8_t* __restrict__ q,
                                                           void* __restrict__ sf, int64_t groups,
                                                           int64_t rows, int64_t rows_pad,
                                                           int64_t cols, int kblocks, int kpacks,
                                                           int64_t rblocks) {
  __shared__ float red[8];
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t j = blockIdx.x % kpacks;
  const int64_t rb = (blockIdx.x / kpacks) % rblocks;
  const int64_t g = blockIdx.x / (kpacks * rblocks);
  const int64_t r0 = rb * 128;
  uint32_t word = 0;
  for (int t = 0; t < 4; ++t) {
    const int kb = (int)(4 * j) + t;
    if (kb >= kblocks) break;
    float4 v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t r = r0 + warp + 8 * i;
      if (r < rows) {
        v[i] = ld_stream_f4(x + (g * rows + r) * cols + (int64_t)kb * 128 + lane * 4);
        amax = fmaxf(amax, abs_max4(v[i]));
      }
    }
    amax = warp_max(amax);
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    __syncthreads();
    const int e = scale_exponent(amax);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t r = r0 + warp + 8 * i;
      if (r < rows)
        *reinterpret_cast<uint32_t*>(q + (g * rows + r) * cols + (int64_t)kb * 128 + lane * 4) =
            quant4(v[i], e);
    }
    word |= (uint32_t)(e + 127) << (8 * t);
    if (!kPacked && threadIdx.x == 0)
      reinterpret_cast<float*>(sf)[(g * rblocks + rb) * kblocks + kb] = pow2f(e);
  }
  if (kPacked) {
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
      const int64_t r = r0 + i;
      if (r < rows_pad)
        reinterpret_cast<int32_t*>(sf)[(g * kpacks + j) * rows_pad + r] =
            (int32_t)(r < rows ? word : 0u);
    }
  }
}

// One scale per 128 rows of each column (operands whose reduction axis is the
// row axis: A and B of the K-grouped GEMM).  Thread i of a CTA handles 4
// adjacent columns over 512 rows (four 128-row blocks = one packed word per
// column); a warp reads 512 contiguous bytes per row.  Each block is read
// twice, once for the column maxima and once to encode (the second read hits
// L2).
template <bool kPacked>
__global__ void __launch_bounds__(128) quant_cols_kernel(const float* __restrict__ x,
                                                         uint8_t* __restrict__ q,
                                                         void* __restrict__ sf, int64_t rows,
                                                         int64_t cols, int64_t cols_pad,
                                                         int rblocks) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  const int j = blockIdx.y;  // 512-row pack
  if (c >= cols_pad) return;
  uint32_t word[4] = {0u, 0u, 0u, 0u};
  if (c < cols) {
    for (int t = 0; t < 4; ++t) {
      const int rb = 4 * j + t;
      if (rb >= rblocks) break;
      const float* xb = x + (int64_t)rb * 128 * cols + c;
      float4 amax = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < 128; ++r) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(xb + (int64_t)r * cols));
        amax.x = fmaxf(amax.x, fabsf(v.x));
        amax.y = fmaxf(amax.y, fabsf(v.y));
        amax.z = fmaxf(amax.z, fabsf(v.z));
        amax.w = fmaxf(amax.w, fabsf(v.w));
      }
      const int e0 = scale_exponent(amax.x), e1 = scale_exponent(amax.y);
      const int e2 = scale_exponent(amax.z), e3 = scale_exponent(amax.w);
      uint8_t* qb = q + (int64_t)rb * 128 * cols + c;
      for (int r = 0; r < 128; ++r) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(xb + (int64_t)r * cols));
        const uint32_t lo = cvt_e4m3x2(scale_down(v.x, e0), scale_down(v.y, e1));
        const uint32_t hi = cvt_e4m3x2(scale_down(v.z, e2), scale_down(v.w, e3));
        *reinterpret_cast<uint32_t*>(qb + (int64_t)r * cols) = lo | (hi << 16);
      }
      word[0] |= (uint32_t)(e0 + 127) << (8 * t);
      word[1] |= (uint32_t)(e1 + 127) << (8 * t);
      word[2] |= (uint32_t)(e2 + 127) << (8 * t);
      word[3] |= (uint32_t)(e3 + 127) << (8 * t);
      if (!kPacked)
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(sf) + (int64_t)rb * cols + c) =
            make_float4(pow2f(e0), pow2f(e1), pow2f(e2), pow2f(e3));
    }
  }
  if (kPacked)
    *reinterpret_cast<uint4*>(reinterpret_cast<int32_t*>(sf) + (int64_t)j * cols_pad + c) =
        make_uint4(word[0], word[1], word[2], word[3]);
}

// Exponent of a power-of-two FP32 scale.  Returns false (and the exponent of
// the next power of two up, or 0 for a non-positive / non-finite value) when
// s is not an exact power of two within 2^-127 .. 2^127.
__device__ __forceinline__ bool pow2_exponent(float s, int* e_out) {
  const uint32_t bits = __float_as_uint(s);
  const uint32_t biased = (bits >> 23) & 0xFFu;
  const uint32_t frac = bits & 0x7FFFFFu;
  if ((bits >> 31) || biased == 255 || (biased == 0 && frac == 0)) {
    *e_out = 0;
    return false;
  }
  if (biased == 0) {  // subnormal: s = frac * 2^-149
    const int top = 31 - __clz(frac);
    const bool exact = (frac & (frac - 1)) == 0;
    int e = top - 149 + (exact ? 0 : 1);
    const bool in_range = e >= -127;
    *e_out = in_range ? e : -127;
    return exact && in_range;
  }
  int e = (int)biased - 127 + (frac ? 1 : 0);
  if (e > 127) e = 127;
  *e_out = e;
  return frac == 0;
}

__global__ void __launch_bounds__(256) transform_sf_kernel(const float* __restrict__ sf,
                                                           int32_t* __restrict__ packed,
                                                           int64_t groups, int64_t mn,
                                                           int64_t mn_pad, int kblocks,
                                                           int kpacks, int block_rows,
                                                           int64_t mn_blocks) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= groups * kpacks * mn_pad) return;
  const int64_t r = idx % mn_pad;
  const int64_t j = (idx / mn_pad) % kpacks;
  const int64_t g = idx / (mn_pad * kpacks);
  uint32_t word = 0;
  if (r < mn) {
    const float* src = sf + (g * mn_blocks + r / block_rows) * kblocks;
    for (int t = 0; t < 4; ++t) {
      const int kb = (int)(4 * j) + t;
      if (kb >= kblocks) break;
      int e;
      if (!pow2_exponent(src[kb], &e)) record_error(&g_quant_err, DG_ERR_DEVICE_BAD_SCALE, kSiteTransformScale);
      word |= (uint32_t)(e + 127) << (8 * t);
    }
  }
  packed[idx] = (int32_t)word;
}

static inline int64_t align4(int64_t x) { return (x + 3) / 4 * 4; }

// Launches with programmatic stream serialisation when pdl is set.
template <class Kern, class... Args>
static cudaError_t launch(Kern kern, dim3 grid, unsigned threads, bool pdl, cudaStream_t stream,
                          Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t quantize_launch(const float* x, void* q, void* sf, int64_t groups, int64_t rows,
                            int64_t cols, int block_rows, int sf_format, bool pdl,
                            cudaStream_t stream) {
  const int kblocks = (int)(cols / 128);
  const int kpacks = (kblocks + 3) / 4;
  const bool packed = sf_format == DG_SF_UE8M0_PACKED;
  if (block_rows == 1) {
    const int64_t rows_out = packed ? align4(rows) : rows;
    const int64_t warps = groups * rows_out * kpacks;
    const int64_t blocks = (warps + 7) / 8;
    return launch(packed ? quant_rows_kernel<true> : quant_rows_kernel<false>, dim3((unsigned)blocks),
                  256, pdl, stream, x, (uint8_t*)q, sf, groups, rows, rows_out, cols, kblocks, kpacks);
  } else {
    const int64_t rblocks = (rows + 127) / 128;
    const int64_t blocks = groups * rblocks * kpacks;
    return launch(packed ? quant_blocks_kernel<true> : quant_blocks_kernel<false>,
                  dim3((unsigned)blocks), 256, pdl, stream, x, (uint8_t*)q, sf, groups, rows,
                  align4(rows), cols, kblocks, kpacks, rblocks);
  }
}

cudaError_t quantize_cols_launch(const float* x, void* q, void* sf, int64_t rows, int64_t cols,
                                 int sf_format, bool pdl, cudaStream_t stream) {
  const int rblocks = (int)(rows / 128);
  const int kpacks = (rblocks + 3) / 4;
  const int64_t cols_pad = align4(cols);
  const int64_t threads = cols_pad / 4;
  const dim3 grid((unsigned)((threads + 127) / 128), (unsigned)kpacks);
  return launch(sf_format == DG_SF_UE8M0_PACKED ? quant_cols_kernel<true> : quant_cols_kernel<false>,
                grid, 128, pdl, stream, x, (uint8_t*)q, sf, rows, cols, cols_pad, rblocks);
}

cudaError_t transform_sf_launch(const float* sf, int32_t* packed, int64_t groups, int64_t mn,
                                int64_t k, int block_rows, bool pdl, cudaStream_t stream) {
  const int kblocks = (int)((k + 127) / 128);
  const int kpacks = (kblocks + 3) / 4;
  const int64_t mn_pad = align4(mn);
  const int64_t mn_blocks = (mn + block_rows - 1) / block_rows;
  const int64_t total = groups * kpacks * mn_pad;
  const int64_t blocks = (total + 255) / 256;
  return launch(transform_sf_kernel, dim3((unsigned)blocks), 256, pdl, stream, sf, packed, groups,
                mn, mn_pad, kblocks, kpacks, block_rows, mn_blocks);
}

cudaError_t quant_fetch_error(unsigned long long* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_quant_err, sizeof(*word));
  if (e != cudaSuccess) return e;
  const unsigned long long zero = 0ull;
  return cudaMemcpyToSymbol(g_quant_err, &zero, sizeof(zero));
}

}  // namespace dg
