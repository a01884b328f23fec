// Declarations shared by the translation units of libdg.so (not part of the
// public C ABI, which is include/dg.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg.h"

namespace dg {

constexpr int kBlockM = 128;  // rows of an output tile (UMMA M)
constexpr int kBlockK = 128;  // K extent of one scale block / pipeline stage
constexpr int kMaxMaskedGroups = 512;

// kKGrouped: experts stacked along K (weight gradients), MN-major operands,
// FP32 output [G, M, N].  kDense is the NT layout; kDenseNN / TN / TT are the
// same dense GEMM with B, both, or A stored MN-major.
enum GemmMode : int {
  kDense = 0,
  kContiguous = 1,
  kMasked = 2,
  kKGrouped = 3,
  kDenseNN = 4,
  kDenseTN = 5,
  kDenseTT = 6,
};
__host__ __device__ constexpr bool is_dense_mode(int mode) {
  return mode == kDense || mode == kDenseNN || mode == kDenseTN || mode == kDenseTT;
}
// A stored [K, M] (M innermost) / B stored [K, N] (N innermost)
__host__ __device__ constexpr bool a_mn_major(int mode) {
  return mode == kDenseTN || mode == kDenseTT || mode == kKGrouped;
}
__host__ __device__ constexpr bool b_mn_major(int mode) {
  return mode == kDenseNN || mode == kDenseTN || mode == kKGrouped;
}

// Sites recorded with device errors (bits 8-23 of the error word).
enum ErrorSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaTmemEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpilogueTmemFull = 4,
  kSiteDrain = 5,
  kSiteProducerDrain = 6,
  kSiteScaleFull = 7,
  kSiteMmaScaleReady = 8,
  kSiteScaleEmpty = 9,
  kSiteSplitFree = 10,
  kSiteSplitFull = 11,
  kSiteStreamKPartial = 12,
  // debug-build checks (DG_DEBUG_CHECKS)
  kSiteCheckLoadA = 40,
  kSiteCheckLoadB = 41,
  kSiteCheckScale = 42,
  kSiteCheckTmem = 43,
  kSiteCheckStore = 44,
  kSiteCheckStreamK = 45,
  kSiteContiguousIndex = 16,
  kSiteMaskedCount = 17,
  kSiteKGroupSize = 18,
  kSiteTransformScale = 32,
};

struct GemmArgs {
  const __nv_bfloat16* c;  // nullable
  __nv_bfloat16* d;
  int64_t ldc, ldd;        // elements
  const int32_t* m_indices;
  const int32_t* masked_m;
  int32_t m;               // dense M, contiguous m_sum, masked max_m
  int32_t n, k;
  int32_t num_groups;
  int32_t m_blocks;        // ceil(m / 128)
  int32_t n_blocks;
  int32_t k_blocks;
  int32_t band;            // raster band height in M blocks
  int32_t a_box_rows;      // rows of A per TMA box when M < 128 (dense), 0 = 128
  uint64_t timeout_ns;
  unsigned long long* err; // device error word
  // K-grouped form only
  const int32_t* ks;       // rows per expert along K, [num_groups]
  const float* c_f32;      // nullable, [num_groups, m, n]
  float* d_f32;            // [num_groups, m, n]
  int32_t pdl;             // host side: launch with programmatic stream serialisation
  // Test hook (dg_debug_set_drop_load): 1 + the K block whose operand copies CTA 0
  // skips on its first tile, so that stage's barrier never completes and the
  // bounded waits must end the launch with DG_ERR_DEVICE_TIMEOUT; 0 = off.
  int32_t debug_drop_load;
  // Test hook (dg_debug_plant_check, debug library only): nonzero makes the
  // MMA issuer's TMEM check fail on purpose; no access changes.
  int32_t debug_plant_check;
  // 256-row dense tiles: drain the accumulator with eight epilogue warps
  int32_t epi8;
  // C's base and row stride are multiples of 32 bytes: rows of C may be read
  // with 32-byte loads
  int32_t c_v8;
  // 256-row dense tiles: clusters of two CTAs on adjacent M blocks share each
  // B tile through TMA multicast (the grid is even)
  int32_t mc;
  // Stream-K (256-row dense tiles with eight epilogue warps; 0 units = off):
  // tiles [0, sk_dp_tiles) are walked one per CTA per wave, the K blocks of
  // the remaining tiles (sk_units = their count x k_blocks) are shared out
  // evenly.  sk_part holds one partial-accumulator slot of 256 x block_n
  // floats per CTA, sk_flags one word per (CTA, epilogue warp); both belong
  // to the caller's workspace, whose flags are zero between launches.
  float* sk_part;
  uint32_t* sk_flags;
  int64_t sk_units;
  int32_t sk_dp_tiles;
  // FP32-scale (promotion) form only
  const float* sfa_f32;    // [ceil(k/128), sfa_ld]: per K block, one scale per row of A
  const float* sfb_f32;    // [ceil(n/128), k/128]: one scale per 128 x 128 block of B
  int32_t sfa_ld;          // align(m, 4)
};

// Arguments of the decode-sized dense NT kernel (gemm_decode.cu): M <= 128
// rows of A against 128-row strips of B, the strip's K blocks split over a
// cluster of `split` CTAs.
struct DecodeArgs {
  const __nv_bfloat16* c;  // nullable, [m, ldc]
  __nv_bfloat16* d;        // [m, ldd]
  int64_t ldc, ldd;        // elements
  int32_t m, n;
  int32_t k_blocks;
  int32_t n_strips;        // ceil(n / 128)
  uint64_t timeout_ns;
  unsigned long long* err; // device error word
  int32_t pdl;             // launched with programmatic stream serialisation
  int32_t debug_plant_check;  // test hook of the debug library (dg_debug_plant_check)
  int32_t debug_drop_load;    // test hook (dg_debug_set_drop_load): 1 + the K block CTA 0 leaves unfilled
};

// gemm_decode.cu: tn = token columns per MMA (32, 64 or 128, >= M), split =
// CTAs per cluster (1, 2, 4 or 8); each CTA's K range spans at most
// gemm_decode_max_packs() scale words of 4 K blocks
cudaError_t gemm_decode_launch(int tn, int split, const CUtensorMap& a, const CUtensorMap& b,
                               const CUtensorMap& sfa, const CUtensorMap& sfb, DecodeArgs args,
                               cudaStream_t stream);
int gemm_decode_max_packs();

// gemm.cu: dispatch over the tile widths compiled in gemm_bn*.cu (single CTA)
// and gemm2_bn*.cu (CTA pairs, 256-row tiles)
int gemm_stages(int block_n);
bool gemm_block_n_supported(int block_n);
bool gemm2_block_n_supported(int block_n);
int gemm2_max_clusters(int mode, int block_n);  // per device, cached
cudaError_t gemm2_launch(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                         const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                         GemmArgs args, int clusters, cudaStream_t stream);
cudaError_t gemm_launch(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                        GemmArgs args, int grid, cudaStream_t stream);
cudaError_t gemm_fetch_error(unsigned long long* word);  // reads and clears
// device address of the error word on the current device (every launch passes
// it as GemmArgs::err)
cudaError_t error_word_address(unsigned long long** out);
// 256-row tiles (dense NT, contiguous): block_n 192 or 224; 0 stages = not compiled
int gemm_tall_stages(int block_n);
// pipeline stages of the 64-row-A-slot kernels (0: width not supported)
int gemm_short_stages(int block_n);
// pipeline stages of the split-K kernels
int gemm_splitk_stages(int ksplit, bool short_a);
// pipeline stages of the FP32-scale (promotion) kernel
int gemm_promote_stages();
constexpr int kMaxTallPairs = 1024;  // contiguous: most block pairs per launch
cudaError_t gemm_tall_launch(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                             const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                             GemmArgs args, int grid, cudaStream_t stream);
// single M block of at most 64 rows, dense NT: 64-row A slots (block_n 128 or 192)
bool gemm_short_supported(int block_n);
cudaError_t gemm_short_launch(int block_n, const CUtensorMap& a, const CUtensorMap& b,
                              const CUtensorMap& sfa, const CUtensorMap& sfb, const CUtensorMap& d,
                              GemmArgs args, int grid, cudaStream_t stream);
cudaError_t gemm_short_launch_impl(int block_n, const CUtensorMap& a, const CUtensorMap& b,
                                   const CUtensorMap& sfa, const CUtensorMap& sfb,
                                   const CUtensorMap& d, const GemmArgs& args, int grid,
                                   cudaStream_t stream);
cudaError_t gemm_tall_launch_impl(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                                  const CUtensorMap& sfa, const CUtensorMap& sfb,
                                  const CUtensorMap& d, const GemmArgs& args, int grid,
                                  cudaStream_t stream);

// gemm_bn*.cu: one tile width each (compiled in parallel)
#define DG_DECLARE_GEMM_BN(BN)                                                                  \
  cudaError_t gemm_launch_bn##BN(int mode, const CUtensorMap& a, const CUtensorMap& b,          \
                                 const CUtensorMap& sfa, const CUtensorMap& sfb,                \
                                 const CUtensorMap& d, const GemmArgs& args, int grid,          \
                                 cudaStream_t stream);                                          \
  int gemm_stages_bn##BN();
#define DG_DECLARE_GEMM2_BN(BN)                                                                 \
  cudaError_t gemm2_launch_bn##BN(int mode, const CUtensorMap& a, const CUtensorMap& b,         \
                                  const CUtensorMap& sfa, const CUtensorMap& sfb,               \
                                  const CUtensorMap& d, const GemmArgs& args, int clusters,     \
                                  cudaStream_t stream);                                         \
  int gemm2_max_clusters_bn##BN(int mode);
DG_DECLARE_GEMM2_BN(192)
DG_DECLARE_GEMM2_BN(224)
DG_DECLARE_GEMM2_BN(256)
#undef DG_DECLARE_GEMM2_BN
// gemm_splitk.cu: dense split-K over 2 or 4 CTAs, 128-column tiles
cudaError_t gemm_splitk_launch(int ksplit, bool short_a, const CUtensorMap& a, const CUtensorMap& b,
                               const CUtensorMap& sfa, const CUtensorMap& sfb,
                               const CUtensorMap& d, GemmArgs args, int clusters,
                               cudaStream_t stream);
int gemm_splitk_max_clusters(int ksplit);
// gemm_promote.cu: arbitrary FP32 scales, partials promoted out of TMEM
cudaError_t gemm_promote_launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                                GemmArgs args, int grid, cudaStream_t stream);
DG_DECLARE_GEMM_BN(128)
DG_DECLARE_GEMM_BN(192)
DG_DECLARE_GEMM_BN(224)
DG_DECLARE_GEMM_BN(256)
#undef DG_DECLARE_GEMM_BN

// gemm_kgrouped.cu: K-grouped 128 x 256 tiles with eight epilogue warps
// (args.err must already be set)
cudaError_t gemm_kgrouped_epi8_launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                                      const CUtensorMap& sfb, const CUtensorMap& d, const GemmArgs& args,
                                      int grid, cudaStream_t stream);

// quant.cu
cudaError_t quantize_launch(const float* x, void* q, void* sf, int64_t groups, int64_t rows,
                            int64_t cols, int block_rows, int sf_format, bool pdl,
                            cudaStream_t stream);
cudaError_t quantize_cols_launch(const float* x, void* q, void* sf, int64_t rows, int64_t cols,
                                 int sf_format, bool pdl, cudaStream_t stream);
cudaError_t transform_sf_launch(const float* sf, int32_t* packed, int64_t groups, int64_t mn,
                                int64_t k, int block_rows, bool pdl, cudaStream_t stream);
cudaError_t quant_fetch_error(unsigned long long* word);  // reads and clears

}  // namespace dg
