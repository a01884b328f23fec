// Host side of the C ABI declared in include/dg.h: argument checks, TMA
// descriptor encoding, tile configuration and launches.  No device memory is
// allocated and no stream is synchronised here (except dg_get_device_error).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxCoord = (int64_t)1 << 31;  // TMA coordinates are 32-bit signed

std::atomic<int32_t> g_num_sms_limit{0};
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_pdl{0};
std::atomic<int32_t> g_debug_drop_load{0};  // test hook, see dg_debug_set_drop_load
std::atomic<int32_t> g_debug_plant_check{0};  // test hook, see dg_debug_plant_check
std::atomic<int32_t> g_mk_alignment{kBlockM};  // dg_set_mk_alignment_for_contiguous_layout

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int cc_major = 0, cc_minor = 0, sms = 0;
};
DeviceInfo g_devices[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool env_flag(const char* name) {
  const char* v = getenv(name);
  return v && *v && strcmp(v, "0") != 0;
}

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  return (v && *v) ? atoi(v) : dflt;
}

// The DG_* overrides, read with getenv only when the process environment may
// have changed since this thread last read them: setenv / putenv / unsetenv
// (os.environ in Python) replace or move entries of `environ`, so a
// fingerprint of the entry pointers (a few tens of loads) stands in for the
// eight getenv scans a call would otherwise make.
struct EnvConfig {
  uintptr_t fingerprint = 0;
  bool valid = false;
  int block_m = 0, block_n = 0, split_k = 0, cta_pair = 0, stream_k = -1, tall_epi8 = 1,
      raster_band = 16, decode = 1, multicast = 1;
  bool print_configs = false;
};

uintptr_t environ_fingerprint() {
  char** const env = ::environ;  // the process environment (POSIX, unistd.h)
  uintptr_t h = reinterpret_cast<uintptr_t>(env);
  uintptr_t n = 0;
  for (char** e = env; e && *e; ++e, ++n) h = h * 1099511628211ull + reinterpret_cast<uintptr_t>(*e);
  return h ^ (n << 48);
}

const EnvConfig& env() {
  thread_local EnvConfig c;
  const uintptr_t f = environ_fingerprint();
  if (!c.valid || c.fingerprint != f) {
    c.block_m = env_int("DG_BLOCK_M", 0);
    c.block_n = env_int("DG_BLOCK_N", 0);
    c.split_k = env_int("DG_SPLIT_K", 0);
    c.cta_pair = env_int("DG_CTA_PAIR", 0);
    c.stream_k = env_int("DG_STREAM_K", -1);
    c.tall_epi8 = env_int("DG_TALL_EPI8", 1);
    c.raster_band = env_int("DG_RASTER_BAND", 16);
    c.decode = env_int("DG_DECODE", 1);
    c.multicast = env_int("DG_MULTICAST", 1);
    c.print_configs = env_flag("DG_PRINT_CONFIGS");
    c.fingerprint = f;
    c.valid = true;
  }
  return c;
}

dg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DG_OK : DG_ERR_CUDA; }

// Current device must be compute capability 10.3; reports its SM count.
dg_status current_device(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return DG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DG_ERR_CUDA;
  DeviceInfo& d = g_devices[dev];
  std::call_once(d.once, [&] {
    d.err = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (d.err == cudaSuccess)
      d.err = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (d.err == cudaSuccess)
      d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  });
  if (d.err != cudaSuccess) return DG_ERR_CUDA;
  if (d.cc_major != 10 || d.cc_minor != 3) return DG_ERR_UNSUPPORTED_ARCH;
  int limit = g_num_sms_limit.load();
  *sms = (limit > 0 && limit < d.sms) ? limit : d.sms;
  return DG_OK;
}

dg_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? DG_OK : DG_ERR_CUDA;
}

// Encodes a tiled TMA descriptor.  dims/box innermost first; strides (bytes)
// for dims 1..rank-1.
dg_status encode(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
  uint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base),
                        reinterpret_cast<const cuuint64_t*>(dims),
                        reinterpret_cast<const cuuint64_t*>(strides),
                        reinterpret_cast<const cuuint32_t*>(box),
                        reinterpret_cast<const cuuint32_t*>(elem_strides),
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DG_OK : DG_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t align4(int64_t x) { return (x + 3) / 4 * 4; }

// Operand descriptors shared by the three GEMM forms.
struct Operands {
  CUtensorMap a, b, sfa, sfb, d;
};

// D as a 2-D BF16 tensor [rows, n] with row stride ldd (elements); 32 x 32
// boxes with the 64-byte swizzle the epilogue stages in.
dg_status encode_d(Operands& o, void* d, int64_t rows, int64_t n, int64_t ldd) {
  uint64_t dims[2] = {(uint64_t)n, (uint64_t)rows};
  uint64_t strides[1] = {(uint64_t)(ldd * 2)};
  uint32_t box[2] = {32, 32};
  return encode(&o.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_64B);
}

// B tiles of `b_rows` rows (block_n, or half of it on a CTA pair) and the
// scale words of `block_n` rows.
dg_status encode_b_side(Operands& o, const void* b, const int32_t* sfb, int64_t groups,
                        int64_t n, int64_t k, int64_t ldb, int block_n, int b_rows) {
  const int64_t kp = (k / kBlockK + 3) / 4;
  const int64_t n_pad = align4(n);
  {
    uint64_t dims[3] = {(uint64_t)k, (uint64_t)n, (uint64_t)groups};
    uint64_t strides[2] = {(uint64_t)ldb, (uint64_t)(n * ldb)};
    uint32_t box[3] = {(uint32_t)kBlockK, (uint32_t)b_rows, 1};
    dg_status s = encode(&o.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, b, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != DG_OK) return s;
  }
  {
    uint64_t dims[3] = {(uint64_t)n_pad, (uint64_t)kp, (uint64_t)groups};
    uint64_t strides[2] = {(uint64_t)(n_pad * 4), (uint64_t)(kp * n_pad * 4)};
    uint32_t box[3] = {(uint32_t)block_n, 1, 1};
    return encode(&o.sfb, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, sfb, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  }
}

// box_rows: rows per A box (kBlockM, fewer for a single short M block, or
// 256 for 256-row tiles); sf_rows: rows per scale box (kBlockM or 256).
dg_status encode_a_2d(Operands& o, const void* a, const int32_t* sfa, int64_t m, int64_t k,
                      int64_t lda, int box_rows = kBlockM, int sf_rows = kBlockM) {
  const int64_t kp = (k / kBlockK + 3) / 4;
  const int64_t m_pad = align4(m);
  {
    uint64_t dims[2] = {(uint64_t)k, (uint64_t)m};
    uint64_t strides[1] = {(uint64_t)lda};
    uint32_t box[2] = {(uint32_t)kBlockK, (uint32_t)box_rows};
    dg_status s = encode(&o.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != DG_OK) return s;
  }
  {
    uint64_t dims[2] = {(uint64_t)m_pad, (uint64_t)kp};
    uint64_t strides[1] = {(uint64_t)(m_pad * 4)};
    uint32_t box[2] = {(uint32_t)sf_rows, 1};
    return encode(&o.sfa, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, sfa, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  }
}

dg_status encode_a_3d(Operands& o, const void* a, const int32_t* sfa, int64_t groups,
                      int64_t max_m, int64_t k) {
  const int64_t kp = (k / kBlockK + 3) / 4;
  const int64_t m_pad = align4(max_m);
  {
    uint64_t dims[3] = {(uint64_t)k, (uint64_t)max_m, (uint64_t)groups};
    uint64_t strides[2] = {(uint64_t)k, (uint64_t)(max_m * k)};
    uint32_t box[3] = {(uint32_t)kBlockK, (uint32_t)kBlockM, 1};
    dg_status s = encode(&o.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != DG_OK) return s;
  }
  {
    uint64_t dims[3] = {(uint64_t)m_pad, (uint64_t)kp, (uint64_t)groups};
    uint64_t strides[2] = {(uint64_t)(m_pad * 4), (uint64_t)(kp * m_pad * 4)};
    uint32_t box[3] = {(uint32_t)kBlockM, 1, 1};
    return encode(&o.sfa, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, sfa, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  }
}

// MN-major operand tiles ([K, MN] storage, MN innermost, row stride ld bytes):
// boxes of 128 (MN) x 128 (K) with 128-byte swizzle.  The scale words are the
// same as for the K-major forms.
dg_status encode_a_mn(Operands& o, const void* a, const int32_t* sfa, int64_t m, int64_t k,
                      int64_t lda) {
  const int64_t kp = (k / kBlockK + 3) / 4;
  const int64_t m_pad = align4(m);
  {
    uint64_t dims[2] = {(uint64_t)m, (uint64_t)k};
    uint64_t strides[1] = {(uint64_t)lda};
    uint32_t box[2] = {(uint32_t)kBlockM, (uint32_t)kBlockK};
    dg_status s = encode(&o.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != DG_OK) return s;
  }
  uint64_t dims[2] = {(uint64_t)m_pad, (uint64_t)kp};
  uint64_t strides[1] = {(uint64_t)(m_pad * 4)};
  uint32_t box[2] = {(uint32_t)kBlockM, 1};
  return encode(&o.sfa, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, sfa, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

dg_status encode_b_mn(Operands& o, const void* b, const int32_t* sfb, int64_t n, int64_t k,
                      int64_t ldb, int block_n) {
  const int64_t kp = (k / kBlockK + 3) / 4;
  const int64_t n_pad = align4(n);
  {
    uint64_t dims[2] = {(uint64_t)n, (uint64_t)k};
    uint64_t strides[1] = {(uint64_t)ldb};
    uint32_t box[2] = {128, (uint32_t)kBlockK};
    dg_status s = encode(&o.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != DG_OK) return s;
  }
  uint64_t dims[3] = {(uint64_t)n_pad, (uint64_t)kp, 1};
  uint64_t strides[2] = {(uint64_t)(n_pad * 4), (uint64_t)(kp * n_pad * 4)};
  uint32_t box[3] = {(uint32_t)block_n, 1, 1};
  return encode(&o.sfb, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, sfb, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Tile width along N.  Wider tiles cut the shared-memory and L2 traffic per
// MMA and amortise the fixed cost of each MMA instruction; narrower tiles
// leave fewer SMs idle in the last wave and, below 256 columns, keep two
// accumulators in TMEM so the epilogue overlaps the next tile.  The estimate
// is waves x (K blocks + epilogue cost) x columns / relative throughput;
// DG_BLOCK_N forces a width.
// m_blocks counts output-tile rows (128 rows, or 256 on a CTA pair) and
// `slots` the tiles that run at once (SMs, or co-resident pairs).
// whole_boxes: only the widths 128 and 256 (MN-major B tiles, other layouts).
int choose_block_n(int64_t m_blocks, int64_t n, int64_t k_blocks, int slots, bool with_c,
                   bool pair, bool whole_boxes = false) {
  const int forced = env().block_n;
  if (whole_boxes ? (forced == 128 || forced == 256)
                  : (pair ? gemm2_block_n_supported(forced) : gemm_block_n_supported(forced)))
    return forced;
  static const int widths[4] = {128, 192, 224, 256};
  static const double rate[4] = {1.0, 1.35, 1.5, 1.6};  // per-column MMA throughput
  // epilogue time not hidden behind MMAs, in K blocks: a little for two
  // accumulators (reading C costs ~3 more), more for the single-accumulator width
  const double epi_blocks[4] = {with_c ? 3.5 : 0.5, with_c ? 3.5 : 0.5, with_c ? 3.5 : 0.5,
                                with_c ? 10.0 : 4.0};
  const int sms = slots > 0 ? slots : 1;
  int best = pair ? 256 : 128;
  double best_cost = 1e300;
  for (int i = pair ? 1 : 0; i < 4; ++i) {
    if (whole_boxes && widths[i] % 128 != 0) continue;
    const int64_t tiles = m_blocks * ((n + widths[i] - 1) / widths[i]);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double cost = (double)waves * ((double)k_blocks + epi_blocks[i]) * widths[i] / rate[i];
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = widths[i];
    }
  }
  return best;
}

// 256-row tiles (dense NT): estimated like choose_block_n, in the same units
// (time of one K block of a 128 x 256 tile = 160), from measured rates: a
// K block of a 256 x 192 tile costs ~221 units and of a 256 x 224 tile ~237;
// the single accumulator's epilogue does not overlap the next tile (~6 K
// blocks without C; ~11 and ~16.5 with C, fetched before the accumulator is
// ready).  Returns the width, or 0 when no 256-row tile beats `best_cost` (the
// 128-row estimate) by 3%.
int choose_tall_block_n(int64_t m, int64_t n, int64_t k_blocks, int slots, bool with_c,
                        double best_cost) {
  const int forced_m = env().block_m;
  if (forced_m == 128) return 0;
  const int forced_n = env().block_n;
  if (forced_m == 256) return (forced_n == 192 || forced_n == 224) ? forced_n : 192;
  if (forced_n != 0) return 0;  // a forced width means 128-row tiles
  static const int widths[2] = {192, 224};
  static const double per_kb[2] = {221.0, 237.0};
  static const double epi[2] = {6.2, 6.5};
  static const double epi_c[2] = {11.0, 16.5};
  const int sms = slots > 0 ? slots : 1;
  const int64_t m_blocks = (m + 2 * kBlockM - 1) / (2 * kBlockM);
  int best = 0;
  for (int i = 0; i < 2; ++i) {
    const int64_t tiles = m_blocks * ((n + widths[i] - 1) / widths[i]);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double cost = (double)waves * ((double)k_blocks + (with_c ? epi_c[i] : epi[i])) * per_kb[i];
    if (cost < best_cost * 0.97) {
      best_cost = cost;
      best = widths[i];
    }
  }
  return best;
}

// Estimated cost of 128-row tiles of width bn (units of choose_tall_block_n).
double dense_tile_cost(int64_t m_blocks, int64_t n, int64_t k_blocks, int slots, bool with_c, int bn) {
  static const int widths[4] = {128, 192, 224, 256};
  static const double rate[4] = {1.0, 1.35, 1.5, 1.6};
  int i = 0;
  while (i < 3 && widths[i] != bn) ++i;
  const double epi = bn == 256 ? (with_c ? 10.0 : 4.0) : (with_c ? 3.5 : 0.5);
  const int sms = slots > 0 ? slots : 1;
  const int64_t tiles = m_blocks * ((n + bn - 1) / bn);
  const int64_t waves = (tiles + sms - 1) / sms;
  return (double)waves * ((double)k_blocks + epi) * bn / rate[i];
}

// Tile width for masked problems with few rows per group, which are bound by
// streaming B from HBM rather than by the tensor cores.  A tile's time then
// grows with its width (its share of B) plus a fixed part (A, scales, set-up).
// The 256-column tile's single accumulator costs little here: its epilogue
// reads the whole row into registers before storing (measured on 16 groups x
// 256 rows, N=7168, K=2048: 50.1 / 53.0 / 55.6 / 57.8 us for 256 / 224 / 192 /
// 128 columns).  The host does not know the per-group counts (they stay on the
// device), so the number of 128-row blocks is estimated from the expected
// count per group: ceil(m / 128) is on average m / 128 + 1/2.
int choose_block_n_masked_streaming(int64_t groups, int64_t expected_m, int64_t n, int slots) {
  const int forced = env().block_n;
  if (gemm_block_n_supported(forced)) return forced;
  static const int widths[4] = {128, 192, 224, 256};
  const double blocks = (double)groups * ((double)expected_m / kBlockM + 0.5);
  const int sms = slots > 0 ? slots : 1;
  int best = 224;
  double best_cost = 1e300;
  for (int i = 0; i < 4; ++i) {
    const double tiles = std::ceil(blocks) * (double)((n + widths[i] - 1) / widths[i]);
    const double waves = std::ceil(tiles / sms);
    const double cost = waves * (widths[i] + 96.0);
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = widths[i];
    }
  }
  return best;
}

// Dense NT tile choice (single CTA, no split-K): every candidate tile of
// block_m x block_n is costed as waves x (K blocks + epilogue) x time per K
// block, the epilogue counted as the K blocks of MMA time it does not hide.
// The two numbers per tile (and per with / without C) are least-squares fits
// of the GB300 prefill sweeps (M = 4096, the five (N, K) pairs of the
// prefill workload, every tile forced in turn; us per K block at the clock of
// those runs): they rank the tiles as the measurements do on every shape of
// that sweep but one near-tie.  256-row tiles drain their single accumulator
// with eight epilogue warps, which is what makes them win at short K.
struct DenseTileCost {
  int block_m, block_n;
  double us_per_kb, epi_kb, us_per_kb_c, epi_kb_c;
};
// (The with-C pairs were refitted after the single-accumulator epilogues
// began fetching the next tile's C during the current tile's stores.)
constexpr DenseTileCost kDenseTiles[] = {
    {128, 128, 0.3278, 3.90, 0.3383, 3.38},  {128, 192, 0.3609, 4.73, 0.3616, 4.20},
    {128, 224, 0.3836, 3.72, 0.3770, 5.33},  {128, 256, 0.4081, 5.88, 0.4204, 6.18},
    {256, 192, 0.5463, 3.79, 0.5414, 7.70},  {256, 224, 0.5795, 5.00, 0.5957, 8.76},
};

double dense_nt_cost(const DenseTileCost& t, int64_t m, int64_t n, int64_t k_blocks, int slots, bool with_c) {
  const int64_t tiles = ((m + t.block_m - 1) / t.block_m) * ((n + t.block_n - 1) / t.block_n);
  const int64_t waves = (tiles + slots - 1) / slots;
  return (double)waves * ((double)k_blocks + (with_c ? t.epi_kb_c : t.epi_kb)) *
         (with_c ? t.us_per_kb_c : t.us_per_kb);
}

// The cheapest dense NT tile; DG_BLOCK_M (128 or 256) and DG_BLOCK_N restrict
// the candidates (DG_BLOCK_N alone means 128-row tiles of that width).  A
// single M block takes 128-row tiles.
void choose_dense_nt_tile(int64_t m, int64_t n, int64_t k_blocks, int slots, bool with_c, int* block_m,
                          int* block_n) {
  int forced_m = env().block_m;
  int forced_n = env().block_n;
  if (forced_m == 256 && gemm_tall_stages(forced_n) == 0) forced_n = 0;  // no such 256-row width
  if (forced_n != 0 && forced_m != 256 && gemm_block_n_supported(forced_n)) forced_m = 128;
  const int sms = slots > 0 ? slots : 1;
  double best = 1e300;
  *block_m = kBlockM;
  *block_n = 128;
  for (const DenseTileCost& t : kDenseTiles) {
    if (t.block_m == 2 * kBlockM && (m <= kBlockM || gemm_tall_stages(t.block_n) == 0)) continue;
    if ((forced_m == 128 || forced_m == 256) && t.block_m != forced_m) continue;
    if (forced_n != 0 && t.block_n != forced_n && gemm_block_n_supported(forced_n)) continue;
    const double c = dense_nt_cost(t, m, n, k_blocks, sms, with_c);
    if (c < best * 0.999) {
      best = c;
      *block_m = t.block_m;
      *block_n = t.block_n;
    }
  }
}

// Raster band of the dense tile walk, in M blocks of block_m rows: inside a
// band the M block varies fastest, so a wave of CTAs shares a few column
// blocks of B and the band's rows of A; B is read from DRAM once per band.
// 2048 rows: on GB300 (M = 4096) bands of the whole of M were 2-3% slower for
// the 256-row tiles at K <= 7168, and at K = 16384 their 64 MB strip of A
// did not survive in L2 between waves (DRAM reads 393 MB against 366.6 MB):
// A is read by SMs of both dies and held in both halves of L2.
// DG_RASTER_BAND (in 128-row blocks) overrides.
int raster_band(int64_t m_blocks, int block_m, int64_t k) {
  (void)k;
  const int band128 = std::max(1, env().raster_band);
  return (int)std::max<int64_t>(1, std::min<int64_t>(m_blocks, (int64_t)band128 * kBlockM / block_m));
}

void print_config(const char* what, int64_t m, int64_t n, int64_t k, int groups, int block_m,
                  int block_n, int stages, int grid, int band) {
  if (!env().print_configs) return;
  fprintf(stderr, "dg: %s m=%lld n=%lld k=%lld groups=%d block_m=%d block_n=%d stages=%d grid=%d band=%d\n",
          what, (long long)m, (long long)n, (long long)k, groups, block_m, block_n, stages, grid, band);
}

// Tile configuration of a dense GEMM: pure host arithmetic on the shape and
// the SM count (the DG_* overrides apply), shared by the launch and by
// dg_plan_fp8_gemm_nt.
struct DensePlan {
  int ksplit = 1;        // CTAs of a cluster sharing each tile's K blocks (1, 2, 4; 1-8 for decode)
  int block_n = 128;     // output columns per tile
  bool pair = false;     // 256-row tiles on a pair of CTAs (only on request)
  bool tall = false;     // 256-row tiles on one CTA
  // 256-row tiles in clusters of two CTAs (adjacent M blocks, one column
  // block of B), each CTA loading half of B into both through TMA multicast
  bool multicast = false;
  bool short_a = false;  // 64-row A slots: a single M block of at most 64 rows
  // stream-K (256-row tiles, only with a workspace): tiles [0, sk_dp_tiles)
  // one per CTA per wave, the K blocks of the rest (sk_units) shared evenly
  bool stream_k = false;
  int32_t sk_dp_tiles = 0;
  int64_t sk_units = 0;
  // decode-sized M: the swapped-operand kernel (tokens on the MMA's N side,
  // decode_tn of them per MMA; 128-column strips, K split over ksplit CTAs)
  bool decode = false;
  int decode_tn = 0;
};

// Cluster size of the decode kernel for T strips of kb K blocks on `sms` SMs,
// 0 when none applies.  The kernel runs one CTA per SM (its pipeline takes
// the SM's shared memory), so the clusters must fit in one wave: T x S <=
// sms; every CTA's K range must span at most gemm_decode_max_packs() scale
// words.  Among those, the largest S (the fewest K blocks per CTA: the
// kernel is bound by how fast each SM streams its part of B).
// DG_SPLIT_K = 1, 2, 4 or 8 forces a size where it applies.
// A cluster's CTAs share one GPC (19 SMs on GB300: 152 SMs in 8 GPCs), so
// at most floor(19 / S) clusters of S CTAs run per GPC at once (measured:
// 17 clusters of 8 CTAs take two waves on 152 SMs, 17 of 4 one).
int decode_split(int64_t strips, int64_t kb, int sms) {
  constexpr int kGpcSms = 19;
  const int gpcs = sms / kGpcSms > 0 ? sms / kGpcSms : 1;
  const int forced = env().split_k;
  int best = 0;
  for (int s : {1, 2, 4, 8}) {
    if (s > kb || strips * s > sms || (s > 1 && strips > (int64_t)gpcs * (kGpcSms / s))) break;
    if (forced != 0 && forced != s) continue;
    bool fits = true;
    for (int r = 0; r < s && fits; ++r) {
      const int64_t k0 = kb * r / s, k1 = kb * (r + 1) / s;
      fits = ((k1 - 1) >> 2) - (k0 >> 2) + 1 <= gemm_decode_max_packs();
    }
    if (fits) best = s;
  }
  return best;
}

// Workspace of a stream-K launch on `sms` CTAs with block_n columns: a fixed
// 32 KiB of flag words (one per (CTA, epilogue warp), for up to 1024 CTAs, so
// the flags sit at the same place whatever the SM count a later call uses),
// then one partial slot of 256 x block_n floats per CTA.
constexpr int kStreamKMaxCtas = 1024;
constexpr uint64_t kStreamKFlagBytes = (uint64_t)kStreamKMaxCtas * 8 * 4;
uint64_t stream_k_workspace_bytes(int sms, int block_n) {
  return kStreamKFlagBytes + (uint64_t)sms * (uint64_t)(2 * kBlockM) * (uint64_t)block_n * 4;
}

// Stream-K split of T tiles of kb K blocks over P CTAs: whole waves but the
// last are walked tile by tile; the last full wave and the partial one
// (P + r tiles, or all T when T < P) have their K blocks shared evenly, so
// every CTA ends at the same time.  False when the waves are already whole,
// or when some CTA would get no K block.
bool stream_k_split(int64_t tiles, int64_t kb, int sms, int32_t* dp_tiles, int64_t* units) {
  if (sms < 2 || sms > kStreamKMaxCtas || tiles <= 0) return false;
  const int64_t q = tiles / sms, r = tiles % sms;
  if (r == 0) return false;
  const int64_t dp = q >= 1 ? (q - 1) * sms : 0;
  const int64_t u = (tiles - dp) * kb;
  if (u < sms) return false;
  if (u * (sms + 1) >= ((int64_t)1 << 32)) return false;  // the kernel's unit arithmetic is 32-bit
  *dp_tiles = (int32_t)dp;
  *units = u;
  return true;
}


DensePlan plan_dense(int mode, int64_t m, int64_t n, int64_t k, bool with_c, int sms, bool ws = false) {
  DensePlan p;
  const int64_t kb = k / kBlockK;
  const int64_t m_blocks = (m + kBlockM - 1) / kBlockM;
  // at most 128 rows of A (NT): the swapped-operand decode kernel unless
  // DG_DECODE = 0 (or a DG_BLOCK_* override asks for the tiled kernels)
  if (mode == kDense && m <= kBlockM && env().decode != 0 && env().block_m == 0 && env().block_n == 0) {
    // Measured on GB300 (M = 64 and 128, the five (N, K) pairs, graph
    // replays over copies larger than L2): with clusters of 4 or 8 CTAs it
    // matches or beats the tiled split-K kernels (N = 4096, K = 7168: 12.8 /
    // 14.9 us against 13.8 / 15.2); with 1 or 2 (many strips) it does not
    // (N = 7168, K = 2048, M = 128: 11.6 us against 10.9), so those shapes
    // keep the tiled kernels.  DG_SPLIT_K forces a size.
    const int s = decode_split((n + 127) / 128, kb, sms);
    if (s >= 4 || (s > 0 && env().split_k != 0)) {
      p.decode = true;
      p.decode_tn = m <= 32 ? 32 : m <= 64 ? 64 : 128;
      p.ksplit = s;
      p.block_n = 128;
      return p;
    }
  }
  // Split-K over a cluster of 2 or 4 CTAs when 128-column tiles would leave
  // most SMs idle (decode-sized M); DG_SPLIT_K = 1, 2 or 4 forces a factor.
  // Every CTA's K slice (ceil(K blocks / factor) blocks) must be non-empty.
  {
    const int64_t tiles128 = m_blocks * ((n + 127) / 128);
    const int forced = env().split_k;
    if (mode != kDense) p.ksplit = 1;
    else if (forced == 1 || forced == 2 || forced == 4) p.ksplit = forced;
    else if (tiles128 * 4 <= sms && kb >= 16) p.ksplit = 4;
    else if (tiles128 * 2 <= sms && kb >= 8) p.ksplit = 2;
    while (p.ksplit > 1) {
      const int64_t per = (kb + p.ksplit - 1) / p.ksplit;
      if ((p.ksplit - 1) * per < kb) break;
      p.ksplit /= 2;
    }
  }
  if (p.ksplit > 1) {
    p.block_n = 128;
    p.short_a = m <= kBlockM / 2;
    return p;
  }
  // CTA pairs (256-row tiles) only on request (DG_CTA_PAIR=1): on the
  // measured shapes they match, not beat, single-CTA tiles.
  p.pair = mode == kDense && sms >= 2 && m_blocks >= 2 && env().cta_pair == 1;
  if (p.pair) {
    const int64_t p_blocks = (m + 2 * kBlockM - 1) / (2 * kBlockM);
    p.block_n = choose_block_n(p_blocks, n, kb, sms / 2, with_c, true);
    return p;
  }
  if (mode == kDense && m_blocks >= 2) {
    // NT with several M blocks: 128- or 256-row tiles from the measured cost
    // table (a single M block is memory-bound, costed below)
    int bm = kBlockM;
    choose_dense_nt_tile(m, n, kb, sms, with_c, &bm, &p.block_n);
    p.tall = bm == 2 * kBlockM;
    // With a workspace, 256-row tiles in stream-K order where the estimate
    // beats the tile-by-tile walk by 10%: the same cost table for each CTA's
    // share of K blocks and of the tiles' final epilogues, plus the fixed cost
    // of the partial sums measured on GB300 (M = 4096, N = 2112, K = 7168,
    // 160 tiles of 256 x 224 on 152 SMs, traced per CTA): ~4.8 us while the
    // contributor writes its 224 KB partial and the MMA waits, ~8 us for the
    // owner's flag wait, partial reads and stores; ~22 K blocks in all.
    // DG_STREAM_K = 0 / 1 disables / forces it where it applies.
    const int forced_sk = env().stream_k;
    const int forced_m = env().block_m, forced_n = env().block_n;
    if (ws && forced_sk != 0 && env().tall_epi8 != 0 && forced_m != 128 && sms >= 2) {
      double cost_dp = 1e300;
      for (const DenseTileCost& t : kDenseTiles)
        if (t.block_m == bm && t.block_n == p.block_n) cost_dp = dense_nt_cost(t, m, n, kb, sms, with_c);
      double best = forced_sk == 1 ? 1e300 : 0.9 * cost_dp;
      for (const DenseTileCost& t : kDenseTiles) {
        if (t.block_m != 2 * kBlockM || gemm_tall_stages(t.block_n) == 0) continue;
        if (forced_n != 0 && forced_n != t.block_n) continue;
        const int64_t tiles = ((m + t.block_m - 1) / t.block_m) * ((n + t.block_n - 1) / t.block_n);
        int32_t dp = 0;
        int64_t units = 0;
        if (!stream_k_split(tiles, kb, sms, &dp, &units)) continue;
        const double e = with_c ? t.epi_kb_c : t.epi_kb;
        const double cost = ((double)dp / sms * ((double)kb + e) + (double)units / sms +
                             (double)(tiles - dp) / sms * e + 22.0) *
                            (with_c ? t.us_per_kb_c : t.us_per_kb);
        if (cost < best) {
          best = cost;
          p.stream_k = true;
          p.tall = true;
          p.block_n = t.block_n;
          p.sk_dp_tiles = dp;
          p.sk_units = units;
        }
      }
    }
  } else {
    p.block_n = choose_block_n(m_blocks, n, kb, sms, with_c, false, mode != kDense);
  }
  // a single M block of at most 64 rows: 64-row A slots, more stages
  p.short_a = mode == kDense && !p.tall && m <= kBlockM / 2 && gemm_short_supported(p.block_n);
  // 256-row dense tiles (eight epilogue warps, tile by tile) share B between
  // the two CTAs of a cluster; DG_MULTICAST = 0 turns it off.  Measured on
  // GB300: 1.3-1.6% faster on the prefill shapes that take 256-row tiles,
  // none slower.
  p.multicast = mode == kDense && p.tall && !p.stream_k && env().tall_epi8 != 0 && env().multicast != 0 &&
                sms >= 2;
  return p;
}

// Tile configuration of the M-grouped forms (pure host arithmetic, the
// DG_* overrides apply), shared by the launches and the plan queries.
struct GroupedPlan {
  int block_n = 128;
  bool tall = false;  // contiguous: 256-row tiles pairing two blocks of one group
  bool pair = false;  // masked: 256-row tiles on a CTA pair (only on request)
};

GroupedPlan plan_contiguous(int64_t m_sum, int64_t n, int64_t k, int32_t num_groups, int sms) {
  GroupedPlan p;
  const int64_t m_blocks = m_sum / kBlockM;
  p.block_n = choose_block_n(m_blocks, n, k / kBlockK, sms, false, false);
  // 256-row tiles pair two 128-row blocks of one group (at most (blocks +
  // groups) / 2 pairs, which must fit the kernel's table); estimated as dense
  // tiles over the expected pairs, blocks / 2 + groups / 2.
  if (num_groups <= kMaxMaskedGroups && m_blocks < 0xFFFF &&
      (m_blocks + num_groups + 1) / 2 <= kMaxTallPairs) {
    const int64_t pairs = (m_blocks + num_groups + 1) / 2;
    const double cost128 = dense_tile_cost(m_blocks, n, k / kBlockK, sms, false, p.block_n);
    const int tall_n = choose_tall_block_n(pairs * 2 * kBlockM, n, k / kBlockK, sms, false, cost128);
    if (tall_n != 0 && gemm_tall_stages(tall_n) > 0) {
      p.tall = true;
      p.block_n = tall_n;
    }
  }
  return p;
}

GroupedPlan plan_masked(int32_t num_groups, int64_t max_m, int64_t n, int64_t k, int64_t expected_m,
                        int sms) {
  GroupedPlan p;
  // CTA pairs only on request (DG_CTA_PAIR=1); with few valid rows per group
  // the peer's half of the tile is mostly empty.
  p.pair = sms >= 2 && max_m > kBlockM && env().cta_pair == 1;
  const int64_t m_est = expected_m > 0 ? expected_m : max_m;
  if (p.pair)
    p.block_n = choose_block_n(((m_est + 2 * kBlockM - 1) / (2 * kBlockM)) * num_groups, n,
                               k / kBlockK, sms / 2, false, true);
  else if (expected_m > 0 && expected_m <= 2 * kBlockM)
    p.block_n = choose_block_n_masked_streaming(num_groups, std::min<int64_t>(expected_m, max_m), n, sms);
  else
    p.block_n = choose_block_n(((m_est + kBlockM - 1) / kBlockM) * num_groups, n, k / kBlockK, sms,
                               false, false);
  return p;
}

dg_status check_common_k_n(int64_t n, int64_t k) {
  if (n < 0 || k < 0) return DG_ERR_INVALID_ARG;
  if (k == 0) return DG_ERR_INVALID_ARG;
  if (k % kBlockK != 0) return DG_ERR_ALIGNMENT;
  if (n % 8 != 0) return DG_ERR_ALIGNMENT;
  if (k >= kMaxCoord || n >= kMaxCoord) return DG_ERR_TOO_LARGE;
  return DG_OK;
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" {

// Dense GEMM in one of the four operand layouts (mode kDense = NT, kDenseNN,
// kDenseTN, kDenseTT).  Split-K and CTA pairs exist for NT only.
static dg_status dense_gemm(int mode, const char* name, const void* a, const int32_t* sfa,
                            const void* b, const int32_t* sfb, const void* c, void* d, int64_t m,
                            int64_t n, int64_t k, int64_t lda, int64_t ldb, int64_t ldc,
                            int64_t ldd, void* stream, void* workspace = nullptr,
                            uint64_t workspace_bytes = 0) {
  if (m < 0) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (m == 0 || n == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d) return DG_ERR_INVALID_ARG;
  if (lda < (a_mn_major(mode) ? m : k) || ldb < (b_mn_major(mode) ? n : k) || ldd < n ||
      (c && ldc < n))
    return DG_ERR_INVALID_ARG;
  if (lda % 16 || ldb % 16 || ldd % 8 || (c && ldc % 8)) return DG_ERR_ALIGNMENT;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(d) ||
      (c && !aligned16(c)) || (workspace && !aligned16(workspace)))
    return DG_ERR_ALIGNMENT;
  if (m >= kMaxCoord) return DG_ERR_TOO_LARGE;
  int sms = 0;
  if ((s = current_device(&sms)) != DG_OK) return s;
  if ((s = get_encoder()) != DG_OK) return s;

  DensePlan plan = plan_dense(mode, m, n, k, c != nullptr, sms, workspace != nullptr);
  if (plan.stream_k && workspace_bytes < stream_k_workspace_bytes(sms, plan.block_n))
    plan = plan_dense(mode, m, n, k, c != nullptr, sms, false);  // too small: tile by tile
  if (plan.decode) {
    // A [m, k] and B [n, k] K-major; scale words [kp, align4(rows)], boxes of
    // 8 packs (the most a CTA's K range spans)
    const int tn = plan.decode_tn;
    const int64_t kp = (k / kBlockK + 3) / 4;
    const int packs = gemm_decode_max_packs();
    Operands o;
    {
      uint64_t dims[2] = {(uint64_t)k, (uint64_t)m};
      uint64_t strides[1] = {(uint64_t)lda};
      uint32_t box[2] = {(uint32_t)kBlockK, (uint32_t)tn};
      if ((s = encode(&o.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != DG_OK)
        return s;
    }
    {
      uint64_t dims[2] = {(uint64_t)k, (uint64_t)n};
      uint64_t strides[1] = {(uint64_t)ldb};
      uint32_t box[2] = {(uint32_t)kBlockK, 128};
      if ((s = encode(&o.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != DG_OK)
        return s;
    }
    {
      uint64_t dims[2] = {(uint64_t)align4(m), (uint64_t)kp};
      uint64_t strides[1] = {(uint64_t)(align4(m) * 4)};
      uint32_t box[2] = {(uint32_t)tn, (uint32_t)packs};
      if ((s = encode(&o.sfa, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, sfa, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) != DG_OK)
        return s;
    }
    {
      uint64_t dims[2] = {(uint64_t)align4(n), (uint64_t)kp};
      uint64_t strides[1] = {(uint64_t)(align4(n) * 4)};
      uint32_t box[2] = {128, (uint32_t)packs};
      if ((s = encode(&o.sfb, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, sfb, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) != DG_OK)
        return s;
    }
    DecodeArgs da = {};
    da.c = static_cast<const __nv_bfloat16*>(c);
    da.d = static_cast<__nv_bfloat16*>(d);
    da.ldc = c ? ldc : 0;
    da.ldd = ldd;
    da.m = (int32_t)m;
    da.n = (int32_t)n;
    da.k_blocks = (int32_t)(k / kBlockK);
    da.n_strips = (int32_t)((n + 127) / 128);
    da.timeout_ns = g_timeout_ns.load();
    da.pdl = g_pdl.load();
    da.debug_plant_check = g_debug_plant_check.load(std::memory_order_relaxed);
    da.debug_drop_load = g_debug_drop_load.load(std::memory_order_relaxed);
    print_config("fp8_gemm_nt (decode, swapped operands)", m, n, k, 1, tn, 128, tn == 128 ? 3 : 4,
                 da.n_strips * plan.ksplit, plan.ksplit);
    return from_cuda(gemm_decode_launch(tn, plan.ksplit, o.a, o.b, o.sfa, o.sfb, da,
                                        static_cast<cudaStream_t>(stream)));
  }
  const int ksplit = plan.ksplit;
  GemmArgs args = {};
  args.m_blocks = (int32_t)((m + kBlockM - 1) / kBlockM);
  // A single M block shorter than 128 rows loads only round_up(M, 8) rows of A
  // per K block (dense NT; decode-sized M).
  if (mode == kDense && m < kBlockM) args.a_box_rows = (int32_t)((m + 7) / 8 * 8);
  if (ksplit > 1) {
    const int block_n = plan.block_n;
    Operands o;
    if ((s = encode_a_2d(o, a, sfa, m, k, lda, args.a_box_rows > 0 ? args.a_box_rows : kBlockM)) != DG_OK)
      return s;
    if ((s = encode_b_side(o, b, sfb, 1, n, k, ldb, block_n, block_n)) != DG_OK) return s;
    if ((s = encode_d(o, d, m, n, ldd)) != DG_OK) return s;
    args.c = static_cast<const __nv_bfloat16*>(c);
    args.c_v8 = (c && (reinterpret_cast<uintptr_t>(c) & 31u) == 0 && (ldc * 2) % 32 == 0) ? 1 : 0;
    args.d = static_cast<__nv_bfloat16*>(d);
    args.ldc = c ? ldc : 0;
    args.ldd = ldd;
    args.m = (int32_t)m;
    args.n = (int32_t)n;
    args.k = (int32_t)k;
    args.num_groups = 1;
    args.n_blocks = (int32_t)((n + block_n - 1) / block_n);
    args.k_blocks = (int32_t)(k / kBlockK);
    args.band = env().raster_band;
    if (args.band < 1) args.band = 1;
    args.timeout_ns = g_timeout_ns.load();
    args.pdl = g_pdl.load();
    const int64_t tiles = (int64_t)args.m_blocks * args.n_blocks;
    int clusters = gemm_splitk_max_clusters(ksplit);
    if (clusters > sms / ksplit) clusters = sms / ksplit;
    if (tiles < clusters) clusters = (int)tiles;
    if (clusters <= 0) return DG_ERR_CUDA;
    print_config(ksplit == 2 ? "fp8_gemm_nt (split-K 2)" : "fp8_gemm_nt (split-K 4)", m, n, k, 1,
                 plan.short_a ? kBlockM / 2 : kBlockM, block_n, gemm_splitk_stages(ksplit, plan.short_a),
                 ksplit * clusters, args.band);
    args.debug_drop_load = g_debug_drop_load.load(std::memory_order_relaxed);
    return from_cuda(gemm_splitk_launch(ksplit, plan.short_a, o.a, o.b, o.sfa, o.sfb, o.d, args, clusters,
                                        static_cast<cudaStream_t>(stream)));
  }
  const bool pair = plan.pair;
  const bool tall = plan.tall;
  const int block_n = plan.block_n;
  const int64_t p_blocks = (m + 2 * kBlockM - 1) / (2 * kBlockM);
  int clusters = 0;
  if (pair) {
    clusters = gemm2_max_clusters(kDense, block_n);
    const int limit = sms / 2;
    if (clusters > limit) clusters = limit;
    if (clusters <= 0) return DG_ERR_CUDA;
  }
  if (tall) args.m_blocks = (int32_t)p_blocks;
  const bool mc = plan.multicast;
  args.mc = mc ? 1 : 0;
  Operands o;
  s = a_mn_major(mode) ? encode_a_mn(o, a, sfa, m, k, lda)
      : tall           ? encode_a_2d(o, a, sfa, m, k, lda, 2 * kBlockM, 2 * kBlockM)
                       : encode_a_2d(o, a, sfa, m, k, lda, args.a_box_rows > 0 ? args.a_box_rows : kBlockM);
  if (s != DG_OK) return s;
  s = b_mn_major(mode) ? encode_b_mn(o, b, sfb, n, k, ldb, block_n)
                       : encode_b_side(o, b, sfb, 1, n, k, ldb, block_n, (pair || mc) ? block_n / 2 : block_n);
  if (s != DG_OK) return s;
  if ((s = encode_d(o, d, m, n, ldd)) != DG_OK) return s;
  args.c = static_cast<const __nv_bfloat16*>(c);
  args.c_v8 = (c && (reinterpret_cast<uintptr_t>(c) & 31u) == 0 && (ldc * 2) % 32 == 0) ? 1 : 0;
  args.d = static_cast<__nv_bfloat16*>(d);
  args.ldc = c ? ldc : 0;
  args.ldd = ldd;
  args.m = (int32_t)m;
  args.n = (int32_t)n;
  args.k = (int32_t)k;
  args.num_groups = 1;
  args.n_blocks = (int32_t)((n + block_n - 1) / block_n);
  args.k_blocks = (int32_t)(k / kBlockK);
  args.band = raster_band(args.m_blocks, (pair || tall) ? 2 * kBlockM : kBlockM, k);
  args.timeout_ns = g_timeout_ns.load();
  args.pdl = g_pdl.load();
  const int64_t tiles = (pair ? p_blocks : (int64_t)args.m_blocks) * args.n_blocks;
  if (tiles >= kMaxCoord) return DG_ERR_TOO_LARGE;
  if (pair) {
    if (tiles < clusters) clusters = (int)tiles;
    print_config("fp8_gemm_nt (cta pair)", m, n, k, 1, 2 * kBlockM, block_n, 6, 2 * clusters, args.band);
    return from_cuda(gemm2_launch(kDense, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, clusters,
                                  static_cast<cudaStream_t>(stream)));
  }
  const int64_t pair_tiles = ((p_blocks + 1) / 2) * args.n_blocks;
  const int grid = plan.stream_k ? sms
                   : mc          ? 2 * (int)(pair_tiles < sms / 2 ? pair_tiles : sms / 2)
                                 : (int)(tiles < sms ? tiles : sms);
  args.debug_drop_load = g_debug_drop_load.load(std::memory_order_relaxed);
  args.debug_plant_check = g_debug_plant_check.load(std::memory_order_relaxed);
  if (plan.stream_k) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    args.sk_flags = reinterpret_cast<uint32_t*>(ws);
    args.sk_part = reinterpret_cast<float*>(ws + kStreamKFlagBytes);
    args.sk_units = plan.sk_units;
    args.sk_dp_tiles = plan.sk_dp_tiles;
  }
  print_config(plan.stream_k ? "fp8_gemm_nt (256-row tiles, stream-K)"
               : mc          ? "fp8_gemm_nt (256-row tiles, clusters of 2 sharing B by multicast)"
               : tall        ? "fp8_gemm_nt (256-row tiles)"
               : plan.short_a ? "fp8_gemm_nt (64-row A slots)" : name,
               m, n, k, 1, tall ? 2 * kBlockM : plan.short_a ? kBlockM / 2 : kBlockM, block_n,
               tall ? gemm_tall_stages(block_n) : plan.short_a ? gemm_short_stages(block_n) : gemm_stages(block_n),
               grid, args.band);
  args.epi8 = (plan.stream_k || env().tall_epi8 != 0) ? 1 : 0;
  if (tall)
    return from_cuda(gemm_tall_launch(kDense, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid,
                                      static_cast<cudaStream_t>(stream)));
  if (plan.short_a)
    return from_cuda(gemm_short_launch(block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid,
                                       static_cast<cudaStream_t>(stream)));
  return from_cuda(gemm_launch(mode, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid,
                               static_cast<cudaStream_t>(stream)));
}

dg_status dg_fp8_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream) {
  return dense_gemm(kDense, "fp8_gemm_nt", a, sfa, b, sfb, c, d, m, n, k, lda, ldb, ldc, ldd,
                    stream);
}

dg_status dg_fp8_gemm_nt_ws(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                            const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                            int64_t ldb, int64_t ldc, int64_t ldd, void* workspace,
                            uint64_t workspace_bytes, void* stream) {
  return dense_gemm(kDense, "fp8_gemm_nt", a, sfa, b, sfb, c, d, m, n, k, lda, ldb, ldc, ldd, stream,
                    workspace, workspace_bytes);
}

dg_status dg_fp8_gemm_nt_workspace_size(int64_t m, int64_t n, int64_t k, int32_t has_c,
                                        int32_t num_sms, uint64_t* bytes) {
  if (!bytes) return DG_ERR_INVALID_ARG;
  *bytes = 0;
  if (m < 0 || num_sms < 1) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (m >= kMaxCoord) return DG_ERR_TOO_LARGE;
  if (m == 0 || n == 0) return DG_OK;
  const DensePlan p = plan_dense(kDense, m, n, k, has_c != 0, num_sms, true);
  if (p.stream_k) *bytes = stream_k_workspace_bytes(num_sms, p.block_n);
  return DG_OK;
}

dg_status dg_plan_fp8_gemm_nt_ws(int64_t m, int64_t n, int64_t k, int32_t has_c, int32_t num_sms,
                                 int32_t* block_m, int32_t* block_n, int32_t* split_k,
                                 int32_t* cta_pair, int32_t* stream_k, int32_t* swap_ab, int32_t* multicast) {
  if (!block_m || !block_n || !split_k || !cta_pair || !stream_k || !swap_ab || !multicast)
    return DG_ERR_INVALID_ARG;
  *block_m = *block_n = *split_k = *cta_pair = *stream_k = *swap_ab = *multicast = 0;
  if (m < 0 || num_sms < 1) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (m >= kMaxCoord) return DG_ERR_TOO_LARGE;
  if (m == 0 || n == 0) return DG_OK;
  const DensePlan p = plan_dense(kDense, m, n, k, has_c != 0, num_sms, true);
  *block_m = p.decode ? p.decode_tn : (p.pair || p.tall) ? 2 * kBlockM : p.short_a ? kBlockM / 2 : kBlockM;
  *block_n = p.block_n;
  *split_k = p.ksplit;
  *cta_pair = p.pair ? 1 : 0;
  *stream_k = p.stream_k ? 1 : 0;
  *swap_ab = p.decode ? 1 : 0;
  *multicast = p.multicast ? 1 : 0;
  return DG_OK;
}

dg_status dg_plan_fp8_gemm_nt(int64_t m, int64_t n, int64_t k, int32_t has_c, int32_t num_sms,
                              int32_t* block_m, int32_t* block_n, int32_t* split_k,
                              int32_t* cta_pair) {
  if (!block_m || !block_n || !split_k || !cta_pair) return DG_ERR_INVALID_ARG;
  *block_m = *block_n = *split_k = *cta_pair = 0;
  if (m < 0 || num_sms < 1) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (m >= kMaxCoord) return DG_ERR_TOO_LARGE;
  if (m == 0 || n == 0) return DG_OK;  // nothing is launched
  const DensePlan p = plan_dense(kDense, m, n, k, has_c != 0, num_sms);
  *block_m = p.decode ? p.decode_tn : (p.pair || p.tall) ? 2 * kBlockM : p.short_a ? kBlockM / 2 : kBlockM;
  *block_n = p.block_n;
  *split_k = p.ksplit;
  *cta_pair = p.pair ? 1 : 0;
  return DG_OK;
}

dg_status dg_plan_m_grouped_fp8_gemm_nt_contiguous(int64_t m_sum, int64_t n, int64_t k,
                                                   int32_t num_groups, int32_t num_sms,
                                                   int32_t* block_m, int32_t* block_n) {
  if (!block_m || !block_n) return DG_ERR_INVALID_ARG;
  *block_m = *block_n = 0;
  if (m_sum < 0 || num_groups < 0 || num_sms < 1) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (m_sum == 0 || n == 0 || num_groups == 0) return DG_OK;
  if (m_sum % kBlockM != 0) return DG_ERR_ALIGNMENT;
  if (m_sum >= kMaxCoord || (int64_t)num_groups * n >= kMaxCoord) return DG_ERR_TOO_LARGE;
  const GroupedPlan p = plan_contiguous(m_sum, n, k, num_groups, num_sms);
  *block_m = p.tall ? 2 * kBlockM : kBlockM;
  *block_n = p.block_n;
  return DG_OK;
}

dg_status dg_plan_m_grouped_fp8_gemm_nt_masked(int32_t num_groups, int64_t max_m, int64_t n,
                                               int64_t k, int64_t expected_m, int32_t num_sms,
                                               int32_t* block_m, int32_t* block_n,
                                               int32_t* cta_pair) {
  if (!block_m || !block_n || !cta_pair) return DG_ERR_INVALID_ARG;
  *block_m = *block_n = *cta_pair = 0;
  if (max_m < 0 || num_groups < 0 || expected_m < 0 || num_sms < 1) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (max_m == 0 || n == 0 || num_groups == 0) return DG_OK;
  if (num_groups > kMaxMaskedGroups) return DG_ERR_TOO_LARGE;
  if (max_m >= kMaxCoord || (int64_t)num_groups * max_m >= kMaxCoord) return DG_ERR_TOO_LARGE;
  const GroupedPlan p = plan_masked(num_groups, max_m, n, k, expected_m, num_sms);
  *block_m = p.pair ? 2 * kBlockM : kBlockM;
  *block_n = p.block_n;
  *cta_pair = p.pair ? 1 : 0;
  return DG_OK;
}

dg_status dg_fp8_gemm_nt_fp32_sf(const void* a, const float* sfa, const void* b, const float* sfb,
                                 const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                                 int64_t ldb, int64_t ldc, int64_t ldd, void* stream) {
  if (m < 0) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (m == 0 || n == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d) return DG_ERR_INVALID_ARG;
  if (lda < k || ldb < k || ldd < n || (c && ldc < n)) return DG_ERR_INVALID_ARG;
  if (lda % 16 || ldb % 16 || ldd % 8 || (c && ldc % 8)) return DG_ERR_ALIGNMENT;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d) || (c && !aligned16(c)) ||
      (reinterpret_cast<uintptr_t>(sfa) & 3u) || (reinterpret_cast<uintptr_t>(sfb) & 3u))
    return DG_ERR_ALIGNMENT;
  if (m >= kMaxCoord) return DG_ERR_TOO_LARGE;
  int sms = 0;
  if ((s = current_device(&sms)) != DG_OK) return s;
  if ((s = get_encoder()) != DG_OK) return s;
  Operands o;
  {
    uint64_t dims_a[2] = {(uint64_t)k, (uint64_t)m};
    uint64_t str_a[1] = {(uint64_t)lda};
    uint32_t box[2] = {(uint32_t)kBlockK, (uint32_t)kBlockM};
    if ((s = encode(&o.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a, dims_a, str_a, box,
                    CU_TENSOR_MAP_SWIZZLE_128B)) != DG_OK)
      return s;
    // B tiles of 256 rows (the promotion kernel's 128 x 256 output tiles)
    uint64_t dims_b[3] = {(uint64_t)k, (uint64_t)n, 1};
    uint64_t str_b[2] = {(uint64_t)ldb, (uint64_t)(n * ldb)};
    uint32_t box_b[3] = {(uint32_t)kBlockK, 256, 1};
    if ((s = encode(&o.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, b, dims_b, str_b, box_b,
                    CU_TENSOR_MAP_SWIZZLE_128B)) != DG_OK)
      return s;
  }
  if ((s = encode_d(o, d, m, n, ldd)) != DG_OK) return s;
  GemmArgs args = {};
  args.c = static_cast<const __nv_bfloat16*>(c);
  args.d = static_cast<__nv_bfloat16*>(d);
  args.ldc = c ? ldc : 0;
  args.ldd = ldd;
  args.m = (int32_t)m;
  args.n = (int32_t)n;
  args.k = (int32_t)k;
  args.num_groups = 1;
  args.m_blocks = (int32_t)((m + kBlockM - 1) / kBlockM);
  args.n_blocks = (int32_t)((n + 255) / 256);
  args.k_blocks = (int32_t)(k / kBlockK);
  args.band = env().raster_band;
  if (args.band < 1) args.band = 1;
  args.timeout_ns = g_timeout_ns.load();
  args.pdl = g_pdl.load();
  args.sfa_f32 = sfa;
  args.sfb_f32 = sfb;
  args.sfa_ld = (int32_t)align4(m);
  const int64_t tiles = (int64_t)args.m_blocks * args.n_blocks;
  if (tiles >= kMaxCoord) return DG_ERR_TOO_LARGE;
  const int grid = (int)(tiles < sms ? tiles : sms);
  print_config("fp8_gemm_nt_fp32_sf (promotion)", m, n, k, 1, kBlockM, 256, gemm_promote_stages(), grid,
               args.band);
  return from_cuda(gemm_promote_launch(o.a, o.b, o.d, args, grid, static_cast<cudaStream_t>(stream)));
}

dg_status dg_fp8_gemm_nn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream) {
  return dense_gemm(kDenseNN, "fp8_gemm_nn", a, sfa, b, sfb, c, d, m, n, k, lda, ldb, ldc, ldd,
                    stream);
}

dg_status dg_fp8_gemm_tn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream) {
  return dense_gemm(kDenseTN, "fp8_gemm_tn", a, sfa, b, sfb, c, d, m, n, k, lda, ldb, ldc, ldd,
                    stream);
}

dg_status dg_fp8_gemm_tt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream) {
  return dense_gemm(kDenseTT, "fp8_gemm_tt", a, sfa, b, sfb, c, d, m, n, k, lda, ldb, ldc, ldd,
                    stream);
}

dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b,
                                              const int32_t* sfb, void* d,
                                              const int32_t* m_indices, int64_t m_sum, int64_t n,
                                              int64_t k, int32_t num_groups, void* stream) {
  if (m_sum < 0 || num_groups < 0) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (m_sum == 0 || n == 0 || num_groups == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d || !m_indices) return DG_ERR_INVALID_ARG;
  if (m_sum % kBlockM != 0) return DG_ERR_ALIGNMENT;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(d))
    return DG_ERR_ALIGNMENT;
  if (m_sum >= kMaxCoord || (int64_t)num_groups * n >= kMaxCoord) return DG_ERR_TOO_LARGE;
  int sms = 0;
  if ((s = current_device(&sms)) != DG_OK) return s;
  if ((s = get_encoder()) != DG_OK) return s;

  GemmArgs args = {};
  args.m_blocks = (int32_t)(m_sum / kBlockM);
  const GroupedPlan plan = plan_contiguous(m_sum, n, k, num_groups, sms);
  const bool tall = plan.tall;
  const int block_n = plan.block_n;
  Operands o;
  if ((s = encode_a_2d(o, a, sfa, m_sum, k, k)) != DG_OK) return s;
  if ((s = encode_b_side(o, b, sfb, num_groups, n, k, k, block_n, block_n)) != DG_OK) return s;
  if ((s = encode_d(o, d, m_sum, n, n)) != DG_OK) return s;
  args.d = static_cast<__nv_bfloat16*>(d);
  args.ldd = n;
  args.m_indices = m_indices;
  args.m = (int32_t)m_sum;
  args.n = (int32_t)n;
  args.k = (int32_t)k;
  args.num_groups = num_groups;
  args.n_blocks = (int32_t)((n + block_n - 1) / block_n);
  args.k_blocks = (int32_t)(k / kBlockK);
  args.band = env().raster_band / (tall ? 2 : 1);
  if (args.band < 1) args.band = 1;
  args.timeout_ns = g_timeout_ns.load();
  args.pdl = g_pdl.load();
  const int64_t tiles = (int64_t)args.m_blocks * args.n_blocks;
  if (tiles >= kMaxCoord) return DG_ERR_TOO_LARGE;
  const int grid = (int)(tiles < sms ? tiles : sms);
  print_config(tall ? "m_grouped_fp8_gemm_nt_contiguous (256-row tiles)" : "m_grouped_fp8_gemm_nt_contiguous",
               m_sum, n, k, num_groups, tall ? 2 * kBlockM : kBlockM, block_n,
               tall ? gemm_tall_stages(block_n) : gemm_stages(block_n), grid, args.band);
  if (tall)
    return from_cuda(gemm_tall_launch(kContiguous, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid,
                                      static_cast<cudaStream_t>(stream)));
  return from_cuda(gemm_launch(kContiguous, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid,
                               static_cast<cudaStream_t>(stream)));
}

dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void* a, const int32_t* sfa, const void* b,
                                              const int32_t* sfb, const float* c, float* d,
                                              const int32_t* ks, int64_t m, int64_t n,
                                              int64_t sum_k, int32_t num_groups, void* stream) {
  if (m < 0 || n < 0 || sum_k < 0 || num_groups < 0) return DG_ERR_INVALID_ARG;
  if (m % 16 != 0 || n % 16 != 0 || sum_k % kBlockK != 0) return DG_ERR_ALIGNMENT;
  if (m == 0 || n == 0 || num_groups == 0) return DG_OK;
  if (num_groups > kMaxMaskedGroups) return DG_ERR_TOO_LARGE;
  if (!d || !ks) return DG_ERR_INVALID_ARG;
  if (!aligned16(d) || (c && !aligned16(c))) return DG_ERR_ALIGNMENT;
  if (m >= kMaxCoord || n >= kMaxCoord || sum_k >= kMaxCoord ||
      (int64_t)num_groups * m >= kMaxCoord)
    return DG_ERR_TOO_LARGE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t out_bytes = (size_t)num_groups * (size_t)m * (size_t)n * sizeof(float);
  if (sum_k == 0) {
    // every expert is empty: D = C (or 0)
    if (c == d) return DG_OK;
    return from_cuda(c ? cudaMemcpyAsync(d, c, out_bytes, cudaMemcpyDeviceToDevice, st)
                       : cudaMemsetAsync(d, 0, out_bytes, st));
  }
  if (!a || !sfa || !b || !sfb) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb)) return DG_ERR_ALIGNMENT;
  dg_status s;
  int sms = 0;
  if ((s = current_device(&sms)) != DG_OK) return s;
  if ((s = get_encoder()) != DG_OK) return s;

  GemmArgs args = {};
  args.m_blocks = (int32_t)((m + kBlockM - 1) / kBlockM);
  // 128 or 256 columns (whole MN-major boxes): the compute-bound estimate
  // over the average K blocks per expert
  const int64_t kb_avg = std::max<int64_t>(1, sum_k / kBlockK / num_groups);
  int block_n = 256;
  {
    const int forced = env().block_n;
    if (forced == 128 || forced == 256) {
      block_n = forced;
    } else {
      double best = 1e300;
      for (int w : {128, 256}) {
        const int64_t tiles = (int64_t)num_groups * args.m_blocks * ((n + w - 1) / w);
        const double waves = (double)((tiles + sms - 1) / sms);
        const double cost = waves * ((double)kb_avg + (w == 256 ? 4.0 : 0.5)) * w / (w == 256 ? 1.6 : 1.0);
        if (cost < best * 0.999) {
          best = cost;
          block_n = w;
        }
      }
    }
  }
  Operands o;
  if ((s = encode_a_mn(o, a, sfa, m, sum_k, m)) != DG_OK) return s;
  if ((s = encode_b_mn(o, b, sfb, n, sum_k, n, block_n)) != DG_OK) return s;
  {
    // FP32 D as a 2-D tensor [num_groups * m, n]: 16 x 32 boxes with the
    // 64-byte swizzle the epilogue stages in
    uint64_t dims_d[2] = {(uint64_t)n, (uint64_t)num_groups * (uint64_t)m};
    uint64_t str_d[1] = {(uint64_t)(n * 4)};
    uint32_t box_d[2] = {16, 32};
    if ((s = encode(&o.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, d, dims_d, str_d, box_d,
                    CU_TENSOR_MAP_SWIZZLE_64B)) != DG_OK)
      return s;
  }
  args.c_f32 = c;
  args.d_f32 = d;
  args.ks = ks;
  args.m = (int32_t)m;
  args.n = (int32_t)n;
  args.k = (int32_t)sum_k;
  args.num_groups = num_groups;
  args.n_blocks = (int32_t)((n + block_n - 1) / block_n);
  args.k_blocks = (int32_t)(sum_k / kBlockK);
  args.band = env().raster_band;
  if (args.band < 1) args.band = 1;
  args.timeout_ns = g_timeout_ns.load();
  args.pdl = g_pdl.load();
  const int64_t tiles = (int64_t)num_groups * args.m_blocks * args.n_blocks;
  if (tiles >= kMaxCoord) return DG_ERR_TOO_LARGE;
  // 256-column tiles drain their accumulator with eight epilogue warps
  // (DG_TALL_EPI8 = 0: four, each reading its 256 columns in two halves);
  // with them, clusters of two CTAs on adjacent M blocks of one expert share
  // each B tile by TMA multicast (DG_MULTICAST = 0 turns it off), on an even grid
  args.epi8 = (block_n == 256 && env().tall_epi8 != 0) ? 1 : 0;
  args.mc = (args.epi8 && env().multicast != 0 && sms >= 2 && args.m_blocks >= 2) ? 1 : 0;
  const int64_t pair_tiles = (int64_t)num_groups * ((args.m_blocks + 1) / 2) * args.n_blocks;
  const int grid = args.mc ? 2 * (int)(pair_tiles < sms / 2 ? pair_tiles : sms / 2)
                           : (int)(tiles < sms ? tiles : sms);
  print_config(args.epi8 ? "k_grouped_fp8_gemm_tn_contiguous (eight epilogue warps)"
                         : "k_grouped_fp8_gemm_tn_contiguous",
               m, n, sum_k, num_groups, kBlockM, block_n, gemm_stages(block_n), grid, args.band);
  return from_cuda(gemm_launch(kKGrouped, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid, st));
}

dg_status dg_m_grouped_fp8_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b,
                                          const int32_t* sfb, void* d, const int32_t* masked_m,
                                          int32_t num_groups, int64_t max_m, int64_t n, int64_t k,
                                          int64_t expected_m, void* stream) {
  if (max_m < 0 || num_groups < 0 || expected_m < 0) return DG_ERR_INVALID_ARG;
  dg_status s = check_common_k_n(n, k);
  if (s != DG_OK) return s;
  if (max_m == 0 || n == 0 || num_groups == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d || !masked_m) return DG_ERR_INVALID_ARG;
  if (num_groups > kMaxMaskedGroups) return DG_ERR_TOO_LARGE;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(d))
    return DG_ERR_ALIGNMENT;
  if (max_m >= kMaxCoord || (int64_t)num_groups * max_m >= kMaxCoord) return DG_ERR_TOO_LARGE;
  int sms = 0;
  if ((s = current_device(&sms)) != DG_OK) return s;
  if ((s = get_encoder()) != DG_OK) return s;

  GemmArgs args = {};
  args.m_blocks = (int32_t)((max_m + kBlockM - 1) / kBlockM);
  const GroupedPlan plan = plan_masked(num_groups, max_m, n, k, expected_m, sms);
  const bool pair = plan.pair;
  const int block_n = plan.block_n;
  int grid_units = sms;
  if (pair) {
    grid_units = gemm2_max_clusters(kMasked, block_n);
    if (grid_units > sms / 2) grid_units = sms / 2;
    if (grid_units <= 0) return DG_ERR_CUDA;
  }
  Operands o;
  if ((s = encode_a_3d(o, a, sfa, num_groups, max_m, k)) != DG_OK) return s;
  if ((s = encode_b_side(o, b, sfb, num_groups, n, k, k, block_n, pair ? block_n / 2 : block_n)) != DG_OK)
    return s;
  if ((s = encode_d(o, d, (int64_t)num_groups * max_m, n, n)) != DG_OK) return s;
  args.d = static_cast<__nv_bfloat16*>(d);
  args.ldd = n;
  args.masked_m = masked_m;
  args.m = (int32_t)max_m;
  args.n = (int32_t)n;
  args.k = (int32_t)k;
  args.num_groups = num_groups;
  args.n_blocks = (int32_t)((n + block_n - 1) / block_n);
  args.k_blocks = (int32_t)(k / kBlockK);
  args.band = 1;
  args.timeout_ns = g_timeout_ns.load();
  args.pdl = g_pdl.load();
  if ((int64_t)num_groups * args.m_blocks * args.n_blocks >= kMaxCoord) return DG_ERR_TOO_LARGE;
  if (pair) {
    print_config("m_grouped_fp8_gemm_nt_masked (cta pair)", max_m, n, k, num_groups, 2 * kBlockM, block_n,
                 6, 2 * grid_units, 0);
    return from_cuda(gemm2_launch(kMasked, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid_units,
                                  static_cast<cudaStream_t>(stream)));
  }
  print_config("m_grouped_fp8_gemm_nt_masked", max_m, n, k, num_groups, kBlockM, block_n,
               gemm_stages(block_n), grid_units, 0);
  return from_cuda(gemm_launch(kMasked, block_n, o.a, o.b, o.sfa, o.sfb, o.d, args, grid_units,
                               static_cast<cudaStream_t>(stream)));
}

dg_status dg_quantize_fp8(const float* x, void* q, void* sf, int64_t groups, int64_t rows,
                          int64_t cols, int32_t block_rows, int32_t sf_format, void* stream) {
  if (groups < 0 || rows < 0 || cols < 0) return DG_ERR_INVALID_ARG;
  if (block_rows != 1 && block_rows != 128) return DG_ERR_INVALID_ARG;
  if (sf_format != DG_SF_FP32 && sf_format != DG_SF_UE8M0_PACKED) return DG_ERR_INVALID_ARG;
  if (cols % kBlockK != 0) return DG_ERR_ALIGNMENT;
  if (groups == 0 || rows == 0 || cols == 0) return DG_OK;
  if (!x || !q || !sf) return DG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return DG_ERR_ALIGNMENT;
  if (groups * rows >= kMaxCoord * 16 || cols >= kMaxCoord) return DG_ERR_TOO_LARGE;
  int sms = 0;
  dg_status s = current_device(&sms);
  if (s != DG_OK) return s;
  return from_cuda(quantize_launch(x, q, sf, groups, rows, cols, block_rows, sf_format, g_pdl.load() != 0,
                                   static_cast<cudaStream_t>(stream)));
}

dg_status dg_quantize_fp8_cols(const float* x, void* q, void* sf, int64_t rows, int64_t cols,
                               int32_t sf_format, void* stream) {
  if (rows < 0 || cols < 0) return DG_ERR_INVALID_ARG;
  if (sf_format != DG_SF_FP32 && sf_format != DG_SF_UE8M0_PACKED) return DG_ERR_INVALID_ARG;
  if (rows % kBlockK != 0 || cols % 4 != 0) return DG_ERR_ALIGNMENT;
  if (rows == 0 || cols == 0) return DG_OK;
  if (!x || !q || !sf) return DG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return DG_ERR_ALIGNMENT;
  if (rows >= kMaxCoord * 16 || cols >= kMaxCoord) return DG_ERR_TOO_LARGE;
  int sms = 0;
  dg_status s = current_device(&sms);
  if (s != DG_OK) return s;
  return from_cuda(quantize_cols_launch(x, q, sf, rows, cols, sf_format, g_pdl.load() != 0,
                                        static_cast<cudaStream_t>(stream)));
}

dg_status dg_transform_sf(const float* sf, int32_t* packed, int64_t groups, int64_t mn, int64_t k,
                          int32_t block_rows, void* stream) {
  if (groups < 0 || mn < 0 || k < 0) return DG_ERR_INVALID_ARG;
  if (block_rows != 1 && block_rows != 128) return DG_ERR_INVALID_ARG;
  if (groups == 0 || mn == 0 || k == 0) return DG_OK;
  if (!sf || !packed) return DG_ERR_INVALID_ARG;
  if (!aligned16(packed) || (reinterpret_cast<uintptr_t>(sf) & 3u)) return DG_ERR_ALIGNMENT;
  if (groups * align4(mn) * ((k + 511) / 512) >= kMaxCoord * 64) return DG_ERR_TOO_LARGE;
  int sms = 0;
  dg_status s = current_device(&sms);
  if (s != DG_OK) return s;
  return from_cuda(transform_sf_launch(sf, packed, groups, mn, k, block_rows, g_pdl.load() != 0,
                                       static_cast<cudaStream_t>(stream)));
}

int64_t dg_get_tma_aligned_size(int64_t x, int32_t element_size) {
  if (x < 0 || element_size <= 0 || 16 % element_size != 0) return -1;
  const int64_t unit = 16 / element_size;
  return (x + unit - 1) / unit * unit;
}

int32_t dg_get_mk_alignment_for_contiguous_layout(void) { return g_mk_alignment.load(); }

dg_status dg_set_mk_alignment_for_contiguous_layout(int32_t alignment) {
  if (alignment <= 0 || alignment % kBlockM != 0 || alignment > 4096) return DG_ERR_INVALID_ARG;
  g_mk_alignment.store(alignment);
  return DG_OK;
}

dg_status dg_set_num_sms(int32_t n) {
  if (n < 0) return DG_ERR_INVALID_ARG;
  g_num_sms_limit.store(n);
  return DG_OK;
}

int32_t dg_get_num_sms(void) {
  const int32_t limit = g_num_sms_limit.load();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return limit;
  int sms = 0;
  if (current_device(&sms) != DG_OK) return limit;
  return sms;
}

dg_status dg_set_pdl(int32_t enable) {
  if (enable != 0 && enable != 1) return DG_ERR_INVALID_ARG;
  g_pdl.store(enable);
  return DG_OK;
}

int32_t dg_get_pdl(void) { return g_pdl.load(); }

dg_status dg_set_wait_timeout_ns(uint64_t ns) {
  if (ns == 0) return DG_ERR_INVALID_ARG;
  g_timeout_ns.store(ns);
  return DG_OK;
}

dg_status dg_debug_set_drop_load(int32_t k) {
  if (k < 0) return DG_ERR_INVALID_ARG;
  g_debug_drop_load.store(k);
  return DG_OK;
}

dg_status dg_debug_plant_check(int32_t on) {
#if defined(DG_DEBUG_CHECKS) && DG_DEBUG_CHECKS
  g_debug_plant_check.store(on != 0 ? 1 : 0);
  return DG_OK;
#else
  if (on != 0) return DG_ERR_INVALID_ARG;  // the release kernels carry no checks
  return DG_OK;
#endif
}

dg_status dg_get_device_error(void* stream, uint64_t* detail) {
  if (detail) *detail = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DG_ERR_CUDA;
  unsigned long long g = 0, q = 0;
  if (gemm_fetch_error(&g) != cudaSuccess) return DG_ERR_CUDA;
  if (quant_fetch_error(&q) != cudaSuccess) return DG_ERR_CUDA;
  const unsigned long long w = g ? g : q;
  if (detail) *detail = w;
  return w ? static_cast<dg_status>(w & 0xFFu) : DG_OK;
}

const char* dg_status_string(dg_status s) {
  switch (s) {
    case DG_OK: return "ok";
    case DG_ERR_INVALID_ARG: return "invalid argument";
    case DG_ERR_ALIGNMENT: return "alignment or divisibility requirement not met";
    case DG_ERR_UNSUPPORTED_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case DG_ERR_CUDA: return "CUDA runtime or driver call failed";
    case DG_ERR_DEVICE_TIMEOUT: return "device: a pipeline wait exceeded its time limit";
    case DG_ERR_DEVICE_BAD_INDEX: return "device: group index or masked count out of range";
    case DG_ERR_TOO_LARGE: return "size beyond the supported range";
    case DG_ERR_DEVICE_BAD_SCALE: return "device: scale is not a positive power of two";
    case DG_ERR_DEVICE_CHECK: return "device: a bound checked by the debug library failed";
  }
  return "unknown status";
}

int32_t dg_version(void) { return 100; }

}  // extern "C"
