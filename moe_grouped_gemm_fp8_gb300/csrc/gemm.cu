// FP8 GEMM with fine-grained scaling on sm_103a: D = C + A @ B.T, dense and
// M-grouped (contiguous / masked).
//
// Operation and layouts: "DeepGEMM: kernels GEMM FP8 limpos e eficientes por
// meio de scaling granular" (pt.news.hada.io), sections "Interface GEMM e
// restrições de layout" and "GEMM denso e grouped".  The Hopper design the
// pages sketch (warp specialisation overlapping TMA data movement, tensor-core
// MMA and CUDA-core promotion; launch report on feifmx.com, Feb 2025) is
// re-done for Blackwell: the per-128-K scales are applied by the tensor core
// itself (tcgen05 block-scaled MMA with UE8M0 scales held in TMEM) and the
// FP32 accumulator lives in TMEM, so no CUDA-core promotion is needed.
//
// One persistent CTA per SM (192 threads, 6 warps):
//   warp 0      TMA producer: A tile [128 x 128], B tile [BN x 128] (E4M3,
//               128-byte swizzle) and the packed scale words of both into an
//               S-stage shared-memory ring guarded by full/empty mbarriers.
//   warp 1      TMEM owner and MMA issuer: turns the scale words of a stage
//               into the 32x128b layout tcgen05.cp expects, copies them to
//               TMEM and issues four 128 x BN x 32 block-scaled MMAs per
//               128-wide K block into a TMEM accumulator (double-buffered
//               when the columns allow it).
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (one 32-lane quarter
//               each), + C, round to BF16, predicated 16-byte stores of the
//               rows the grouped layouts allow.
// Every mbarrier wait is bounded; on expiry the kernel records an error,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_device.cuh"

namespace dg {

__device__ unsigned long long g_gemm_err = 0ull;

template <int BN>
struct GemmLayout {
  static constexpr int kSfbChunks = (BN + 127) / 128;  // 128-row chunks of B scales
  static constexpr int kBytesA = kBlockM * kBlockK;
  static constexpr int kBytesB = BN * kBlockK;
  static constexpr int kOffB = kBytesA;
  static constexpr int kOffSfaRaw = kOffB + kBytesB;          // 128 words from TMA
  static constexpr int kOffSfbRaw = kOffSfaRaw + 512;         // BN words from TMA
  static constexpr int kOffSfaT = kOffSfbRaw + kSfbChunks * 512;  // 32x128b chunk
  static constexpr int kOffSfbT = kOffSfaT + 512;                 // kSfbChunks chunks
  static constexpr int kStageBytes = (kOffSfbT + kSfbChunks * 512 + 1023) / 1024 * 1024;
  static constexpr uint32_t kTxBytes = kBytesA + kBytesB + 128 * 4 + BN * 4;
  static constexpr int kSfCols = 4 + 4 * kSfbChunks;  // TMEM columns per stage for scales
};

template <int BN, int STAGES>
struct TmemPlan {
  static constexpr int kNumAcc = (2 * BN + STAGES * GemmLayout<BN>::kSfCols <= 512) ? 2 : 1;
  static constexpr int kSfBase = kNumAcc * BN;
  static_assert(kSfBase + STAGES * GemmLayout<BN>::kSfCols <= 512, "TMEM over-subscribed");
};

// Control block after the stage ring.
struct Ctrl {
  static constexpr int kBarriers(int stages, int num_acc) { return 2 * stages + 2 * num_acc + 1; }
};

static constexpr size_t ctrl_bytes(int stages, int num_acc, int mode) {
  return (size_t)8 * (2 * stages + 2 * num_acc + 1) + 16 +
         (mode == kMasked ? (size_t)4 * (2 * kMaxMaskedGroups + 1) : 0);
}

struct Tile {
  int g, mb, nb;
};

// Maps a linear tile index to (group, M block, N block).  Dense and
// contiguous tiles are rastered in bands of `band` M blocks: inside a band the
// M block varies fastest, so a wave of CTAs shares a few B column blocks and
// one band of A.  Masked tiles are enumerated group by group (M block
// fastest) from a prefix table built at kernel start.
template <int MODE>
struct Scheduler {
  const GemmArgs* args;
  const int* tile_start;   // masked: [G + 1]
  const int* group_valid;  // masked: [G]
  int total;
  int cursor;              // masked: current group (tile indices only increase)

  __device__ bool get(int t, Tile& tile) {
    if (MODE == kMasked) {
      while (t >= tile_start[cursor + 1]) ++cursor;
      const int local = t - tile_start[cursor];
      const int mbs = (group_valid[cursor] + kBlockM - 1) / kBlockM;
      tile.g = cursor;
      tile.mb = local % mbs;
      tile.nb = local / mbs;
      return true;
    }
    const int per_band = args->band * args->n_blocks;
    const int b = t / per_band;
    const int rem = t - b * per_band;
    const int rows = min(args->band, args->m_blocks - b * args->band);
    tile.nb = rem / rows;
    tile.mb = b * args->band + rem % rows;
    tile.g = 0;
    if (MODE == kContiguous) {
      const int g = __ldg(args->m_indices + (int64_t)tile.mb * kBlockM);
      if (g < 0) return false;
      if (g >= args->num_groups) {
        record_error(&g_gemm_err, DG_ERR_DEVICE_BAD_INDEX, kSiteContiguousIndex);
        return false;
      }
      tile.g = g;
    }
    return true;
  }
};

// Waits until the phase with `parity` of `bar` has completed, ignoring the
// abort flag (used to drain in-flight work before exit), bounded in time.
static __device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                        uint32_t site) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0 && (global_timer_ns() - t0 > timeout_ns || it >= (1u << 30))) {
      record_error(&g_gemm_err, DG_ERR_DEVICE_TIMEOUT, site);
      return;
    }
  }
}

// Lane 0 waits, the result is broadcast, and the warp reconverges (so the
// other lanes observe what lane 0 acquired).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, uint32_t site) {
  const int lane = threadIdx.x & 31;
  int ok = 0;
  if (lane == 0) ok = wait_bounded(bar, parity, abort_flag, timeout_ns, &g_gemm_err, site) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Byte `shift/8` of a packed scale word, repeated in all four bytes, so the
// MMA reads the scale of the current K block whichever byte it selects.
__device__ __forceinline__ uint32_t splat_byte(uint32_t w, int shift) {
  return ((w >> shift) & 0xFFu) * 0x01010101u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int BN, int STAGES, int MODE>
__global__ void __launch_bounds__(192, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfa,
                    const __grid_constant__ CUtensorMap tm_sfb, const GemmArgs args) {
  using L = GemmLayout<BN>;
  using T = TmemPlan<BN, STAGES>;
  constexpr int NUM_ACC = T::kNumAcc;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * L::kStageBytes);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto tempty = [&](int a) { return smem_u32(bars + 2 * STAGES + NUM_ACC + a); };
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 2 * NUM_ACC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NUM_ACC + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
  int* group_valid = tile_start + (kMaxMaskedGroups + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_sfa);
    tma_prefetch_desc(&tm_sfb);
  }
  if (MODE == kMasked && warp == 2) {
    for (int g = lane; g < args.num_groups; g += 32) {
      const int v = __ldg(args.masked_m + g);
      const int c = v < 0 ? 0 : (v > args.m ? args.m : v);
      if (c != v) record_error(&g_gemm_err, DG_ERR_DEVICE_BAD_INDEX, kSiteMaskedCount);
      group_valid[g] = c;
    }
    __syncwarp();
    if (lane == 0) {
      int acc = 0;
      for (int g = 0; g < args.num_groups; ++g) {
        tile_start[g] = acc;
        acc += (group_valid[g] + kBlockM - 1) / kBlockM * args.n_blocks;
      }
      tile_start[args.num_groups] = acc;
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  Scheduler<MODE> sched;
  sched.args = &args;
  sched.tile_start = tile_start;
  sched.group_valid = group_valid;
  sched.cursor = 0;
  sched.total = MODE == kMasked ? tile_start[args.num_groups] : args.m_blocks * args.n_blocks;
  const uint64_t tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      for (int t = blockIdx.x; t < sched.total; t += gridDim.x) {
        Tile tile;
        if (!sched.get(t, tile)) continue;
        bool ok = true;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!wait_bounded(empty(stage), phase ^ 1u, abort_flag, tmo, &g_gemm_err,
                            kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t sb = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t fb = full(stage);
          mbar_arrive_expect_tx(fb, L::kTxBytes);
          const int kx = kb * kBlockK, my = tile.mb * kBlockM, kp = kb >> 2;
          if (MODE == kMasked) {
            tma_load_3d(sb, &tm_a, fb, kx, my, tile.g);
            tma_load_3d(sb + L::kOffSfaRaw, &tm_sfa, fb, my, kp, tile.g);
          } else {
            tma_load_2d(sb, &tm_a, fb, kx, my);
            tma_load_2d(sb + L::kOffSfaRaw, &tm_sfa, fb, my, kp);
          }
          tma_load_3d(sb + L::kOffB, &tm_b, fb, kx, tile.nb * BN, tile.g);
          tma_load_3d(sb + L::kOffSfbRaw, &tm_sfb, fb, tile.nb * BN, kp, tile.g);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Drain: every copy this thread issued has landed before smem is released.
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) wait_drain(full(s), (issued_parity >> s) & 1u, tmo, kSiteProducerDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_mxf8_e4m3(kBlockM, BN, 0, 0);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < sched.total && ok; t += gridDim.x) {
      Tile tile;
      if (!sched.get(t, tile)) continue;
      if (!warp_wait(tempty(acc), acc_phase ^ 1u, abort_flag, tmo, kSiteMmaTmemEmpty)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < args.k_blocks; ++kb) {
        if (!warp_wait(full(stage), phase, abort_flag, tmo, kSiteMmaFull)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * L::kStageBytes;
        const int shift = 8 * (kb & 3);
        {
          const uint32_t* raw = reinterpret_cast<const uint32_t*>(st + L::kOffSfaRaw);
          uint4 v;
          v.x = splat_byte(raw[lane], shift);
          v.y = splat_byte(raw[32 + lane], shift);
          v.z = splat_byte(raw[64 + lane], shift);
          v.w = splat_byte(raw[96 + lane], shift);
          *reinterpret_cast<uint4*>(st + L::kOffSfaT + lane * 16) = v;
        }
#pragma unroll
        for (int c = 0; c < L::kSfbChunks; ++c) {
          const uint32_t* raw = reinterpret_cast<const uint32_t*>(st + L::kOffSfbRaw + c * 512);
          uint4 v;
          v.x = splat_byte(raw[lane], shift);
          v.y = splat_byte(raw[32 + lane], shift);
          v.z = splat_byte(raw[64 + lane], shift);
          v.w = splat_byte(raw[96 + lane], shift);
          *reinterpret_cast<uint4*>(st + L::kOffSfbT + c * 512 + lane * 16) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sf_tmem = tmem_base + (uint32_t)(T::kSfBase + stage * L::kSfCols);
          tc_cp_32x128b_warpx4(sf_tmem, smem_desc_sf_chunk(smem_u32(st + L::kOffSfaT)));
#pragma unroll
          for (int c = 0; c < L::kSfbChunks; ++c)
            tc_cp_32x128b_warpx4(sf_tmem + 4 + 4 * c,
                                 smem_desc_sf_chunk(smem_u32(st + L::kOffSfbT + c * 512)));
          const uint64_t adesc = smem_desc_kmajor_sw128(smem_u32(st));
          const uint64_t bdesc = smem_desc_kmajor_sw128(smem_u32(st + L::kOffB));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_mxf8(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sf_tmem, sf_tmem + 4,
                        (kb | j) != 0 ? 1u : 0u);
          tc_commit(empty(stage));
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(tfull(acc));
      __syncwarp();
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Drain: all MMAs and TMEM copies issued here complete before TMEM is freed.
    if (lane == 0) {
      tc_commit(drain);
      wait_drain(drain, 0, tmo, kSiteDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < sched.total; t += gridDim.x) {
      Tile tile;
      if (!sched.get(t, tile)) continue;
      if (!warp_wait(tfull(acc), acc_phase, abort_flag, tmo, kSiteEpilogueTmemFull)) break;
      tc_fence_after();
      const int row = tile.mb * kBlockM + row_in_tile;
      bool row_ok;
      int64_t out_row;
      if (MODE == kDense) {
        row_ok = row < args.m;
        out_row = row;
      } else if (MODE == kContiguous) {
        const int gi = row < args.m ? __ldg(args.m_indices + row) : -1;
        row_ok = gi == tile.g;
        if (gi >= 0 && gi != tile.g)
          record_error(&g_gemm_err, DG_ERR_DEVICE_BAD_INDEX, kSiteContiguousIndex);
        out_row = row;
      } else {
        row_ok = row < group_valid[tile.g];
        out_row = (int64_t)tile.g * args.m + row;
      }
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tc_ld_32x32b_x32(taddr + ch * 32, r);
        tc_wait_ld();
        const int col0 = tile.nb * BN + ch * 32;
        if (row_ok && col0 < args.n) {
          __nv_bfloat16* dp = args.d + out_row * args.ldd + col0;
          const __nv_bfloat16* cp = args.c ? args.c + out_row * args.ldc + col0 : nullptr;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            if (col0 + 8 * p < args.n) {
              float f[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(r[8 * p + i]);
              if (cp) {
                const uint4 cv = *reinterpret_cast<const uint4*>(cp + 8 * p);
                const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  f[2 * i] += __uint_as_float(cw[i] << 16);
                  f[2 * i + 1] += __uint_as_float(cw[i] & 0xFFFF0000u);
                }
              }
              uint4 o;
              o.x = pack_bf16x2(f[0], f[1]);
              o.y = pack_bf16x2(f[2], f[3]);
              o.z = pack_bf16x2(f[4], f[5]);
              o.w = pack_bf16x2(f[6], f[7]);
              *reinterpret_cast<uint4*>(dp + 8 * p) = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(acc));
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------- host side

int gemm_max_stages(int block_n) { return block_n <= 128 ? 6 : 4; }

template <int BN, int STAGES>
static size_t smem_bytes_impl(int mode) {
  return (size_t)STAGES * GemmLayout<BN>::kStageBytes + 1024 +
         ctrl_bytes(STAGES, TmemPlan<BN, STAGES>::kNumAcc, mode);
}

size_t gemm_smem_bytes(int block_n, int stages, int mode) {
  (void)stages;
  return block_n <= 128 ? smem_bytes_impl<128, 6>(mode) : smem_bytes_impl<256, 4>(mode);
}

template <int BN, int STAGES, int MODE>
static cudaError_t launch_impl(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                               const CUtensorMap& sfb, const GemmArgs& args, int grid,
                               cudaStream_t stream) {
  auto kern = fp8_gemm_kernel<BN, STAGES, MODE>;
  const size_t smem = smem_bytes_impl<BN, STAGES>(MODE);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, a, b, sfa, sfb, args);
}

cudaError_t gemm_launch(int mode, int block_n, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& sfa, const CUtensorMap& sfb, const GemmArgs& args,
                        int grid, cudaStream_t stream) {
  if (block_n == 128) {
    switch (mode) {
      case kDense: return launch_impl<128, 6, kDense>(a, b, sfa, sfb, args, grid, stream);
      case kContiguous: return launch_impl<128, 6, kContiguous>(a, b, sfa, sfb, args, grid, stream);
      case kMasked: return launch_impl<128, 6, kMasked>(a, b, sfa, sfb, args, grid, stream);
    }
  } else if (block_n == 256) {
    switch (mode) {
      case kDense: return launch_impl<256, 4, kDense>(a, b, sfa, sfb, args, grid, stream);
      case kContiguous: return launch_impl<256, 4, kContiguous>(a, b, sfa, sfb, args, grid, stream);
      case kMasked: return launch_impl<256, 4, kMasked>(a, b, sfa, sfb, args, grid, stream);
    }
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
