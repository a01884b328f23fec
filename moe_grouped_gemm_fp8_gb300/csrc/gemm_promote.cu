// FP8 GEMM with arbitrary FP32 scales (the scale format the pages give for the
// Hopper path): D = C + sum_kb (A_kb @ B_kb^T) * sa[m, kb] * sb[n / 128, kb],
// one FP32 scale per 1x128 group of A and per 128x128 block of B, any value.
//
// "DeepGEMM: kernels GEMM FP8 limpos e eficientes por meio de scaling
// granular" (pt.news.hada.io), section "Interface GEMM e restrições de
// layout" (FP32 scale factors on SM90; LHS scales TMA-aligned and
// transposed), and the launch report on feifmx.com (Feb 2025): the tensor
// cores' FP8 partial sums are promoted to FP32 on the CUDA cores once per
// 128-wide K block (two-level accumulation).
//
// The block-scaled MMA of the main kernel only takes power-of-two (UE8M0)
// scales, so here the promotion is done explicitly, Blackwell-style: per K
// block the tensor core writes a fresh FP32 partial tile P = A_kb @ B_kb^T
// (tcgen05.mma kind::f8f6f4, no scaling) into one of four TMEM buffers; eight
// promotion warps (two per TMEM lane quarter, 64 columns each) read P with
// tcgen05.ld (both 32-column loads in flight at once), multiply by sa * sb and
// accumulate into FP32 registers (64 columns of one output row per thread),
// then run the usual epilogue (+ C, BF16, TMA store).  The MMAs run up to three K blocks ahead of the promotion (the
// commit-to-wake latency of a partial, ~650 cycles, is longer than its MMAs),
// and the next tile's MMAs overlap this tile's epilogue.
//
// One persistent CTA per SM, 10 warps: 0 TMA producer, 1 MMA issuer, 2-9
// promotion + epilogue.  128 x 128 output tiles.
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace dg {

constexpr int kPromoteThreads = 320;
constexpr int kPromoteWarps = 8;  // promotion / epilogue warps
constexpr int kPromoteBN = 128;
constexpr int kPromoteStages = 6;
constexpr int kPromoteStageBytes = 32768;  // A 128 x 128 + B 128 x 128, E4M3
constexpr int kPromoteBufs = 4;            // TMEM partial buffers of 128 columns

static constexpr size_t promote_smem_bytes() {
  return (size_t)kPromoteStages * kPromoteStageBytes + (size_t)kPromoteWarps * 2 * kEpiBuf + 1024 +
         8 * (2 * kPromoteStages + 2 * kPromoteBufs + 1) + 16;
}

// Instruction descriptor of kind::f8f6f4 without block scaling: FP32 D
// (bits 4-5 = 1), E4M3 A and B (bits 7-9, 10-12 = 0), both K-major, N / 8 at
// bit 17, M / 16 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f8_e4m3(uint32_t m, uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kPromoteThreads, 1)
    fp8_gemm_promote_kernel(const __grid_constant__ CUtensorMap tm_a,
                            const __grid_constant__ CUtensorMap tm_b,
                            const __grid_constant__ CUtensorMap tm_d, const GemmArgs args) {
  constexpr int STAGES = kPromoteStages;
  constexpr int BN = kPromoteBN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  uint8_t* epi_smem = smem + STAGES * kPromoteStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_smem + kPromoteWarps * 2 * kEpiBuf);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  constexpr int NB = kPromoteBufs;
  auto pfull = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
  auto pempty = [&](int b) { return smem_u32(bars + 2 * STAGES + NB + b); };
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 2 * NB);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NB + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned long long* const err = args.err;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(pfull(b), 1);
      mbar_init(pempty(b), kPromoteWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_d);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), NB * BN);  // NB 128-column partial buffers
    tmem_relinquish();
    tc_fence_before();
  }
  griddep_wait();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();

  Scheduler<kDense> sched;
  sched.args = &args;
  sched.tile_start = nullptr;
  sched.group_valid = nullptr;
  sched.cursor = 0;
  sched.kb_lo = 0;
  sched.kb_hi = args.k_blocks;
  sched.total = args.m_blocks * args.n_blocks;
  const int first_tile = (int)blockIdx.x, tile_stride = (int)gridDim.x;
  const uint64_t tmo = args.timeout_ns;
  const int kbs = args.k_blocks;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_parity = 0;
      bool ok = true;
      for (int t = first_tile; t < sched.total && ok; t += tile_stride) {
        Tile tile;
        sched.get(t, tile);
        for (int kb = 0; kb < kbs; ++kb) {
          if (!wait_one<kSuspendHintNs>(empty(stage), phase ^ 1u, abort_flag, tmo, err,
                                        kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t sb = smem_u32(smem + stage * kPromoteStageBytes);
          const uint32_t fb = full(stage);
          mbar_arrive_expect_tx(fb, kPromoteStageBytes);
          tma_load_2d(sb, &tm_a, fb, kb * kBlockK, tile.mb * kBlockM);
          tma_load_3d(sb + 16384, &tm_b, fb, kb * kBlockK, tile.nb * BN, 0);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s))
          wait_drain(full(s), (issued_parity >> s) & 1u, tmo, err, kSiteProducerDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f8_e4m3(kBlockM, BN);
      int stage = 0;
      uint32_t phase = 0, pk = 0;  // pk: partial tiles issued so far (buffer pk % NB)
      bool ok = true;
      for (int t = first_tile; t < sched.total && ok; t += tile_stride) {
        for (int kb = 0; kb < kbs; ++kb, ++pk) {
          if (!wait_one<kSuspendHintNs>(full(stage), phase, abort_flag, tmo, err, kSiteMmaFull) ||
              !wait_one<kSuspendHintNs>(pempty(pk % NB), ((pk / NB) & 1u) ^ 1u, abort_flag, tmo,
                                        err, kSiteMmaTmemEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = smem + stage * kPromoteStageBytes;
          const uint64_t adesc = smem_desc_kmajor_sw128(smem_u32(st));
          const uint64_t bdesc = smem_desc_kmajor_sw128(smem_u32(st + 16384));
          const uint32_t d_tmem = tmem_base + (pk % NB) * BN;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_f8(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, j != 0 ? 1u : 0u);
          tc_commit(empty(stage));
          tc_commit(pfull(pk % NB));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      tc_commit(drain);
      wait_drain(drain, 0, tmo, err, kSiteDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ promotion + epilogue
    const int quarter = warp & 3;
    const int colh = (warp - 2) >> 2;  // which 64 columns of the quarter's rows
    constexpr int HC = BN / 2;
    uint8_t* ebuf = epi_smem + (warp - 2) * 2 * kEpiBuf;
    uint32_t nchunk = 0, pk = 0;
    bool ok = true;
    for (int t = first_tile; t < sched.total && ok; t += tile_stride) {
      Tile tile;
      sched.get(t, tile);
      const int row0 = tile.mb * kBlockM + quarter * 32;
      const int row = row0 + lane;
      const bool row_ok = row < args.m;
      const float* sa_col = args.sfa_f32 + row;                       // + kb * sfa_ld
      const float* sb_row = args.sfb_f32 + (int64_t)tile.nb * kbs;    // + kb
      float acc[HC];
#pragma unroll
      for (int i = 0; i < HC; ++i) acc[i] = 0.0f;
      // scales are fetched kSd K blocks ahead (a global load's latency is
      // longer than one K block's promotion); slot j of the unrolled loop
      // always holds the scales of K block kb + j
      constexpr int kSd = 4;
      float sa_q[kSd], sb_q[kSd];
#pragma unroll
      for (int j = 0; j < kSd; ++j) {
        sa_q[j] = (row_ok && j < kbs) ? __ldg(sa_col + (int64_t)j * args.sfa_ld) : 0.0f;
        sb_q[j] = j < kbs ? __ldg(sb_row + j) : 0.0f;
      }
      for (int kb0 = 0; kb0 < kbs && ok; kb0 += kSd) {
#pragma unroll
      for (int j = 0; j < kSd; ++j) {
        const int kb = kb0 + j;
        if (kb >= kbs) break;
        const float s = sa_q[j] * sb_q[j];
        if (kb + kSd < kbs) {
          sa_q[j] = row_ok ? __ldg(sa_col + (int64_t)(kb + kSd) * args.sfa_ld) : 0.0f;
          sb_q[j] = __ldg(sb_row + kb + kSd);
        }
        if (!warp_wait<kSuspendHintNs>(pfull(pk % NB), (pk / NB) & 1u, abort_flag, tmo, err,
                                       kSiteEpilogueTmemFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + (pk % NB) * BN + colh * HC + ((uint32_t)(quarter * 32) << 16);
        uint32_t ra[32], rb[32];
        tc_ld_32x32b_x32(taddr, ra);
        tc_ld_32x32b_x32(taddr + 32, rb);
        tc_wait_ld_regs(ra);
        tc_wait_ld_regs(rb);
        // the partial is in registers: hand the buffer back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pempty(pk % NB));
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = fmaf(__uint_as_float(ra[i]), s, acc[i]);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[32 + i] = fmaf(__uint_as_float(rb[i]), s, acc[32 + i]);
        ++pk;
      }
      }
      if (!ok) break;
#pragma unroll
      for (int ch = 0; ch < HC / 32; ++ch) {
        const int col0 = tile.nb * BN + colh * HC + ch * 32;
        if (col0 >= args.n) continue;
        uint8_t* buf = ebuf + (nchunk & 1u) * kEpiBuf;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = acc[ch * 32 + i];
        emit_chunk_tma(f, buf, &tm_d, args, col0, row0, row0, true, lane);
        ++nchunk;
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, NB * BN);
  }
}

int gemm_promote_stages() { return kPromoteStages; }

cudaError_t gemm_promote_launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                                GemmArgs args, int grid, cudaStream_t stream) {
  static_assert(promote_smem_bytes() <= (size_t)kSmemLimit, "shared memory over the per-CTA limit");
  const size_t smem = promote_smem_bytes();
  unsigned long long* err = nullptr;
  cudaError_t e = error_word_address(&err);
  if (e != cudaSuccess) return e;
  args.err = err;
  e = set_smem_once<KernelTag<kPromoteBN, kPromoteStages, 100, 1, 1>>(
      fp8_gemm_promote_kernel, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kPromoteThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = args.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fp8_gemm_promote_kernel, a, b, d, args);
}

}  // namespace dg
