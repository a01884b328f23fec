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
// (tcgen05.mma kind::f8f6f4, no scaling, 128 x 256) into one of two TMEM
// buffers of 256 columns; eight promotion warps (two per TMEM lane quarter,
// 128 columns each: one 128 x 128 block of B, so one scale sb per warp and K
// block) read P with tcgen05.ld, 64 columns at a time, hand the buffer back,
// and accumulate acc = fma(P, sa * sb, acc) into 128 FP32 registers per
// thread (one output row's 128 columns); at the end of a tile the same warps
// add C, round to BF16 and TMA-store.  The MMA runs up to two K blocks ahead
// of the promotion, and the next tile's MMAs start while this tile's
// epilogue runs.
//
// One persistent CTA per SM, 12 warps: 0 TMA producer, 1 MMA issuer, 2-3
// idle, 4-11 promotion + epilogue.  The role warps give registers back with
// setmaxnreg (56 each) so that the promotion warps can hold their 128
// accumulators (224 each; 128 x 56 + 256 x 224 = 384 x 168, the launch's
// allotment).  128 x 256 output tiles: 48 KB of operands per K block for
// 8.4 MFLOP, against 32 KB for 4.2 MFLOP with 128 x 128 tiles.
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace dg {

constexpr int kPromoteThreads = 384;
constexpr int kPromoteWarps = 8;  // promotion / epilogue warps (4-11)
constexpr int kPromoteBN = 256;
constexpr int kPromoteStages = 4;
constexpr int kPromoteStageBytes = 16384 + 32768;  // A 128 x 128 + B 256 x 128, E4M3
constexpr int kPromoteBufs = 2;                     // TMEM partial buffers of 256 columns

// two staging chunks per promotion warp, so a chunk is staged while the
// previous one's TMA store still reads its buffer
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
    tmem_alloc(smem_u32(tmem_slot), NB * BN);  // NB 256-column partial buffers
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

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsRoles) : "memory");
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
            if (!wait_one<kSuspendHintNs, true>(empty(stage), phase ^ 1u, abort_flag, tmo, err,
                                                kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            const uint32_t sb = smem_u32(smem + stage * kPromoteStageBytes);
            const uint32_t fb = full(stage);
            DG_CHECK(err, tile.nb * BN < args.n && tile.mb * kBlockM < args.m, kSiteCheckLoadB);
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
            wait_drain<true>(full(s), (issued_parity >> s) & 1u, tmo, err, kSiteProducerDrain);
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
            if (!wait_one<kSuspendHintNs, true>(full(stage), phase, abort_flag, tmo, err, kSiteMmaFull) ||
                !wait_one<kSuspendHintNs, true>(pempty(pk % NB), ((pk / NB) & 1u) ^ 1u, abort_flag, tmo,
                                                err, kSiteMmaTmemEmpty)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint8_t* st = smem + stage * kPromoteStageBytes;
            const uint64_t adesc = smem_desc_kmajor_sw128(smem_u32(st));
            const uint64_t bdesc = smem_desc_kmajor_sw128(smem_u32(st + 16384));
            const uint32_t d_tmem = tmem_base + (pk % NB) * BN;
            DG_CHECK(err, args.debug_plant_check == 0 && (pk % NB) * BN + BN <= (uint32_t)(NB * BN),
                     kSiteCheckTmem);
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
        wait_drain<true>(drain, 0, tmo, err, kSiteDrain);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi) : "memory");
    // ------------------------------------------------------------ promotion + epilogue
    const int quarter = warp & 3;
    const int colh = (warp - 4) >> 2;  // which 128 columns (one block of B) of the quarter's rows
    constexpr int HC = BN / 2;
    uint8_t* ebuf = epi_smem + (warp - 4) * 2 * kEpiBuf;  // two staging chunks per warp
    uint32_t pk = 0;
    const int sb_blocks = (args.n + 127) / 128;  // rows of the B scale table
    bool ok = true;
    for (int t = first_tile; t < sched.total && ok; t += tile_stride) {
      Tile tile;
      sched.get(t, tile);
      const int row0 = tile.mb * kBlockM + quarter * 32;
      const int row = row0 + lane;
      const bool row_ok = row < args.m;
      const int bblk = tile.nb * 2 + colh;  // this warp's 128-column block of B
      const bool cols_ok = bblk < sb_blocks;
      const float* sa_col = args.sfa_f32 + row;                               // + kb * sfa_ld
      const float* sb_row = args.sfb_f32 + (int64_t)(cols_ok ? bblk : 0) * kbs;  // + kb
      float acc[HC];
#pragma unroll
      for (int i = 0; i < HC; ++i) acc[i] = 0.0f;
      // scales are fetched kSd K blocks ahead (a global load's latency is
      // longer than one K block's promotion); slot j of the unrolled loop
      // always holds the scales of K block kb + j.  Two ahead keeps the
      // promotion warps within their 224 registers (four spilled).
      constexpr int kSd = 2;
      float sa_q[kSd], sb_q[kSd];
#pragma unroll
      for (int j = 0; j < kSd; ++j) {
        sa_q[j] = (row_ok && j < kbs) ? __ldg(sa_col + (int64_t)j * args.sfa_ld) : 0.0f;
        sb_q[j] = (cols_ok && j < kbs) ? __ldg(sb_row + j) : 0.0f;
      }
      for (int kb0 = 0; kb0 < kbs && ok; kb0 += kSd) {
#pragma unroll
        for (int j = 0; j < kSd; ++j) {
          const int kb = kb0 + j;
          if (kb >= kbs) break;
          const float s = sa_q[j] * sb_q[j];
          if (kb + kSd < kbs) {
            sa_q[j] = row_ok ? __ldg(sa_col + (int64_t)(kb + kSd) * args.sfa_ld) : 0.0f;
            sb_q[j] = cols_ok ? __ldg(sb_row + kb + kSd) : 0.0f;
          }
          if (!warp_wait<kSuspendHintNs, true>(pfull(pk % NB), (pk / NB) & 1u, abort_flag, tmo, err,
                                               kSiteEpilogueTmemFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr =
              tmem_base + (pk % NB) * BN + colh * HC + ((uint32_t)(quarter * 32) << 16);
          // 128 columns as four 32-column loads through two register sets:
          // the third and fourth loads are issued while the first two
          // chunks are being added, so the buffer goes back after two load
          // latencies and half the FMAs
          uint32_t ra[32], rb[32];
          tc_ld_32x32b_x32(taddr, ra);
          tc_ld_32x32b_x32(taddr + 32, rb);
          tc_wait_ld_regs(ra);
          tc_wait_ld_regs(rb);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = fmaf(__uint_as_float(ra[i]), s, acc[i]);
          tc_ld_32x32b_x32(taddr + 64, ra);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[32 + i] = fmaf(__uint_as_float(rb[i]), s, acc[32 + i]);
          tc_ld_32x32b_x32(taddr + 96, rb);
          tc_wait_ld_regs(ra);
          tc_wait_ld_regs(rb);
          // the partial is in registers: hand the buffer back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(pempty(pk % NB));
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[64 + i] = fmaf(__uint_as_float(ra[i]), s, acc[64 + i]);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[96 + i] = fmaf(__uint_as_float(rb[i]), s, acc[96 + i]);
          ++pk;
        }
      }
      if (!ok) break;
      // chunk ch stages into buffer ch & 1; the first chunk waits until every
      // earlier store has read its buffer (they were issued a K loop ago)
#pragma unroll
      for (int ch = 0; ch < HC / 32; ++ch) {
        const int col0 = tile.nb * BN + colh * HC + ch * 32;
        if (col0 >= args.n) continue;
        uint8_t* buf = ebuf + (ch & 1) * kEpiBuf;
        if (lane == 0) {
          if (ch == 0) bulk_wait_group_read<0>();
          else bulk_wait_group_read<1>();  // this buffer's previous store (chunk ch - 2) has read it
        }
        __syncwarp();
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = acc[ch * 32 + i];
        emit_chunk_tma(f, buf, &tm_d, args, col0, row0, row0, true, lane);
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
