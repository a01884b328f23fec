// Dense NT FP8 GEMM for decode-sized M (at most 128 rows of A), with the
// operand roles swapped: 128 rows of B (128 output columns) fill the MMA's
// 128 lanes and A's rows (the tokens) are the MMA's N side.  No MMA lane
// computes padding, the accumulator is 128 lanes x TN token columns, and a
// pipeline stage holds 16 KB of B and only TN x 128 bytes of A.
//
// Work split: the K blocks of every 128-column strip of D are divided among
// the S CTAs of a cluster (one strip per cluster, one K range per CTA, no
// tile loop).  When every CTA of the cluster has its partial sum, each sends
// the other CTAs' slices of it (TN / S token columns each) through
// distributed shared memory, into the pipeline buffers they no longer use;
// each then adds the S partials of its own slice in rank order (the same
// result whatever the timing), adds C and stores BF16.
//
// Memory-bound by design: B is read once, A (at most 128 x K bytes) once per
// strip, mostly from L2.  Launched with programmatic dependent launch, a CTA
// asks for its range of B to be brought into L2 before it waits for the
// preceding kernel; L2 is coherent, so the prefetch is safe even for data
// that kernel writes.
//
// The operation and its scaling are those of the pages' dense GEMM
// ("DeepGEMM" on pt.news.hada.io, section "Interface GEMM e restrições de
// layout": D = C + A @ B.T with 1 x 128 scales for A and 128 x 128 for B).
#include <atomic>

#include "dg_device.cuh"

namespace dg {
namespace {

constexpr int kDecThreads = 192;  // warp 0: TMA; warp 1: TMEM, scales, MMA; warps 2-5: epilogue
constexpr int kDecMaxPacks = 8;   // scale words (4 K blocks each) a CTA loads: K ranges of <= 29 blocks

constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }

constexpr int kDecSmemBudget = 227 * 1024;  // dynamic shared memory of one CTA (one per SM)

template <int TN, int S>
struct DecLayout {
  static_assert(TN == 32 || TN == 64 || TN == 128, "token tile");
  static_assert(S == 1 || S == 2 || S == 4 || S == 8, "cluster size");
  static constexpr int kBTile = 128 * kBlockK;  // 128 rows of B x 128 K, 128-byte swizzle
  static constexpr int kATile = TN * kBlockK;   // TN rows of A x 128 K
  static constexpr int kStage = kBTile + kATile;
  static constexpr int kW = TN / S;             // token columns each CTA adds up and stores
  static_assert(kW % 4 == 0, "slices are sent 4 columns (16 bytes) at a time");
  // received partials, [sender slot][lane quarter][kW / 4][32 lanes][4 floats]
  static constexpr int kRecv = (S - 1) * 4 * kW * 32 * 4;
  // scale words as loaded, [pack][128] for B and [pack][TN] for A, then
  // rearranged into the 512-byte sources of tcgen05.cp: in place where a
  // pack's words take 512 bytes, else (A with TN < 128) in a region of their own
  static constexpr int kSfB = kDecMaxPacks * 512;
  static constexpr int kSfA = align1k(kDecMaxPacks * TN * 4);
  static constexpr int kCpA = TN == 128 ? 0 : kDecMaxPacks * 512;
  static constexpr int kFixed = align1k(kRecv) + kSfB + kSfA + kCpA + 1024 + 1024;  // + barriers, + alignment slack
  // as many stages as fit: the CTA's whole K range is in flight at once when
  // it spans at most this many K blocks
  static constexpr int kStages = (kDecSmemBudget - kFixed) / kStage < 12 ? (kDecSmemBudget - kFixed) / kStage : 12;
  static_assert(kStages >= 2, "pipeline depth");
  static constexpr int kOffRecv = kStages * kStage;
  static constexpr int kOffSfB = kOffRecv + align1k(kRecv);
  static constexpr int kOffSfA = kOffSfB + kSfB;
  static constexpr int kOffCpA = TN == 128 ? kOffSfA : kOffSfA + kSfA;
  static constexpr int kOffBar = kOffCpA + (TN == 128 ? kSfA : kCpA);
  static constexpr int kNumBars = 2 * kStages + 4;  // full, empty, scales, accumulator, received, TMEM read
  static constexpr int kOffCtl = kOffBar + 8 * kNumBars;
  static constexpr int kSmem = kOffCtl + 16 + 1024;  // + slack: the window is aligned to 1024 in the kernel
  static_assert(kSmem <= kDecSmemBudget, "shared memory");
  // accumulator TN columns, then 8 scale columns per pack (4 for B's rows, 4 for A's)
  static constexpr uint32_t kTmemCols = TN + 8 * kDecMaxPacks <= 128 ? 128u : 256u;
};

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 bytes into the shared memory of a CTA of the cluster, counted (16 bytes
// of complete_tx) on that CTA's mbarrier `bar`; both are cluster addresses.
// Asynchronous: no fence or remote arrive follows it, the receiver's
// mbarrier phase completes when all the bytes it expects have landed.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
               : "memory");
}

// Brings a box of a tiled tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// W consecutive TMEM columns of the warp's 32 lanes into registers (W = 4, 8,
// 16 or 32); thread t receives lane (quarter base + t).
template <int W>
__device__ __forceinline__ void tc_ld_cols(uint32_t taddr, uint32_t (&r)[W]) {
  if constexpr (W == 32) {
    tc_ld_32x32b_x32(taddr, r);
  } else if constexpr (W == 16) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  } else if constexpr (W == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  } else {
    static_assert(W == 4, "TMEM load width");
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
  }
}

// Waits for this thread's TMEM loads and ties the W registers to the wait.
template <int W>
__device__ __forceinline__ void tc_wait_cols(uint32_t (&r)[W]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < W; ++i) asm volatile("" : "+r"(r[i]));
}

// Lane 0 waits (bounded) and the warp learns the outcome.
__device__ __forceinline__ bool dec_warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint64_t tmo, unsigned long long* err, uint32_t site,
                                              bool cluster_scope = false) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0)
    ok = (cluster_scope ? wait_bounded_cluster(bar, parity, abort_flag, tmo, err, site)
                        : wait_bounded(bar, parity, abort_flag, tmo, err, site))
             ? 1
             : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// Waits for a phase ignoring the abort flag (in-flight work landing before
// exit), bounded in time.
__device__ __noinline__ void dec_drain(uint32_t bar, uint32_t parity, uint64_t tmo,
                                       unsigned long long* err, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0 && (global_timer_ns() - t0 > tmo || it >= (1u << 30))) {
      record_error(err, DG_ERR_DEVICE_TIMEOUT, site);
      return;
    }
  }
}

template <int TN, int S>
__global__ void __launch_bounds__(kDecThreads, 1)
    fp8_gemm_decode_kernel(const __grid_constant__ CUtensorMap tm_a,
                           const __grid_constant__ CUtensorMap tm_b,
                           const __grid_constant__ CUtensorMap tm_sfa,
                           const __grid_constant__ CUtensorMap tm_sfb, const DecodeArgs args) {
  using L = DecLayout<TN, S>;
  constexpr int STAGES = L::kStages;
  constexpr int W = L::kW;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  const uint32_t sf_full = smem_u32(bars + 2 * STAGES);
  const uint32_t acc_full = smem_u32(bars + 2 * STAGES + 1);
  const uint32_t recv_full = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t tmem_read = smem_u32(bars + 2 * STAGES + 3);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffCtl);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffCtl + 4);
  unsigned long long* const err = args.err;
  const uint64_t tmo = args.timeout_ns;

  // this CTA's strip of 128 output columns and its K blocks [kb0, kb1)
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  const int n0 = (int)(blockIdx.x / S) * 128;
  const int kb0 = (int)(((int64_t)args.k_blocks * rank) / S);
  const int kb1 = (int)(((int64_t)args.k_blocks * (rank + 1)) / S);
  const int nkb = kb1 - kb0;  // >= 1: the host keeps S <= K blocks
  const int kp0 = kb0 >> 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(sf_full, 1);
    mbar_init(acc_full, 1);
    mbar_init(recv_full, 1);
    mbar_init(tmem_read, 4);
    // the partials the other CTAs send land here: one arrival (this one) and
    // their bytes (S = 1: nothing is exchanged, the phase completes now)
    mbar_arrive_expect_tx(recv_full, (uint32_t)L::kRecv);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_sfa);
    tma_prefetch_desc(&tm_sfb);
    // B is not written by the preceding kernel of a GEMM chain; either way
    // an L2 prefetch cannot return stale data
    if (args.pdl)
      for (int kb = kb0; kb < kb1; ++kb) tma_prefetch_l2_2d(&tm_b, kb * kBlockK, n0);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  // from here on every thread may read what the preceding kernel wrote
  griddep_wait();
  __syncthreads();
  // Cluster barrier 1: every CTA's mbarriers exist before another CTA
  // writes into its memory (waited for just before the first such write).
  // Cluster barrier 2: a thread arrives once it writes no other CTA's memory
  // any more; every thread waits for it before the CTA exits, so no CTA
  // exits while another may still write into it.
  if constexpr (S > 1) cluster_arrive_release();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();
  int issued = 0;  // stages the producer has armed (warp 0, lane 0)

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // scale words of the K range: B's 128 rows and A's TN rows, 8 packs
      // from kp0 (packs past the end of K read as zero and are not used)
      mbar_arrive_expect_tx(sf_full, (uint32_t)(kDecMaxPacks * (128 + TN) * 4));
      DG_CHECK(err, (n0 & 3) == 0 && n0 < args.n && kp0 >= 0 && kp0 < (args.k_blocks + 3) / 4,
               kSiteCheckScale);
      tma_load_2d(smem_u32(smem + L::kOffSfB), &tm_sfb, sf_full, n0, kp0);
      tma_load_2d(smem_u32(smem + L::kOffSfA), &tm_sfa, sf_full, 0, kp0);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        // a wait that gives up leaves the abort flag raised (drained at teardown)
        if (i >= STAGES && !wait_bounded(empty(s), (uint32_t)((i / STAGES) - 1) & 1u, abort_flag, tmo, err,
                                         kSiteProducerEmpty))
          break;
        const uint32_t st = smem_u32(smem + s * L::kStage);
        const int kx = (kb0 + i) * kBlockK;
        DG_CHECK(err, kb0 + i < args.k_blocks && (kx & 15) == 0, kSiteCheckLoadB);
        mbar_arrive_expect_tx(full(s), (uint32_t)L::kStage);
        issued = i + 1;
        // test hook (dg_debug_set_drop_load): CTA 0 arms this stage and
        // never fills it, so the bounded waits must end the launch
        if (args.debug_drop_load && blockIdx.x == 0 && i + 1 == args.debug_drop_load) continue;
        tma_load_2d(st, &tm_b, full(s), kx, n0);
        tma_load_2d(st + L::kBTile, &tm_a, full(s), kx, 0);
      }
    }
    __syncwarp();
    if constexpr (S > 1) {
      cluster_wait_acquire();
      cluster_arrive_release();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ scales + MMA
    bool ok = dec_warp_wait(sf_full, 0, abort_flag, tmo, err, kSiteScaleFull);
    if (ok) {
      // scale words -> the 32 x 16-byte chunks of tcgen05.cp (lane l: the
      // words of rows l, 32 + l, 64 + l, 96 + l); A's rows past TN are 0.
      // Every lane reads a pack's words before any lane writes its chunk.
      const int npk = ((kb1 - 1) >> 2) - kp0 + 1;
      uint32_t* const rb = reinterpret_cast<uint32_t*>(smem + L::kOffSfB);
      const uint32_t* const ra = reinterpret_cast<const uint32_t*>(smem + L::kOffSfA);
      for (int p = 0; p < npk; ++p) {
        const uint4 wb = make_uint4(rb[p * 128 + lane], rb[p * 128 + 32 + lane], rb[p * 128 + 64 + lane],
                                    rb[p * 128 + 96 + lane]);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = 32 * j + lane < TN ? ra[p * TN + 32 * j + lane] : 0u;
        __syncwarp();
        *reinterpret_cast<uint4*>(smem + L::kOffSfB + p * 512 + lane * 16) = wb;
        *reinterpret_cast<uint4*>(smem + L::kOffCpA + p * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const uint32_t sf0 = tmem_base + (uint32_t)TN;
        DG_CHECK(err, args.debug_plant_check == 0 && npk >= 1 && npk <= kDecMaxPacks &&
                          (uint32_t)TN + 8u * (uint32_t)npk <= L::kTmemCols,
                 kSiteCheckTmem);
        for (int p = 0; p < npk; ++p) {
          tc_cp_32x128b_warpx4(sf0 + 8 * p, smem_desc_sf_chunk(smem_u32(smem + L::kOffSfB + p * 512)));
          tc_cp_32x128b_warpx4(sf0 + 8 * p + 4, smem_desc_sf_chunk(smem_u32(smem + L::kOffCpA + p * 512)));
        }
        constexpr uint32_t idesc0 = idesc_mxf8_e4m3(kBlockM, TN, 0, 0);
        for (int i = 0; i < nkb; ++i) {
          const int s = i % STAGES;
          if (!wait_bounded(full(s), (uint32_t)(i / STAGES) & 1u, abort_flag, tmo, err, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int kb = kb0 + i;
          const uint32_t sel = (uint32_t)(kb & 3);
          const uint32_t sft = sf0 + 8u * (uint32_t)((kb >> 2) - kp0);
          const uint32_t st = smem_u32(smem + s * L::kStage);
          const uint64_t bw = smem_desc_kmajor_sw128(st);              // B's rows: the MMA's A side
          const uint64_t at = smem_desc_kmajor_sw128(st + L::kBTile);  // A's rows: the MMA's B side
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_mxf8(tmem_base, bw + 2u * j, at + 2u * j, idesc0 | (sel << 4) | (sel << 29), sft, sft + 4,
                        (i != 0 || j != 0) ? 1u : 0u);
          tc_commit(empty(s));
        }
        // every MMA (and scale copy) completes before TMEM can be freed
        tc_commit(acc_full);
        dec_drain(acc_full, 0, tmo, err, kSiteDrain);
      }
      __syncwarp();
    }
    // TMEM goes back as soon as the epilogue has read it
    if (lane == 0) dec_drain(tmem_read, 0, tmo, err, kSiteDrain);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
    if constexpr (S > 1) {
      cluster_wait_acquire();
      cluster_arrive_release();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                     // TMEM lane quarter of this warp
    const int col = n0 + q * 32 + lane;         // output column of this lane
    const bool col_ok = col < args.n;
    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
    bool ok = dec_warp_wait(acc_full, 0, abort_flag, tmo, err, kSiteEpilogueTmemFull);
    tc_fence_after();
    // the warp's 32 lanes x TN accumulator columns, loaded at once
    uint32_t v[TN];
    if (ok) {
#pragma unroll
      for (int c = 0; c < TN; c += 32) tc_ld_32x32b_x32(taddr + (uint32_t)c, *reinterpret_cast<uint32_t(*)[32]>(&v[c]));
      tc_wait_cols<TN>(v);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_read);
    // this CTA's slice (token columns [rank * W, rank * W + W))
    float f[W];
#pragma unroll
    for (int r = 0; r < S; ++r)
      if (r == (int)rank) {
#pragma unroll
        for (int j = 0; j < W; ++j) f[j] = __uint_as_float(v[r * W + j]);
      }
    if constexpr (S > 1) {
      cluster_wait_acquire();
      // the other CTAs' slices of this partial, 16 bytes per lane at a time,
      // counted on their mbarriers
      if (ok) {
#pragma unroll
        for (int o = 0; o < S; ++o) {
          if (o == (int)rank) continue;
          const int slot = (int)rank < o ? (int)rank : (int)rank - 1;
          const uint32_t dst0 = mapa_shared(
              smem_u32(smem + L::kOffRecv) + (uint32_t)((((slot * 4 + q) * (W / 4)) * 32 + lane) * 16), (uint32_t)o);
          const uint32_t rbar = mapa_shared(recv_full, (uint32_t)o);
#pragma unroll
          for (int j = 0; j < W / 4; ++j)
            st_async_v4(dst0 + (uint32_t)(j * 512), v[o * W + 4 * j], v[o * W + 4 * j + 1], v[o * W + 4 * j + 2],
                        v[o * W + 4 * j + 3], rbar);
        }
      }
      cluster_arrive_release();  // barrier 2: no more writes to other CTAs
      if (ok) ok = dec_warp_wait(recv_full, 0, abort_flag, tmo, err, kSiteSplitFull, true);
      if (ok) {
        // the S partials of the slice in rank order
        const uint8_t* recv = smem + L::kOffRecv;
        float g[W];
#pragma unroll
        for (int s = 0; s < S; ++s) {
          if (s == (int)rank) {
#pragma unroll
            for (int j = 0; j < W; ++j) g[j] = s == 0 ? f[j] : g[j] + f[j];
          } else {
            const int slot = s < (int)rank ? s : s - 1;
            const uint8_t* src = recv + (((slot * 4 + q) * (W / 4)) * 32 + lane) * 16;
#pragma unroll
            for (int j = 0; j < W / 4; ++j) {
              const float4 w = *reinterpret_cast<const float4*>(src + j * 512);
              g[4 * j] = s == 0 ? w.x : g[4 * j] + w.x;
              g[4 * j + 1] = s == 0 ? w.y : g[4 * j + 1] + w.y;
              g[4 * j + 2] = s == 0 ? w.z : g[4 * j + 2] + w.z;
              g[4 * j + 3] = s == 0 ? w.w : g[4 * j + 3] + w.w;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < W; ++j) f[j] = g[j];
      }
    }
    if (ok && col_ok) {
      // + C, rounded to BF16
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int t = (int)rank * W + j;
        if (t < args.m) {
          float x = f[j];
          if (args.c) x += __bfloat162float(args.c[(int64_t)t * args.ldc + col]);
          DG_CHECK(err, (int64_t)t * args.ldd + col < (int64_t)args.m * args.ldd, kSiteCheckStore);
          args.d[(int64_t)t * args.ldd + col] = __float2bfloat16_rn(x);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // After a wait gave up (the abort flag), the loads still in flight land
  // before the CTA may exit.
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    dec_drain(sf_full, 0, tmo, err, kSiteProducerDrain);
    for (int i = issued - STAGES < 0 ? 0 : issued - STAGES; i < issued; ++i)
      dec_drain(full(i % STAGES), (uint32_t)(i / STAGES) & 1u, tmo, err, kSiteProducerDrain);
  }
  if constexpr (S > 1) {
    cluster_wait_acquire();
    // Normally this CTA has received every partial sent to it (its recv wait
    // completed).  After an abort it may not have: the other CTAs issued
    // their st.async before arriving at the barrier just passed, but nothing
    // orders their landing before it.  Wait for them, briefly: a peer that
    // sent lands within microseconds, one that did not send never will.
    if (threadIdx.x == 0 && *abort_flag)
      dec_drain(recv_full, 0, tmo < 1000000u ? tmo : 1000000u, err, kSiteSplitFull);
  }
}

template <int TN, int S>
cudaError_t decode_launch_impl(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                               const CUtensorMap& sfb, const DecodeArgs& args, int grid,
                               cudaStream_t stream) {
  using L = DecLayout<TN, S>;
  auto kern = fp8_gemm_decode_kernel<TN, S>;
  static std::atomic<bool> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    done[dev].store(true, std::memory_order_release);
  }
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (S > 1) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = S;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  if (args.pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  return cudaLaunchKernelEx(&cfg, kern, a, b, sfa, sfb, args);
}

template <int TN>
cudaError_t decode_launch_tn(int split, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sfa,
                             const CUtensorMap& sfb, const DecodeArgs& args, int grid, cudaStream_t stream) {
  switch (split) {
    case 1: return decode_launch_impl<TN, 1>(a, b, sfa, sfb, args, grid, stream);
    case 2: return decode_launch_impl<TN, 2>(a, b, sfa, sfb, args, grid, stream);
    case 4: return decode_launch_impl<TN, 4>(a, b, sfa, sfb, args, grid, stream);
    case 8: return decode_launch_impl<TN, 8>(a, b, sfa, sfb, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int gemm_decode_max_packs() { return kDecMaxPacks; }

cudaError_t gemm_decode_launch(int tn, int split, const CUtensorMap& a, const CUtensorMap& b,
                               const CUtensorMap& sfa, const CUtensorMap& sfb, DecodeArgs args,
                               cudaStream_t stream) {
  unsigned long long* err = nullptr;
  cudaError_t e = error_word_address(&err);
  if (e != cudaSuccess) return e;
  args.err = err;
  const int grid = args.n_strips * split;
  if (grid <= 0) return cudaErrorInvalidValue;
  switch (tn) {
    case 32: return decode_launch_tn<32>(split, a, b, sfa, sfb, args, grid, stream);
    case 64: return decode_launch_tn<64>(split, a, b, sfa, sfb, args, grid, stream);
    case 128: return decode_launch_tn<128>(split, a, b, sfa, sfb, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg
