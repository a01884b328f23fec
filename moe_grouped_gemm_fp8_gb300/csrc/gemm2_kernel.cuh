// FP8 GEMM with fine-grained scaling on a CTA pair (tcgen05 cta_group::2):
// output tiles of 256 rows x BN columns, each CTA of a 2-CTA cluster holding
// 128 rows of A, half of the B tile and its 128 rows of the accumulator.
//
// Same operation, layouts and roles as gemm_kernel.cuh (dense and masked
// forms); what changes on the pair:
//   - each CTA's producer loads its own A rows and its half of B (BN / 2
//     rows); both CTAs' copies complete on the leader's stage barrier, which
//     alone expects the bytes of the two;
//   - the leader's MMA lane issues 256 x BN x 32 block-scaled MMAs reading A
//     and B from both CTAs' shared memory, TMEM copies of both CTAs' scale
//     chunks, and commits that arrive on the barrier of both CTAs;
//   - every CTA's TMEM holds the A scales of its own 128 rows and the B scales
//     of all BN rows, so each scale warp loads its A rows and the full B tile
//     of scale words, and reports to the leader;
//   - each epilogue drains its own CTA's TMEM and reports to the leader.
// Per SM, every 128-wide K block moves 16 KB of A and BN x 64 bytes of B
// instead of BN x 128: half the B traffic of a single-CTA tile of the same
// width, and one MMA instruction covers twice the work.
#pragma once

#include "gemm_kernel.cuh"

namespace dg {

template <int BN>
struct Gemm2Layout {
  static constexpr int kHalfN = BN / 2;
  static constexpr int kSfbChunks = (BN + 127) / 128;  // B scales of all BN rows
  static constexpr int kBytesA = kBlockM * kBlockK;
  static constexpr int kBytesB = kHalfN * kBlockK;
  static constexpr int kOffB = kBytesA;
  static constexpr int kStageBytes = (kBytesA + kBytesB + 1023) / 1024 * 1024;
  static constexpr int kRawA = 0;
  static constexpr int kRawB = 512;
  static constexpr int kCpA = kRawB + kSfbChunks * 512;
  static constexpr int kCpB = kCpA + 512;
  static constexpr int kSfBufBytes = kCpB + kSfbChunks * 512;
  static constexpr uint32_t kTxPair = 2u * (kBytesA + kBytesB);  // both CTAs, on the leader
  static constexpr uint32_t kTxSF = 128 * 4 + BN * 4;
  static constexpr int kSfCols = 4 + 4 * kSfbChunks;
};

static constexpr size_t gemm2_ctrl_bytes(int stages, int mode) {
  return (size_t)8 * (2 * stages + 3 * kSfSlots + 6) + 16 +
         (mode == kMasked ? (size_t)4 * (2 * kMaxMaskedGroups + 1) : 0);
}

template <int BN, int STAGES>
struct Gemm2Plan {
  using L = Gemm2Layout<BN>;
  static constexpr int kNumAcc = (2 * BN + kSfSlots * L::kSfCols <= 512) ? 2 : 1;
  static constexpr int kSfBase = kNumAcc * BN;
  static_assert(kSfBase + kSfSlots * L::kSfCols <= 512, "TMEM over-subscribed");
  static constexpr size_t smem_bytes(int mode) {
    return (size_t)STAGES * L::kStageBytes + (size_t)kSfSlots * L::kSfBufBytes + kEpiBytes +
           1024 + gemm2_ctrl_bytes(STAGES, mode);
  }
};

// Pair tiles: (group, 256-row block, N block).  Dense tiles are rastered in
// bands of `band` pair blocks (pair block fastest); masked tiles group by
// group from a prefix table.
template <int MODE>
struct PairScheduler {
  const GemmArgs* args;
  const int* tile_start;
  const int* group_valid;
  int total;
  int cursor;
  int p_blocks;  // dense: ceil(m / 256)
  int first, stride;  // this cluster's first tile and the stride of its tile walk

  __device__ void k_range(const Tile&, int& kb0, int& kb1) const {
    kb0 = 0;
    kb1 = args->k_blocks;
  }

  // The it-th tile of this cluster's walk with its K blocks (-1: no more).
  __device__ int item(int it, Tile& tile, int& kb0, int& kb1) {
    const int t = first + it * stride;
    if (t >= total) return -1;
    tile.kind = kItemFull;
    tile.sk = -1;
    if (!get(t, tile)) return 0;
    k_range(tile, kb0, kb1);
    return 1;
  }

  __device__ bool get(int t, Tile& tile) {
    if (MODE == kMasked) {
      while (t >= tile_start[cursor + 1]) ++cursor;
      const int local = t - tile_start[cursor];
      const int pbs = (group_valid[cursor] + 2 * kBlockM - 1) / (2 * kBlockM);
      tile.g = cursor;
      tile.mb = local % pbs;
      tile.nb = local / pbs;
      return true;
    }
    const int per_band = args->band * args->n_blocks;
    const int b = t / per_band;
    const int rem = t - b * per_band;
    const int rows = min(args->band, p_blocks - b * args->band);
    tile.nb = rem / rows;
    tile.mb = b * args->band + rem % rows;
    tile.g = 0;
    return true;
  }
};

template <int BN, int STAGES, int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a,
                         const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_sfa,
                         const __grid_constant__ CUtensorMap tm_sfb,
                         const __grid_constant__ CUtensorMap tm_d, const GemmArgs args) {
  static_assert(MODE == kDense || MODE == kMasked, "only dense and masked tiles are paired");
  using L = Gemm2Layout<BN>;
  using P = Gemm2Plan<BN, STAGES>;
  constexpr int NUM_ACC = P::kNumAcc;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  uint8_t* sfbuf = smem + STAGES * L::kStageBytes;
  uint8_t* epi_smem = sfbuf + kSfSlots * L::kSfBufBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster_id = (int)(blockIdx.x >> 1);
  const int num_clusters = (int)(gridDim.x >> 1);

  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_smem + kEpiBytes);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto sffull = [&](int p) { return smem_u32(bars + 2 * STAGES + p); };
  auto sfready = [&](int p) { return smem_u32(bars + 2 * STAGES + kSfSlots + p); };
  auto sfempty = [&](int p) { return smem_u32(bars + 2 * STAGES + 2 * kSfSlots + p); };
  constexpr int kB0 = 2 * STAGES + 3 * kSfSlots;
  auto tfull = [&](int a) { return smem_u32(bars + kB0 + a); };
  auto tempty = [&](int a) { return smem_u32(bars + kB0 + 2 + a); };
  const uint32_t drain = smem_u32(bars + kB0 + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kB0 + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
  int* group_valid = tile_start + (kMaxMaskedGroups + 1);
  unsigned long long* const err = args.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int p = 0; p < kSfSlots; ++p) {
      mbar_init(sffull(p), 1);
      mbar_init(sfready(p), 2);  // both CTAs' scale warps
      mbar_init(sfempty(p), 1);
    }
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 8);  // both CTAs' epilogue warps
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_sfa);
    tma_prefetch_desc(&tm_sfb);
    tma_prefetch_desc(&tm_d);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  griddep_wait();  // see fp8_gemm_kernel
  if (MODE == kMasked && warp == 2) {
    for (int g = lane; g < args.num_groups; g += 32) {
      const int v = __ldg(args.masked_m + g);
      const int c = v < 0 ? 0 : (v > args.m ? args.m : v);
      if (c != v && leader) record_error(err, DG_ERR_DEVICE_BAD_INDEX, kSiteMaskedCount);
      group_valid[g] = c;
    }
    __syncwarp();
    if (lane == 0) {
      int acc = 0;
      for (int g = 0; g < args.num_groups; ++g) {
        tile_start[g] = acc;
        acc += (group_valid[g] + 2 * kBlockM - 1) / (2 * kBlockM) * args.n_blocks;
      }
      tile_start[args.num_groups] = acc;
    }
  }
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();

  PairScheduler<MODE> sched;
  sched.args = &args;
  sched.tile_start = tile_start;
  sched.group_valid = group_valid;
  sched.cursor = 0;
  sched.p_blocks = (args.m + 2 * kBlockM - 1) / (2 * kBlockM);
  sched.total = MODE == kMasked ? tile_start[args.num_groups] : sched.p_blocks * args.n_blocks;
  sched.first = cluster_id;
  sched.stride = num_clusters;
  const uint64_t tmo = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int t = cluster_id; t < sched.total && ok; t += num_clusters) {
        Tile tile;
        if (!sched.get(t, tile)) continue;
        const int my = (2 * tile.mb + (int)rank) * kBlockM;
        const int ny = tile.nb * BN + (int)rank * L::kHalfN;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!wait_one(empty(stage), phase ^ 1u, abort_flag, tmo, err, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t sb = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t fb = mapa_shared(full(stage), 0);  // the leader's barrier
          if (leader) mbar_arrive_expect_tx(full(stage), L::kTxPair);
          const int kx = kb * kBlockK;
          if (MODE == kMasked) tma_load_3d_pair(sb, &tm_a, fb, kx, my, tile.g);
          else tma_load_2d_pair(sb, &tm_a, fb, kx, my);
          tma_load_3d_pair(sb + L::kOffB, &tm_b, fb, kx, ny, tile.g);
          if (leader) {
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
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
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc0 = idesc_mxf8_e4m3(2 * kBlockM, BN, 0, 0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pack = 0;
      uint32_t sf_tmem = tmem_base + (uint32_t)P::kSfBase;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = cluster_id; t < sched.total && ok; t += num_clusters) {
        Tile tile;
        if (!sched.get(t, tile)) continue;
        if (!(mbar_try_wait_cluster(tempty(acc), acc_phase ^ 1u) ||
              wait_bounded_cluster(tempty(acc), acc_phase ^ 1u, abort_flag, tmo, err,
                                   kSiteMmaTmemEmpty))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!wait_one(full(stage), phase, abort_flag, tmo, err, kSiteMmaFull)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * L::kStageBytes;
          const int slot = (int)(pack % kSfSlots);
          if ((kb & 3) == 0) {
            const uint32_t par = (pack / kSfSlots) & 1u;
            if (!(mbar_try_wait_cluster(sfready(slot), par) ||
                  wait_bounded_cluster(sfready(slot), par, abort_flag, tmo, err,
                                       kSiteMmaScaleReady))) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint8_t* buf = sfbuf + slot * L::kSfBufBytes;
            sf_tmem = tmem_base + (uint32_t)(P::kSfBase + slot * L::kSfCols);
            tc_cp_32x128b_warpx4_pair(sf_tmem, smem_desc_sf_chunk(smem_u32(buf + L::kCpA)));
#pragma unroll
            for (int c = 0; c < L::kSfbChunks; ++c)
              tc_cp_32x128b_warpx4_pair(sf_tmem + 4 + 4 * c,
                                        smem_desc_sf_chunk(smem_u32(buf + L::kCpB + c * 512)));
          }
          const uint32_t sel = (uint32_t)(kb & 3);
          const uint32_t idesc = idesc0 | (sel << 4) | (sel << 29);
          const uint64_t adesc = smem_desc_kmajor_sw128(smem_u32(st));
          const uint64_t bdesc = smem_desc_kmajor_sw128(smem_u32(st + L::kOffB));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_mxf8_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sf_tmem, sf_tmem + 4,
                             (kb | j) != 0 ? 1u : 0u);
          tc_commit_pair(empty(stage));
          if ((kb & 3) == 3 || kb == args.k_blocks - 1) {
            tc_commit_pair(sfempty(slot));
            ++pack;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(tfull(acc));
        if (++acc == NUM_ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit_pair(drain);  // arrives in both CTAs once every MMA and copy has completed
      wait_drain(drain, 0, tmo, err, kSiteDrain);
    } else if (lane == 0) {
      // the peer waits for the leader's last MMA before its TMEM can be freed
      wait_drain(drain, 0, tmo, err, kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale warp (both CTAs)
    PackCursor<PairScheduler<MODE>> ld, lay;
    ld.init(sched);
    lay.init(sched);
    uint32_t n_loaded = 0, n_laid = 0;
    bool ok = true;
    while (!lay.done && ok) {
      while (!ld.done && n_loaded < n_laid + kSfLookahead) {
        const int slot = (int)(n_loaded % kSfSlots);
        int go = 1;
        if (lane == 0) {
          go = wait_one(sfempty(slot), ((n_loaded / kSfSlots) & 1u) ^ 1u, abort_flag, tmo, err,
                        kSiteScaleEmpty) ? 1 : 0;
          if (go) {
            const uint32_t buf = smem_u32(sfbuf + slot * L::kSfBufBytes);
            const uint32_t bar = sffull(slot);
            const int my = (2 * ld.tile.mb + (int)rank) * kBlockM, kp = ld.kp;
            mbar_arrive_expect_tx(bar, L::kTxSF);
            if (MODE == kMasked) tma_load_3d(buf + L::kRawA, &tm_sfa, bar, my, kp, ld.tile.g);
            else tma_load_2d(buf + L::kRawA, &tm_sfa, bar, my, kp);
            tma_load_3d(buf + L::kRawB, &tm_sfb, bar, ld.tile.nb * BN, kp, ld.tile.g);
          }
        }
        go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) {
          ok = false;
          break;
        }
        ++n_loaded;
        ld.advance();
      }
      if (!ok) break;
      const int slot = (int)(n_laid % kSfSlots);
      if (!warp_wait(sffull(slot), (n_laid / kSfSlots) & 1u, abort_flag, tmo, err, kSiteScaleFull)) {
        ok = false;
        break;
      }
      uint8_t* buf = sfbuf + slot * L::kSfBufBytes;
      {
        const uint32_t* raw = reinterpret_cast<const uint32_t*>(buf + L::kRawA);
        const uint4 v = make_uint4(raw[lane], raw[32 + lane], raw[64 + lane], raw[96 + lane]);
        *reinterpret_cast<uint4*>(buf + L::kCpA + lane * 16) = v;
      }
#pragma unroll
      for (int c = 0; c < L::kSfbChunks; ++c) {
        const uint32_t* raw = reinterpret_cast<const uint32_t*>(buf + L::kRawB + c * 512);
        const uint4 v = make_uint4(raw[lane], raw[32 + lane], raw[64 + lane], raw[96 + lane]);
        *reinterpret_cast<uint4*>(buf + L::kCpB + c * 512 + lane * 16) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(sfready(slot), 0));
      ++n_laid;
      lay.advance();
    }
    if (lane == 0)
      for (uint32_t q = n_laid; q < n_loaded; ++q)
        wait_drain(sffull((int)(q % kSfSlots)), (q / kSfSlots) & 1u, tmo, err, kSiteProducerDrain);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;
    uint8_t* ebuf = epi_smem + (warp - 3) * 2 * kEpiBuf;
    const uint32_t my_row_off = (uint32_t)lane * 64u;
    const uint32_t my_swz = ((uint32_t)lane >> 1) & 3u;
    uint32_t nchunk = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cluster_id; t < sched.total; t += num_clusters) {
      Tile tile;
      if (!sched.get(t, tile)) continue;
      if (!warp_wait(tfull(acc), acc_phase, abort_flag, tmo, err, kSiteEpilogueTmemFull)) break;
      tc_fence_after();
      const int row0 = (2 * tile.mb + (int)rank) * kBlockM + quarter * 32;
      const int row = row0 + lane;
      bool row_ok;
      int64_t out_row0;
      if (MODE == kDense) {
        row_ok = row < args.m;
        out_row0 = row0;
      } else {
        row_ok = row < group_valid[tile.g];
        out_row0 = (int64_t)tile.g * args.m + row0;
      }
      const bool use_tma = (MODE == kDense) ? true : (__all_sync(0xffffffffu, row_ok) != 0);
      __nv_bfloat16* drow = args.d + (out_row0 + lane) * args.ldd;
      const __nv_bfloat16* crow = args.c ? args.c + (out_row0 + lane) * args.ldc : nullptr;
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
      constexpr int NCH = BN / 32;
      uint32_t ra[32], rb[32];
      tc_ld_32x32b_x32(taddr, ra);
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t(&cur)[32] = (ch & 1) ? rb : ra;
        uint32_t(&nxt)[32] = (ch & 1) ? ra : rb;
        tc_wait_ld_regs(cur);
        if (ch + 1 < NCH) {
          tc_ld_32x32b_x32(taddr + (ch + 1) * 32, nxt);
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty(acc), 0));
        }
        const int col0 = tile.nb * BN + ch * 32;
        if (col0 >= args.n) continue;
        if (use_tma) {
          uint8_t* buf = ebuf + (nchunk & 1u) * kEpiBuf;
          const uint32_t sbuf = smem_u32(buf);
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
          float f[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(cur[i]);
          if (args.c) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = (lane >> 2) + 8 * i, pc = lane & 3;
              const int gcol = col0 + pc * 8;
              uint4 v = make_uint4(0u, 0u, 0u, 0u);
              if (gcol < args.n && (MODE != kDense || row0 + r < args.m))
                v = __ldg(reinterpret_cast<const uint4*>(args.c + (out_row0 + r) * args.ldc + gcol));
              *reinterpret_cast<uint4*>(buf + r * 64 + 16 * (pc ^ ((r >> 1) & 3))) = v;
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 cv = *reinterpret_cast<const uint4*>(buf + my_row_off + 16u * ((uint32_t)j ^ my_swz));
              const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                f[8 * j + 2 * i] += __uint_as_float(cw[i] << 16);
                f[8 * j + 2 * i + 1] += __uint_as_float(cw[i] & 0xFFFF0000u);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 o;
            o.x = pack_bf16x2(f[8 * j + 0], f[8 * j + 1]);
            o.y = pack_bf16x2(f[8 * j + 2], f[8 * j + 3]);
            o.z = pack_bf16x2(f[8 * j + 4], f[8 * j + 5]);
            o.w = pack_bf16x2(f[8 * j + 6], f[8 * j + 7]);
            *reinterpret_cast<uint4*>(buf + my_row_off + 16u * ((uint32_t)j ^ my_swz)) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tm_d, sbuf, col0, (int32_t)out_row0);
            bulk_commit_group();
          }
          ++nchunk;
        } else if (row_ok) {
          store_row_chunk(cur, drow + col0, crow ? crow + col0 : nullptr, args.n - col0);
        }
      }
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  __syncthreads();
  cluster_sync_all();  // both CTAs are done with every role
  {
    // After an abort, copies the peer issued towards this CTA's barriers may
    // still be in flight: give them time to land before the memory goes away.
    // The release/acquire barriers around this block order every thread's
    // own loads and stores, but not TMA copies: those are asynchronous, and
    // a peer's operand copy completes on the leader's stage barrier, never
    // on one of its own.  The leader drains every stage it armed, but after
    // an abort the peer may have issued a copy into a stage the leader never
    // armed (its wait ran out first), and no barrier in either CTA tracks
    // that copy.  Nothing can be waited on for it, so a fixed grace period
    // (many times a copy's latency) is the only bound; it is spent only on
    // the abort path, never in a clean launch.
    const int peer_abort = (int)ld_shared_cluster_u32(
        mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u));
    if (*abort_flag || peer_abort) {
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 200000ull) {
      }
    }
  }
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

template <int BN, int STAGES, int MODE>
static cudaError_t gemm2_launch_impl(const CUtensorMap& a, const CUtensorMap& b,
                                     const CUtensorMap& sfa, const CUtensorMap& sfb,
                                     const CUtensorMap& d, const GemmArgs& args, int clusters,
                                     cudaStream_t stream) {
  static_assert(Gemm2Plan<BN, STAGES>::smem_bytes(kMasked) <= (size_t)kSmemLimit,
                "shared memory over the per-CTA limit");
  auto kern = fp8_gemm_pair_kernel<BN, STAGES, MODE>;
  const size_t smem = Gemm2Plan<BN, STAGES>::smem_bytes(MODE);
  cudaError_t e = set_smem_once<KernelTag<BN, STAGES, MODE, 1, 2>>(kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = args.pdl ? 2 : 1;
  if (clusters <= 0) return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, kern, a, b, sfa, sfb, d, args);
}

// Largest number of co-resident 2-CTA clusters of this configuration.
template <int BN, int STAGES, int MODE>
static int gemm2_max_clusters() {
  auto kern = fp8_gemm_pair_kernel<BN, STAGES, MODE>;
  const size_t smem = Gemm2Plan<BN, STAGES>::smem_bytes(MODE);
  if (set_smem_once<KernelTag<BN, STAGES, MODE, 1, 2>>(kern, smem) != cudaSuccess) return 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace dg

// Defines the pair launch entry of one tile width (one translation unit each).
#define DG_DEFINE_GEMM2_BN(BN, STAGES)                                                       \
  namespace dg {                                                                           \
  cudaError_t gemm2_launch_bn##BN(int mode, const CUtensorMap& a, const CUtensorMap& b,    \
                                  const CUtensorMap& sfa, const CUtensorMap& sfb,          \
                                  const CUtensorMap& d, const GemmArgs& args,              \
                                  int clusters, cudaStream_t stream) {                     \
    if (mode == kDense)                                                                    \
      return gemm2_launch_impl<BN, STAGES, kDense>(a, b, sfa, sfb, d, args, clusters,      \
                                                   stream);                                \
    if (mode == kMasked)                                                                   \
      return gemm2_launch_impl<BN, STAGES, kMasked>(a, b, sfa, sfb, d, args, clusters,     \
                                                    stream);                               \
    return cudaErrorInvalidValue;                                                          \
  }                                                                                        \
  int gemm2_max_clusters_bn##BN(int mode) {                                                \
    return mode == kMasked ? gemm2_max_clusters<BN, STAGES, kMasked>()                     \
                           : gemm2_max_clusters<BN, STAGES, kDense>();                     \
  }                                                                                        \
  }
