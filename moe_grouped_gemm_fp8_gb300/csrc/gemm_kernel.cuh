// FP8 GEMM with fine-grained scaling on sm_103a: D = C + A @ B.T, dense and
// M-grouped (contiguous / masked), K-grouped, and the NN / TN / TT layouts.
// Kernel template; each tile width BN is instantiated in its own translation
// unit (gemm_bn*.cu), the split-K clusters in gemm_splitk.cu, the 256-row and
// 64-row-A-slot tiles in gemm_tall.cu.
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
// One persistent CTA per SM, 7 warps:
//   warp 0      TMA producer (one lane): A tile [BM x 128] and B tile
//               [BN x 128] (E4M3, 128-byte swizzle) per 128-wide K block into
//               an S-stage ring.
//   warp 1      MMA issuer (one lane, kept free of any other work): per K
//               block issues four 128 x BN x 32 block-scaled MMAs per 128-row
//               half of the tile (BM = 256: two halves sharing B), the
//               instruction descriptor selecting the byte of the current K
//               block in the pack's scale slot; commits the stage back to the
//               producer.  Also owns the TMEM allocation.
//   warp 2      scale warp: loads the packed scale words (one 32-bit word =
//               the UE8M0 scales of four K blocks) of A's 128 rows and B's BN
//               rows by TMA, up to three packs ahead of use, into a ring of
//               kSfSlots buffers, turns them (M-major row order) into the
//               32-row x 16-byte chunks tcgen05.cp reads (row r of a 128-row
//               group at byte 16 (r % 32) + 4 (r / 32)), copies them into the
//               slot's TMEM columns (tcgen05.cp 32x128b.warpx4) and commits
//               the slot as ready.
//   warps 3-6   epilogue: tcgen05.ld of the accumulator (one 32-lane TMEM
//               quarter each, 32 columns at a time, the next chunk loading
//               while the current one is converted), + C, round to BF16.  A
//               32 x 32 chunk is staged in shared memory (64-byte swizzle,
//               conflict-free for one row per thread; two staging chunks
//               per warp) and written by a TMA store; C arrives through
//               coalesced loads staged the same way, the quarter's whole C
//               tile issued before the accumulator is ready.
//               Quarters of grouped tiles with rows that must stay untouched
//               use row-predicated 16-byte stores instead.  TMEM is released
//               as soon as the last chunk is in registers.
// The accumulator is double-buffered in TMEM when 2 x BM/128 x BN columns
// leave room for the scales, so the epilogue of one tile overlaps the next
// tile's MMAs.  A single accumulator (128 x 256, 256-row tiles) is read into
// registers in as few steps as registers allow before any store, so the MMA
// waits only for the TMEM loads: each lane's row of C (BF16 pairs, fetched
// before the accumulator is ready) is added in place and rounded to BF16.
//
// Split-K (KSPLIT = 2 or 4, dense only, for problems with fewer output tiles
// than SMs): a cluster of KSPLIT CTAs shares each output tile, CTA r taking a
// slice of ceil(K blocks / KSPLIT) K blocks (a slice may start inside a
// scale pack; the pack is then loaded by both CTAs).  CTA r owns the r-th column
// slice (BN / KSPLIT columns) of every 32-row quarter: each epilogue warp
// writes the other slices of its FP32 partial into their owners' shared
// memory (distributed shared memory) and arrives on their barriers, then adds
// the partials of its own slice in rank order - the same order whatever the
// timing, so results are deterministic - adds C, rounds to BF16 and stores.
// All four epilogue warps of every CTA share the exchange and the stores.
// No global scratch memory is used.
//
// Multicast pairs (MC: dense 256-row tiles and K-grouped 128 x 256 tiles,
// eight epilogue warps): clusters of two CTAs walk the same tiles of B with
// adjacent row blocks of A; each CTA loads half of the B tile into both
// CTAs' stage (TMA multicast) and its MMA commit frees the stage in both, so
// the pair moves through the ring in lockstep and L2 serves B once per pair.
//
// Every mbarrier wait is bounded; on expiry the kernel records an error,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "dg_device.cuh"

namespace dg {

constexpr int kGemmThreads = 224;
// 256-row dense tiles with eight epilogue warps (two per TMEM lane quarter,
// one per 128-row half): warps 0-2 keep their roles, warp 3 idles, warps
// 4-11 drain the single accumulator.  Registers are shifted to the epilogue
// warpgroups with setmaxnreg: 128 x kRegsRoles + 256 x kRegsEpi must equal
// the 384 x 168 registers the block is launched with.
constexpr int kGemmThreadsEpi8 = 384;
constexpr int kRegsRoles = 56, kRegsEpi = 224;
static_assert(128 * kRegsRoles + 256 * kRegsEpi == kGemmThreadsEpi8 * 168, "setmaxnreg split");
constexpr int kSmemLimit = 232448;  // dynamic shared memory per CTA on sm_103

// BM: rows of A per tile, 128 or 256 (two 128-row MMAs sharing B), or 64:
// a single M block of at most 64 rows, whose A slot holds only those rows
// (the 128-row MMA then reads rows 64-127 from the B slot that follows; they
// reach only accumulator rows that are never stored), so more stages fit.
template <int BN, int BM = kBlockM>
struct GemmLayout {
  static constexpr int kMH = (BM + kBlockM - 1) / kBlockM;  // 128-row halves of the tile
  static constexpr int kSfbChunks = (BN + 127) / 128;  // 128-row chunks of B scales
  static constexpr int kBytesA = BM * kBlockK;
  static constexpr int kBytesB = BN * kBlockK;
  static constexpr int kOffB = kBytesA;
  static constexpr int kStageBytes = (kBytesA + kBytesB + 1023) / 1024 * 1024;
  // scale buffer: TMA-loaded words of A (BM) and B (BN), then the same words
  // in tcgen05.cp order
  static constexpr int kRawA = 0;
  static constexpr int kRawB = kMH * kBlockM * 4;
  static constexpr int kCpA = kRawB + kSfbChunks * 512;
  static constexpr int kCpB = kCpA + kMH * 512;
  static constexpr int kSfBufBytes = kCpB + kSfbChunks * 512;
  static constexpr uint32_t kTxAB = kBytesA + kBytesB;
  static constexpr uint32_t kTxSF = kMH * kBlockM * 4 + BN * 4;
  // TMEM columns of one scale slot: A scales of each half, then B scales
  static constexpr int kSfCols = 4 * kMH + 4 * kSfbChunks;
};

constexpr int kSfSlots = 4;      // scale buffers / TMEM scale slots
constexpr int kEpiBuf = 32 * 32 * 2;  // one 32 x 32 BF16 staging chunk
constexpr int kEpiBytes = 4 * 2 * kEpiBuf;  // 4 epilogue warps x 2 buffers
constexpr int kSfLookahead = 3;  // packs loaded ahead of the one being laid out

// Contiguous form with 256-row tiles: most 128-row block pairs per launch
// (block indices kept as 16-bit halves of one word).
constexpr int kMaxBlockPairs = kMaxTallPairs;

static constexpr size_t gemm_ctrl_bytes(int stages, int mode, int bm = kBlockM) {
  return (size_t)8 * (2 * stages + 3 * kSfSlots + 5 + 8) + 32 +
         ((mode == kMasked || mode == kKGrouped) ? (size_t)4 * (2 * kMaxMaskedGroups + 1) : 0) +
         ((mode == kContiguous && bm == 2 * kBlockM)
              ? (size_t)4 * (2 * kMaxMaskedGroups + 1) + (size_t)4 * kMaxBlockPairs
              : 0);
}

// Scale buffers and TMEM scale slots are indexed by a running count of scale
// packs modulo kSfSlots.  Each slot has three barriers whose phases advance
// once per pack - words landed (TMA), words laid out (scale warp), slot free
// (tcgen05.commit after the pack's last MMA) - and every waiter visits every
// pack in order, so no wait ever skips a phase.
template <int BN, int STAGES, int KSPLIT = 1, int BM = kBlockM>
struct GemmPlan {
  using L = GemmLayout<BN, BM>;
  // accumulators of BM x BN (kMH blocks of BN columns each)
  static constexpr int kNumAcc = (2 * L::kMH * BN + kSfSlots * L::kSfCols <= 512) ? 2 : 1;
  static constexpr int kSfBase = kNumAcc * L::kMH * BN;
  static_assert(kSfBase + kSfSlots * L::kSfCols <= 512, "TMEM over-subscribed");
  static_assert(KSPLIT == 1 || KSPLIT == 2 || KSPLIT == 4, "split-K over 1, 2 or 4 CTAs");
  // split-K: CTA r of a cluster owns columns [r, r + 1) * kSlice of every
  // quarter.  Its receive buffer holds, per quarter and per other CTA, that
  // CTA's FP32 partial of the slice: 32-column chunks of 32 rows, stored
  // lane-interleaved (16-byte group j of row l at 512 j + 16 l) so that the
  // remote stores and the owner's loads are both contiguous per warp.
  static constexpr int kSlice = BN / KSPLIT;
  static constexpr int kXSlot = 32 * kSlice * 4;
  static constexpr int kRecvBytes = KSPLIT > 1 ? 4 * (KSPLIT - 1) * kXSlot : 0;
  static constexpr size_t smem_bytes(int mode) {
    return (size_t)STAGES * L::kStageBytes + (size_t)kSfSlots * L::kSfBufBytes + kEpiBytes +
           (size_t)kRecvBytes + 1024 + gemm_ctrl_bytes(STAGES, mode, BM);
  }
};

// Stream-K work items (dense 256-row tiles): a tile whose K blocks are split
// between CTAs is finished by its owner, the CTA that holds its first K
// blocks (as its last item); the others contribute partial sums.
enum ItemKind : int { kItemFull = 0, kItemOwner = 1, kItemPart = 2 };

struct Tile {
  int g, mb, nb;
  int b0, b1;  // contiguous 256-row tiles: the two 128-row blocks (b1 < 0: none)
  int kind;    // ItemKind
  int sk;      // stream-K: index of the tile among the split tiles
};

// Maps a linear tile index to (group, M block, N block).  Dense and
// contiguous tiles are rastered in bands of `band` M blocks: inside a band the
// M block varies fastest, so a wave of CTAs shares a few B column blocks and
// one band of A.  Masked tiles are enumerated group by group (M block
// fastest) from a prefix table built at kernel start.  K-grouped tiles are
// enumerated expert by expert, each expert's M x N tiles rastered like dense
// ones.  k_range gives the K blocks a tile accumulates: this CTA's split-K
// slice, or the expert's own K blocks for the K-grouped form.
template <int MODE, int BM = kBlockM, bool SK = false>
struct Scheduler {
  const GemmArgs* args;
  const int* tile_start;   // masked: [G + 1] first tile; K-grouped: [G + 1] first K block;
                           // contiguous 256-row tiles: [G + 1] first block pair
  const int* group_valid;  // masked: [G]
  const uint32_t* pairs;   // contiguous 256-row tiles: 128-row blocks of each pair
  int total;
  int cursor;              // masked: current group (tile indices only increase)
  int kb_lo, kb_hi;        // K blocks of every tile (not K-grouped)
  int first, stride;       // this CTA's first tile and the stride of its tile walk
  int pair_rank = -1;      // dense multicast pairs: this CTA's rank (tiles are pairs of M blocks), else -1
  const uint32_t* sk_ctl;  // stream-K kernels: this CTA's units [sk_ctl[0], sk_ctl[1])

  __device__ void k_range(const Tile& tile, int& kb0, int& kb1) const {
    if (MODE == kKGrouped) {
      kb0 = tile_start[tile.g];
      kb1 = tile_start[tile.g + 1];
    } else {
      kb0 = kb_lo;
      kb1 = kb_hi;
    }
  }

  // The it-th work item of this CTA: a tile and the K blocks [kb0, kb1) this
  // CTA accumulates for it.  Returns -1 past the last item, 0 for a tile the
  // walk skips (contiguous blocks of padding), 1 otherwise.  Items are
  // visited with it = 0, 1, 2, ... by every role.
  __device__ int item(int it, Tile& tile, int& kb0, int& kb1) {
    tile.kind = kItemFull;
    tile.sk = -1;
    if constexpr (SK) {
      // stream-K: tiles [0, dp) go one per CTA per wave; the K blocks of the
      // tiles [dp, total) form sk_units units of which CTA c takes
      // [c * U / P, (c + 1) * U / P), tile after tile (the host keeps
      // sk_units * P below 2^32; the range is computed once per CTA)
      const int dp = args->sk_dp_tiles;
      const int n_dp = first < dp ? (dp - first + stride - 1) / stride : 0;
      if (it < n_dp) {
        get(first + it * stride, tile);
        kb0 = 0;
        kb1 = args->k_blocks;
        return 1;
      }
      const uint32_t lo = sk_ctl[0], hi = sk_ctl[1], kbt = (uint32_t)args->k_blocks;
      const uint32_t ts = lo / kbt + (uint32_t)(it - n_dp);
      const uint32_t t0 = ts * kbt;
      if (lo >= hi || t0 >= hi) return -1;
      kb0 = (int)((lo > t0 ? lo : t0) - t0);
      kb1 = (int)((hi < t0 + kbt ? hi : t0 + kbt) - t0);
      get(dp + (int)ts, tile);
      tile.kind = kb0 > 0 ? kItemPart : ((uint32_t)kb1 < kbt ? kItemOwner : kItemFull);
      tile.sk = (int)ts;
      return 1;
    }
    const int t = first + it * stride;
    if (t >= total) return -1;
    if (!get(t, tile)) return 0;
    k_range(tile, kb0, kb1);
    return 1;
  }
  // Stream-K units of CTA c: [c * U / P, (c + 1) * U / P).
  __device__ void sk_range(int c, uint32_t& lo, uint32_t& hi) const {
    const uint32_t u = (uint32_t)args->sk_units;
    lo = u * (uint32_t)c / gridDim.x;
    hi = u * (uint32_t)(c + 1) / gridDim.x;
  }
  // Whether the tile walk (without stream-K) has an item after the it-th.
  __device__ bool has_next(int it) const { return first + (it + 1) * stride < total; }

  __device__ bool get(int t, Tile& tile) {
    if (MODE == kContiguous && BM == 2 * kBlockM) {
      // pairs of one group's 128-row blocks, rastered like dense M blocks
      const int npairs = tile_start[args->num_groups];
      const int per_band = args->band * args->n_blocks;
      const int b = t / per_band;
      const int rem = t - b * per_band;
      const int rows = min(args->band, npairs - b * args->band);
      tile.nb = rem / rows;
      const int p = b * args->band + rem % rows;
      tile.mb = p;
      const uint32_t w = pairs[p];
      tile.b0 = (int)(w & 0xFFFFu);
      tile.b1 = (w >> 16) == 0xFFFFu ? -1 : (int)(w >> 16);
      // the group: the last g with tile_start[g] <= p (it has pairs)
      int lo = 0, hi = args->num_groups;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_start[mid] <= p) lo = mid;
        else hi = mid;
      }
      tile.g = lo;
      return true;
    }
    if (MODE == kKGrouped) {
      // multicast pairs: the walk covers pairs of M blocks, a CTA takes one
      const int mbs = pair_rank >= 0 ? (args->m_blocks + 1) >> 1 : args->m_blocks;
      const int per_group = mbs * args->n_blocks;
      tile.g = t / per_group;
      const int r = t - tile.g * per_group;
      const int per_band = args->band * args->n_blocks;
      const int b = r / per_band;
      const int rem = r - b * per_band;
      const int rows = min(args->band, mbs - b * args->band);
      tile.nb = rem / rows;
      tile.mb = b * args->band + rem % rows;
      if (pair_rank >= 0) tile.mb = 2 * tile.mb + pair_rank;
      return true;
    }
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
    const int mbs = pair_rank >= 0 ? (args->m_blocks + 1) >> 1 : args->m_blocks;
    const int rows = min(args->band, mbs - b * args->band);
    tile.nb = rem / rows;
    tile.mb = b * args->band + rem % rows;
    // a pair's second M block may lie past M (odd count): its loads read
    // zeros and its epilogue stores nothing
    if (pair_rank >= 0) tile.mb = 2 * tile.mb + pair_rank;
    tile.g = 0;
    if (MODE == kContiguous) {
      const int g = __ldg(args->m_indices + (int64_t)tile.mb * kBlockM);
      if (g < 0) return false;
      if (g >= args->num_groups) {
        record_error(args->err, DG_ERR_DEVICE_BAD_INDEX, kSiteContiguousIndex);
        return false;
      }
      tile.g = g;
    }
    return true;
  }
};

// Walks the scale packs (tile, K block / 4) of this CTA in the order the MMA
// consumes them, skipping the tiles the scheduler skips and tiles without K
// blocks.  A tile's K blocks [kb0, kb1) touch the packs kb0 / 4 ..
// (kb1 - 1) / 4; the MMA thread starts a pack at kb0 and at every K block
// that is a multiple of 4, so both walk the same sequence.
template <class Sched>
struct PackCursor {
  Sched s;
  int it, kp, kp_end;
  Tile tile;
  bool done;

  __device__ void init(const Sched& sch) {
    s = sch;
    it = -1;
    next_tile();
  }
  __device__ void next_tile() {
    done = true;
    for (++it;; ++it) {
      int kb0, kb1;
      const int st = s.item(it, tile, kb0, kb1);
      if (st < 0) return;
      if (st == 0 || kb0 >= kb1) continue;
      kp = kb0 >> 2;
      kp_end = ((kb1 - 1) >> 2) + 1;
      done = false;
      return;
    }
  }
  __device__ void advance() {
    if (++kp >= kp_end) next_tile();
  }
};

// Waits until the phase with `parity` of `bar` has completed, ignoring the
// abort flag (used to drain in-flight work before exit), bounded in time.
// INL: inlined (kernels using setmaxnreg), else out of line.
__device__ __forceinline__ void wait_drain_body(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                unsigned long long* err, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0 && (global_timer_ns() - t0 > timeout_ns || it >= (1u << 30))) {
      record_error(err, DG_ERR_DEVICE_TIMEOUT, site);
      return;
    }
  }
}
static __device__ __noinline__ void wait_drain_outlined(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                        unsigned long long* err, uint32_t site) {
  wait_drain_body(bar, parity, timeout_ns, err, site);
}
template <bool INL = false>
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           unsigned long long* err, uint32_t site) {
  if constexpr (INL) wait_drain_body(bar, parity, timeout_ns, err, site);
  else wait_drain_outlined(bar, parity, timeout_ns, err, site);
}

// Suspend-time hint of the single-CTA kernel's waits (see mbar_try_wait_hint).
constexpr uint32_t kSuspendHintNs = 32;

// Single-thread wait: one try first (the usual case), the bounded loop only
// when the phase is not complete yet.
template <uint32_t HINT_NS = 0, bool INL = false>
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t timeout_ns, unsigned long long* err,
                                         uint32_t site) {
  if (mbar_try_wait_hint<HINT_NS>(bar, parity)) return true;
  if constexpr (INL) return wait_bounded_body<HINT_NS>(bar, parity, abort_flag, timeout_ns, err, site);
  else return wait_bounded<HINT_NS>(bar, parity, abort_flag, timeout_ns, err, site);
}

// Whole-warp wait: lane 0 waits, the result is broadcast, and the warp
// reconverges (so the other lanes observe what lane 0 acquired).
template <uint32_t HINT_NS = 0, bool INL = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, unsigned long long* err,
                                          uint32_t site) {
  const int lane = threadIdx.x & 31;
  int ok = 0;
  if (lane == 0) ok = wait_one<HINT_NS, INL>(bar, parity, abort_flag, timeout_ns, err, site) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Whole-warp wait with cluster-scope acquire (barriers other CTAs arrive on).
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, uint64_t timeout_ns,
                                                  unsigned long long* err, uint32_t site) {
  const int lane = threadIdx.x & 31;
  int ok = 0;
  if (lane == 0)
    ok = (mbar_try_wait_cluster(bar, parity) ||
          wait_bounded_cluster(bar, parity, abort_flag, timeout_ns, err, site)) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Stores 32 accumulator columns of one row (+ C), 16 bytes at a time, the
// columns at or past n skipped (n % 8 == 0).
__device__ __forceinline__ void store_row_chunk(const uint32_t (&r)[32], __nv_bfloat16* dp,
                                                const __nv_bfloat16* cp, int cols_left) {
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    if (8 * p < cols_left) {
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

// Stores 32 FP32 accumulator columns of one row (+ FP32 C), 16 bytes at a
// time, the columns at or past n skipped (n % 4 == 0).  `zero`: the tile had
// no K blocks, so the result is C (or 0) and the accumulator is not read.
__device__ __forceinline__ void store_row_chunk_f32(const uint32_t (&r)[32], float* dp,
                                                    const float* cp, int cols_left, bool zero) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    if (4 * p < cols_left) {
      float4 v = zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                      : make_float4(__uint_as_float(r[4 * p]), __uint_as_float(r[4 * p + 1]),
                                    __uint_as_float(r[4 * p + 2]), __uint_as_float(r[4 * p + 3]));
      if (cp) {
        const float4 c = *reinterpret_cast<const float4*>(cp + 4 * p);
        if (zero) {
          v = c;
        } else {
          v.x += c.x;
          v.y += c.y;
          v.z += c.z;
          v.w += c.w;
        }
      }
      *reinterpret_cast<float4*>(dp + 4 * p) = v;
    }
  }
}

// FP32 output: one 32 x 32 chunk of a warp's quarter as two 32 x 16 halves,
// each written into a free staging buffer (64-byte rows, 16-byte piece j of
// row r at r * 64 + 16 * (j ^ ((r >> 1) & 3)), the layout of
// CU_TENSOR_MAP_SWIZZLE_64B) and TMA-stored at (col0 + 16 h, out_row0).  A
// half that starts at or past n is skipped (n % 16 == 0).
__device__ __forceinline__ void emit_chunk_tma_f32(const float (&f)[32], uint8_t* ebuf,
                                                   uint32_t& nchunk, const CUtensorMap* tm_d,
                                                   int col0, int n, int64_t out_row0, int lane) {
  const uint32_t my_row_off = (uint32_t)lane * 64u;
  const uint32_t my_swz = ((uint32_t)lane >> 1) & 3u;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (col0 + 16 * h >= n) break;
    uint8_t* buf = ebuf + (nchunk & 1u) * kEpiBuf;
    if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4*>(buf + my_row_off + 16u * ((uint32_t)j ^ my_swz)) =
          make_float4(f[16 * h + 4 * j], f[16 * h + 4 * j + 1], f[16 * h + 4 * j + 2],
                      f[16 * h + 4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm_d, smem_u32(buf), col0 + 16 * h, (int32_t)out_row0);
      bulk_commit_group();
    }
    ++nchunk;
  }
}

// One 32 x 32 output chunk of a warp's quarter (row = lane): + C (coalesced
// loads staged through `buf`), round to BF16 and write into `buf` with the
// 64-byte swizzle.  `buf` must be free.  Rows past m are skipped for C when
// dense_rows.
__device__ __forceinline__ void stage_chunk_bf16(float (&f)[32], uint8_t* buf, const GemmArgs& args,
                                                 int col0, int64_t out_row0, int row0,
                                                 bool dense_rows, int lane) {
  const uint32_t my_row_off = (uint32_t)lane * 64u;
  const uint32_t my_swz = ((uint32_t)lane >> 1) & 3u;
  if (args.c) {
    // coalesced: lane l fetches 16 bytes of rows l/4 + 8i, piece l % 4
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (lane >> 2) + 8 * i, pc = lane & 3;
      const int gcol = col0 + pc * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (gcol < args.n && (!dense_rows || row0 + r < args.m))
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
}

// One row of a chunk already rounded to BF16, 16 bytes at a time, the columns
// at or past n skipped (n % 8 == 0).
__device__ __forceinline__ void store_packed_row(const uint32_t (&p)[16], __nv_bfloat16* dp,
                                                 int cols_left) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (8 * q < cols_left)
      *reinterpret_cast<uint4*>(dp + 8 * q) = make_uint4(p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
}

// A chunk already rounded to BF16 (row = lane, 16 words of column pairs)
// written into `buf` with the 64-byte swizzle and TMA-stored at
// (col0, out_row0).  `buf` must be free.
__device__ __forceinline__ void emit_packed_tma(const uint32_t (&p)[16], uint8_t* buf,
                                                const CUtensorMap* tm_d, int col0, int64_t out_row0,
                                                int lane) {
  const uint32_t my_row_off = (uint32_t)lane * 64u;
  const uint32_t my_swz = ((uint32_t)lane >> 1) & 3u;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(buf + my_row_off + 16u * ((uint32_t)j ^ my_swz)) =
        make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm_d, smem_u32(buf), col0, (int32_t)out_row0);
    bulk_commit_group();
  }
}

// 32 columns of row `crow` of C from col0, as BF16 pairs (dst[i] holds
// columns 2i, 2i + 1); 0 past M or N.  The register-held epilogues fetch C
// row by row (a lane's own row), so a warp load touches 32 rows: where C's
// base and row stride are multiples of 32 bytes (args.c_v8) each lane reads
// a whole 32-byte sector per load, halving the loads of the 16-byte form.
__device__ __forceinline__ void load_c_row32(uint32_t (&dst)[16], const GemmArgs& args, int crow, int col0) {
  const __nv_bfloat16* src = args.c + (int64_t)crow * args.ldc + col0;
  const bool row_ok = crow < args.m;
  if (args.c_v8) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t* o = dst + 8 * h;
      if (row_ok && col0 + 16 * h + 16 <= args.n) {
        asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]), "=r"(o[4]), "=r"(o[5]), "=r"(o[6]),
                       "=r"(o[7])
                     : "l"(src + 16 * h));
      } else {
        // the last 8 columns of a row ending inside this 16-column piece (N % 16 == 8)
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row_ok && col0 + 16 * h < args.n) v = __ldg(reinterpret_cast<const uint4*>(src + 16 * h));
        o[0] = v.x;
        o[1] = v.y;
        o[2] = v.z;
        o[3] = v.w;
        o[4] = o[5] = o[6] = o[7] = 0u;
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (row_ok && col0 + 8 * q < args.n) v = __ldg(reinterpret_cast<const uint4*>(src + 8 * q));
      dst[4 * q] = v.x;
      dst[4 * q + 1] = v.y;
      dst[4 * q + 2] = v.z;
      dst[4 * q + 3] = v.w;
    }
  }
}

// C of one 32 x 32 chunk, fetched coalesced (lane l: 16 bytes of rows l/4 + 8i,
// piece l % 4) into registers, ahead of the chunk's turn; zero past M and N.
__device__ __forceinline__ void load_c_chunk(uint4 (&cv)[4], const GemmArgs& args, int col0,
                                             int64_t out_row0, int row0, int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (lane >> 2) + 8 * i, pc = lane & 3;
    const int gcol = col0 + pc * 8;
    cv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (gcol < args.n && row0 + r < args.m)
      cv[i] = __ldg(reinterpret_cast<const uint4*>(args.c + (out_row0 + r) * args.ldc + gcol));
  }
}

// The chunk + C (prefetched by load_c_chunk, passed through `buf` to reach
// each row's lane), rounded to BF16, staged and TMA-stored at (col0,
// out_row0).  `buf` must be free.
__device__ __forceinline__ void emit_chunk_tma_c(float (&f)[32], const uint4 (&cv)[4], uint8_t* buf,
                                                 const CUtensorMap* tm_d, int col0, int64_t out_row0,
                                                 int lane) {
  const uint32_t my_row_off = (uint32_t)lane * 64u;
  const uint32_t my_swz = ((uint32_t)lane >> 1) & 3u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (lane >> 2) + 8 * i, pc = lane & 3;
    *reinterpret_cast<uint4*>(buf + r * 64 + 16 * (pc ^ ((r >> 1) & 3))) = cv[i];
  }
  __syncwarp();
  uint32_t p[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 c4 = *reinterpret_cast<const uint4*>(buf + my_row_off + 16u * ((uint32_t)j ^ my_swz));
    const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      p[4 * j + i] = pack_bf16x2(f[8 * j + 2 * i] + __uint_as_float(cw[i] << 16),
                                 f[8 * j + 2 * i + 1] + __uint_as_float(cw[i] & 0xFFFF0000u));
  }
  emit_packed_tma(p, buf, tm_d, col0, out_row0, lane);
}

// The chunk staged, then TMA-stored at (col0, out_row0) (the store clips at M
// and N).  `buf` must be free: its previous store has finished reading it.
__device__ __forceinline__ void emit_chunk_tma(float (&f)[32], uint8_t* buf,
                                               const CUtensorMap* tm_d, const GemmArgs& args,
                                               int col0, int64_t out_row0, int row0,
                                               bool dense_rows, int lane) {
  stage_chunk_bf16(f, buf, args, col0, out_row0, row0, dense_rows, lane);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm_d, smem_u32(buf), col0, (int32_t)out_row0);
    bulk_commit_group();
  }
}

template <int BN, int STAGES, int MODE, int KSPLIT, int BM = kBlockM, bool EPI8 = false, bool SK = false,
          bool MC = false>
__global__ void __launch_bounds__(EPI8 ? kGemmThreadsEpi8 : kGemmThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfa,
                    const __grid_constant__ CUtensorMap tm_sfb,
                    const __grid_constant__ CUtensorMap tm_d, const GemmArgs args) {
  using L = GemmLayout<BN, BM>;
  using P = GemmPlan<BN, STAGES, KSPLIT, BM>;
  // MC: clusters of two CTAs on the same column block of B (of the same
  // expert, K-grouped) and adjacent row blocks of A; each loads half of the B
  // tile into both CTAs' stage (TMA multicast: half the rows of a K-major
  // tile, one of the two 128-column boxes of an MN-major one), so L2 serves B
  // once per pair
  static_assert(!MC || (!SK && KSPLIT == 1 && EPI8 &&
                        ((MODE == kDense && BM == 2 * kBlockM) || (MODE == kKGrouped && BM == kBlockM && BN == 256))),
                "multicast pairs: dense 256-row tiles or K-grouped 128 x 256 tiles, eight epilogue warps");
  constexpr int CL = MC ? 2 : KSPLIT;  // CTAs per cluster
  constexpr int NUM_ACC = P::kNumAcc;
  constexpr int MH = L::kMH;  // 128-row halves of a tile
  static_assert(KSPLIT == 1 || MODE == kDense, "split-K is for the dense form");
  static_assert(!EPI8 || (NUM_ACC == 1 && ((BM == 2 * kBlockM && MODE == kDense) ||
                                            (BM == kBlockM && MODE == kKGrouped && BN == 256))),
                "eight epilogue warps: 256-row dense tiles, or 128 x 256 K-grouped tiles, with one accumulator");
  static_assert(!SK || EPI8, "stream-K: 256-row dense tiles with eight epilogue warps");
  // setmaxnreg split of the eight-epilogue-warp layout: the K-grouped role
  // warps (MN-major loads, per-expert K ranges) need more than 56 registers,
  // its epilogue (128 FP32 columns per thread) fewer than 224
  // (the K-grouped role warps spill at 56, and with multicast pairs below 104)
  constexpr int kRolesRegs = MODE == kKGrouped ? (MC ? 104 : 72) : kRegsRoles;
  constexpr int kEpiRegs = MODE == kKGrouped ? (MC ? 192 : 208) : kRegsEpi;
  static_assert(128 * kRolesRegs + 256 * kEpiRegs <= kGemmThreadsEpi8 * 168 && kRolesRegs % 8 == 0 &&
                    kEpiRegs % 8 == 0,
                "setmaxnreg split within the launch's registers");
  static_assert(BM == kBlockM || (BM == 2 * kBlockM && (MODE == kDense || MODE == kContiguous) && KSPLIT == 1) ||
                    (BM == kBlockM / 2 && MODE == kDense),
                "256-row tiles are for the dense NT and contiguous forms without split-K; "
                "64-row A slots for the dense NT form");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  uint8_t* sfbuf = smem + STAGES * L::kStageBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t* epi_smem = sfbuf + kSfSlots * L::kSfBufBytes;  // 1024-aligned
  uint8_t* recv = epi_smem + kEpiBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(recv + P::kRecvBytes);
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto sffull = [&](int p) { return smem_u32(bars + 2 * STAGES + p); };
  auto sfready = [&](int p) { return smem_u32(bars + 2 * STAGES + kSfSlots + p); };
  auto sfempty = [&](int p) { return smem_u32(bars + 2 * STAGES + 2 * kSfSlots + p); };
  constexpr int kB0 = 2 * STAGES + 3 * kSfSlots;
  auto tfull = [&](int a) { return smem_u32(bars + kB0 + a); };
  auto tempty = [&](int a) { return smem_u32(bars + kB0 + 2 + a); };
  const uint32_t drain = smem_u32(bars + kB0 + 4);
  // split-K: quarter q's partials from the other CTAs have landed / every
  // other CTA has consumed what this CTA sent it for quarter q
  auto recv_full = [&](int q) { return smem_u32(bars + kB0 + 5 + q); };
  auto recv_free = [&](int q) { return smem_u32(bars + kB0 + 9 + q); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kB0 + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // split-K: set by another CTA of the cluster that aborted (see the teardown)
  volatile int* peer_abort = reinterpret_cast<volatile int*>(tmem_slot + 2);
  // stream-K: this CTA's units [sk_ctl[0], sk_ctl[1]) and its tile-walk items
  uint32_t* const sk_ctl = tmem_slot + 4;
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 8);
  int* group_valid = tile_start + (kMaxMaskedGroups + 1);
  unsigned long long* const err = args.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), MC ? 2 : 1);  // MC: a stage is free once both CTAs' MMAs are done with it
    }
    for (int p = 0; p < kSfSlots; ++p) {
      mbar_init(sffull(p), 1);
      mbar_init(sfready(p), 1);
      mbar_init(sfempty(p), 1);
    }
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), EPI8 ? 8 : 4);
    }
    mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(recv_full(q), KSPLIT > 1 ? KSPLIT - 1 : 1);
      mbar_init(recv_free(q), KSPLIT > 1 ? KSPLIT - 1 : 1);
    }
    *abort_flag = 0;
    *peer_abort = 0;
    if constexpr (SK) {
      const uint32_t u = (uint32_t)args.sk_units;
      sk_ctl[0] = u * blockIdx.x / gridDim.x;
      sk_ctl[1] = u * (blockIdx.x + 1) / gridDim.x;
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_sfa);
    tma_prefetch_desc(&tm_sfb);
    tma_prefetch_desc(&tm_d);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  // Set-up above overlaps the previous kernel's tail under PDL; from here on
  // every thread may read what that kernel wrote.
  griddep_wait();
  if (MODE == kMasked && warp == 2) {
    for (int g = lane; g < args.num_groups; g += 32) {
      const int v = __ldg(args.masked_m + g);
      const int c = v < 0 ? 0 : (v > args.m ? args.m : v);
      if (c != v) record_error(err, DG_ERR_DEVICE_BAD_INDEX, kSiteMaskedCount);
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
  // Contiguous form with 256-row tiles: each group's 128-row blocks (found by
  // the group id of their first row; all -1 blocks are skipped) are paired in
  // any order - rows are independent, so the pairing does not change a
  // result - and a group with an odd count ends with a half-empty pair.
  // tile_start[g] = first pair of group g; pairs[p] = block ids (16 bits each,
  // 0xFFFF = none).  The host bounds the pairs by kMaxBlockPairs.
  uint32_t* const pair_words = reinterpret_cast<uint32_t*>(group_valid + kMaxMaskedGroups);
  if (MODE == kContiguous && BM == 2 * kBlockM && warp == 2) {
    int* counts = group_valid;
    uint16_t* slot = reinterpret_cast<uint16_t*>(pair_words);
    for (int g = lane; g < args.num_groups; g += 32) counts[g] = 0;
    for (int i = lane; i < kMaxBlockPairs; i += 32) pair_words[i] = 0xFFFFFFFFu;
    __syncwarp();
    for (int b = lane; b < args.m_blocks; b += 32) {
      const int g = __ldg(args.m_indices + (int64_t)b * kBlockM);
      if (g >= args.num_groups) record_error(err, DG_ERR_DEVICE_BAD_INDEX, kSiteContiguousIndex);
      else if (g >= 0) atomicAdd(counts + g, 1);
    }
    __syncwarp();
    if (lane == 0) {
      int acc = 0;
      for (int g = 0; g < args.num_groups; ++g) {
        tile_start[g] = acc;
        const int c = counts[g];
        counts[g] = 2 * acc;  // from here: the group's next free block slot
        acc += (c + 1) / 2;
      }
      // the host bounds the pairs; past the table a block would be dropped
      if (acc > kMaxBlockPairs) record_error(err, DG_ERR_DEVICE_BAD_INDEX, kSiteContiguousIndex);
      tile_start[args.num_groups] = acc < kMaxBlockPairs ? acc : kMaxBlockPairs;
    }
    __syncwarp();
    for (int b = lane; b < args.m_blocks; b += 32) {
      const int g = __ldg(args.m_indices + (int64_t)b * kBlockM);
      if (g >= 0 && g < args.num_groups) {
        const int pos = atomicAdd(counts + g, 1);
        if (pos < 2 * kMaxBlockPairs) slot[pos] = (uint16_t)b;
      }
    }
  }
  if (MODE == kKGrouped && warp == 2) {
    // Experts' K blocks: sizes must be >= 0 and multiples of 128; a bad size
    // counts as 0 and K blocks past the end of A and B are dropped, both
    // flagged.
    for (int g = lane; g < args.num_groups; g += 32) {
      const int v = __ldg(args.ks + g);
      const bool bad = v < 0 || (v % kBlockK) != 0;
      if (bad) record_error(err, DG_ERR_DEVICE_BAD_INDEX, kSiteKGroupSize);
      group_valid[g] = bad ? 0 : v / kBlockK;
    }
    __syncwarp();
    if (lane == 0) {
      int acc = 0;
      for (int g = 0; g < args.num_groups; ++g) {
        tile_start[g] = acc;
        int next = acc + group_valid[g];
        if (next > args.k_blocks) {
          record_error(err, DG_ERR_DEVICE_BAD_INDEX, kSiteKGroupSize);
          next = args.k_blocks;
        }
        acc = next;
      }
      tile_start[args.num_groups] = acc;
    }
  }
  __syncthreads();
  if (CL > 1) cluster_sync_all();  // every CTA's barriers exist before remote arrivals
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();

  // tile loop of this CTA (of this cluster, with split-K) and its K slice
  const uint32_t krank = CL > 1 ? cluster_ctarank() : 0u;
  const int first_tile = (int)blockIdx.x / CL;
  const int tile_stride = (int)gridDim.x / CL;
  const int kb_per = (args.k_blocks + KSPLIT - 1) / KSPLIT;
  const int kb_begin = KSPLIT > 1 ? min(args.k_blocks, (int)krank * kb_per) : 0;
  const int kb_end = KSPLIT > 1 ? min(args.k_blocks, kb_begin + kb_per) : args.k_blocks;

  Scheduler<MODE, BM, SK> sched;
  sched.sk_ctl = sk_ctl;
  sched.args = &args;
  sched.tile_start = tile_start;
  sched.group_valid = group_valid;
  sched.pairs = pair_words;
  sched.cursor = 0;
  sched.kb_lo = kb_begin;
  sched.kb_hi = kb_end;
  sched.first = first_tile;
  sched.stride = tile_stride;
  sched.pair_rank = MC ? (int)krank : -1;
  sched.total = MODE == kMasked      ? tile_start[args.num_groups]
                : MODE == kKGrouped ? args.num_groups * (MC ? (args.m_blocks + 1) >> 1 : args.m_blocks) * args.n_blocks
                : (MODE == kContiguous && BM == 2 * kBlockM) ? tile_start[args.num_groups] * args.n_blocks
                : MC                ? ((args.m_blocks + 1) >> 1) * args.n_blocks
                                    : args.m_blocks * args.n_blocks;
  const uint64_t tmo = args.timeout_ns;

  // Roles: warp 0 producer, warp 1 MMA issuer, warp 2 scale warp, the rest
  // epilogue.  With eight epilogue warps, warpgroup 0 (the three role warps
  // and an idle warp) hands registers to the two epilogue warpgroups at the
  // start of each warpgroup's branch.
  if (EPI8 ? warp < 4 : warp < 3) {
    if constexpr (EPI8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRolesRegs) : "memory");
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // A single M block of fewer than 128 rows is loaded as a box of
      // round_up(M, 8) rows: the rest of the A tile keeps stale bytes, which
      // only reach accumulator rows that are never stored.
      const uint32_t tx_ab = args.a_box_rows > 0 ? (uint32_t)(args.a_box_rows * kBlockK + L::kBytesB) : L::kTxAB;
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0, issued_parity = 0;  // stages: last fill's phase parity
        bool ok = true;
        for (int it = 0; ok; ++it) {
          Tile tile;
          int kb0, kb1;
          const int st_it = sched.item(it, tile, kb0, kb1);
          if (st_it < 0) break;
          if (st_it == 0) continue;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_one<kSuspendHintNs, EPI8>(empty(stage), phase ^ 1u, abort_flag, tmo, err, kSiteProducerEmpty)) {
              ok = false;
              break;
            }
            const uint32_t sb = smem_u32(smem + stage * L::kStageBytes);
            const uint32_t fb = full(stage);
            mbar_arrive_expect_tx(fb, tx_ab);
            const int kx = kb * kBlockK, my = tile.mb * BM;
            if (args.debug_drop_load && blockIdx.x == 0 && it == 0 &&
                kb + 1 == args.debug_drop_load) {
              // injected failure: the stage is armed but never filled
              issued |= 1u << stage;
              issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            // MN-major tiles ([K, M] / [K, N] storage): 128 K rows of 128 bytes
            // per box; a 256-column B tile is two boxes 16 KB apart
            if constexpr (DG_DEBUG_CHECKS) {
              // K block in range; innermost coordinates on 16-byte boundaries;
              // rows, column tiles and groups inside their tensors
              DG_CHECK(err, kb >= 0 && kb < args.k_blocks && (kx & 15) == 0, kSiteCheckLoadA);
              if constexpr (a_mn_major(MODE)) DG_CHECK(err, (my & 15) == 0 && my < (MC ? args.m + BM : args.m), kSiteCheckLoadA);
              else if (MODE == kContiguous && BM == 2 * kBlockM)
                DG_CHECK(err, tile.b0 >= 0 && tile.b0 < args.m_blocks && tile.b1 < args.m_blocks, kSiteCheckLoadA);
              else DG_CHECK(err, my >= 0 && my < (MC ? args.m + BM : args.m), kSiteCheckLoadA);
              DG_CHECK(err, tile.nb >= 0 && tile.nb * BN < args.n && ((tile.nb * BN) & 7) == 0 &&
                                (MODE == kKGrouped || (tile.g >= 0 && tile.g < args.num_groups)),
                       kSiteCheckLoadB);
            }
            if constexpr (a_mn_major(MODE)) tma_load_2d(sb, &tm_a, fb, my, kx);
            else if (MODE == kMasked) tma_load_3d(sb, &tm_a, fb, kx, my, tile.g);
            else if (MODE == kContiguous && BM == 2 * kBlockM) {
              // the pair's two blocks (a half-empty pair loads its block twice)
              tma_load_2d(sb, &tm_a, fb, kx, tile.b0 * kBlockM);
              tma_load_2d(sb + kBlockM * kBlockK, &tm_a, fb, kx, (tile.b1 >= 0 ? tile.b1 : tile.b0) * kBlockM);
            } else tma_load_2d(sb, &tm_a, fb, kx, my);
            if constexpr (b_mn_major(MODE) && MC) {
              // this CTA's 128-column box of the B tile, into the same place in both CTAs
              tma_load_2d_both(sb + L::kOffB + krank * 16384u, &tm_b, fb, tile.nb * BN + (int)krank * 128, kx);
            } else if constexpr (b_mn_major(MODE)) {
  #pragma unroll
              for (int h = 0; h < BN / 128; ++h)
                tma_load_2d(sb + L::kOffB + h * 16384, &tm_b, fb, tile.nb * BN + h * 128, kx);
            } else if constexpr (MC) {
              // this CTA's half of the B tile, into the same place in both CTAs
              tma_load_3d_both(sb + L::kOffB + krank * (uint32_t)(BN / 2 * kBlockK), &tm_b, fb, kx,
                               tile.nb * BN + (int)krank * (BN / 2), tile.g);
            } else {
              tma_load_3d(sb + L::kOffB, &tm_b, fb, kx, tile.nb * BN, tile.g);
            }
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // Drain: every copy this thread issued has landed before smem is released.
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s))
            wait_drain<EPI8>(full(s), (issued_parity >> s) & 1u, tmo, err, kSiteProducerDrain);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc0 = idesc_mxf8_e4m3(kBlockM, BN, 0, 0);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t pack = 0;
        uint32_t sf_tmem = tmem_base + (uint32_t)P::kSfBase;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int it = 0; ok; ++it) {
          Tile tile;
          int kb0, kb1;
          const int st_it = sched.item(it, tile, kb0, kb1);
          if (st_it < 0) break;
          if (st_it == 0) continue;
          if (!wait_one<kSuspendHintNs, EPI8>(tempty(acc), acc_phase ^ 1u, abort_flag, tmo, err, kSiteMmaTmemEmpty)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * MH * BN);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_one<kSuspendHintNs, EPI8>(full(stage), phase, abort_flag, tmo, err, kSiteMmaFull)) {
              ok = false;
              break;
            }
            uint8_t* st = smem + stage * L::kStageBytes;
            const int slot = (int)(pack % kSfSlots);
            if (kb == kb0 || (kb & 3) == 0) {
              if (!wait_one<kSuspendHintNs, EPI8>(sfready(slot), (pack / kSfSlots) & 1u, abort_flag, tmo, err,
                            kSiteMmaScaleReady)) {
                ok = false;
                break;
              }
              // the scale warp has copied this pack into the slot's TMEM columns
              tc_fence_after();
              sf_tmem = tmem_base + (uint32_t)(P::kSfBase + slot * L::kSfCols);
            }
            DG_CHECK(err, args.debug_plant_check == 0 && sf_tmem - tmem_base + (uint32_t)L::kSfCols <= 512u &&
                              d_tmem - tmem_base + (uint32_t)(MH * BN) <= (uint32_t)P::kSfBase,
                     kSiteCheckTmem);
            const uint32_t sel = (uint32_t)(kb & 3);
            const uint32_t idesc = idesc0 | (sel << 4) | (sel << 29);
            // K-major operands advance 32 bytes per 32-deep K step; MN-major
            // ones 4 groups of 8 K rows (4096 bytes): descriptor units of 16 B
            const uint64_t adesc = a_mn_major(MODE) ? smem_desc_mnmajor_sw128(smem_u32(st))
                                                    : smem_desc_kmajor_sw128(smem_u32(st));
            const uint64_t bdesc = b_mn_major(MODE) ? smem_desc_mnmajor_sw128(smem_u32(st + L::kOffB))
                                                    : smem_desc_kmajor_sw128(smem_u32(st + L::kOffB));
            constexpr uint32_t a_step = a_mn_major(MODE) ? 256u : 2u;
            constexpr uint32_t b_step = b_mn_major(MODE) ? 256u : 2u;
            constexpr uint32_t major_bits = (a_mn_major(MODE) ? kIdescMnMajorA : 0u) |
                                            (b_mn_major(MODE) ? kIdescMnMajorB : 0u);
            // a 256-row tile: the second half's A rows start 16 KB further
            // (1024 descriptor units), its accumulator BN columns further
  #pragma unroll
            for (int j = 0; j < 4; ++j)
  #pragma unroll
              for (int h = 0; h < MH; ++h)
                tc_mma_mxf8(d_tmem + h * BN, adesc + 1024u * h + a_step * j, bdesc + b_step * j,
                            idesc | major_bits, sf_tmem + 4 * h, sf_tmem + 4 * MH,
                            (kb != kb0 || j != 0) ? 1u : 0u);
            // MC: the other CTA writes half of this stage too, so both are told
            if constexpr (MC) tc_commit_both(empty(stage));
            else tc_commit(empty(stage));
            if ((kb & 3) == 3 || kb == kb1 - 1) {
              tc_commit(sfempty(slot));  // the pack's buffer and TMEM slot are free
              ++pack;
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(tfull(acc));
          if (++acc == NUM_ACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        // Drain: all MMAs and TMEM copies issued here complete before TMEM is freed.
        tc_commit(drain);
        wait_drain<EPI8>(drain, 0, tmo, err, kSiteDrain);
      }
      __syncwarp();
    } else if (warp == 2) {
      // ------------------------------------------------------------ scale warp
      // Two cursors walk the same sequence of packs (tile, K block / 4): one
      // loads up to kSfLookahead packs ahead, the other lays them out in order.
      PackCursor<Scheduler<MODE, BM, SK>> ld, lay;
      ld.init(sched);
      lay.init(sched);
      uint32_t n_loaded = 0, n_laid = 0;
      bool ok = true;
      while (!lay.done && ok) {
        while (!ld.done && n_loaded < n_laid + kSfLookahead) {
          const int slot = (int)(n_loaded % kSfSlots);
          int go = 1;
          if (lane == 0) {
            go = wait_one<kSuspendHintNs, EPI8>(sfempty(slot), ((n_loaded / kSfSlots) & 1u) ^ 1u, abort_flag, tmo, err,
                          kSiteScaleEmpty) ? 1 : 0;
            if (go) {
              const uint32_t buf = smem_u32(sfbuf + slot * L::kSfBufBytes);
              const uint32_t bar = sffull(slot);
              const int my = ld.tile.mb * BM, kp = ld.kp;
              mbar_arrive_expect_tx(bar, L::kTxSF);
              DG_CHECK(err, kp >= 0 && kp < (args.k_blocks + 3) / 4 && my >= 0 &&
                                (MODE == kContiguous && BM == 2 * kBlockM ? ld.tile.b0 < args.m_blocks
                                                                          : my < (MC ? args.m + BM : args.m)),
                       kSiteCheckScale);
              if (MODE == kMasked) tma_load_3d(buf + L::kRawA, &tm_sfa, bar, my, kp, ld.tile.g);
              else if (MODE == kContiguous && BM == 2 * kBlockM) {
                tma_load_2d(buf + L::kRawA, &tm_sfa, bar, ld.tile.b0 * kBlockM, kp);
                tma_load_2d(buf + L::kRawA + 512, &tm_sfa, bar,
                            (ld.tile.b1 >= 0 ? ld.tile.b1 : ld.tile.b0) * kBlockM, kp);
              } else tma_load_2d(buf + L::kRawA, &tm_sfa, bar, my, kp);
              tma_load_3d(buf + L::kRawB, &tm_sfb, bar, ld.tile.nb * BN, kp,
                          MODE == kKGrouped ? 0 : ld.tile.g);
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
        if (!warp_wait<kSuspendHintNs, EPI8>(sffull(slot), (n_laid / kSfSlots) & 1u, abort_flag, tmo, err, kSiteScaleFull)) {
          ok = false;
          break;
        }
        uint8_t* buf = sfbuf + slot * L::kSfBufBytes;
  #pragma unroll
        for (int h = 0; h < MH; ++h) {
          const uint32_t* raw = reinterpret_cast<const uint32_t*>(buf + L::kRawA + h * 512);
          const uint4 v = make_uint4(raw[lane], raw[32 + lane], raw[64 + lane], raw[96 + lane]);
          *reinterpret_cast<uint4*>(buf + L::kCpA + h * 512 + lane * 16) = v;
        }
  #pragma unroll
        for (int c = 0; c < L::kSfbChunks; ++c) {
          const uint32_t* raw = reinterpret_cast<const uint32_t*>(buf + L::kRawB + c * 512);
          const uint4 v = make_uint4(raw[lane], raw[32 + lane], raw[64 + lane], raw[96 + lane]);
          *reinterpret_cast<uint4*>(buf + L::kCpB + c * 512 + lane * 16) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        // Copy the pack into the slot's TMEM columns from this warp (keeping the
        // copies out of the MMA issuer's instruction stream; measured 2-5%
        // faster) and signal the slot when they have completed.  The slot's
        // previous pack is no longer read: its MMAs completed (sfempty) before
        // this pack was loaded.
        if (lane == 0) {
          const uint32_t sft = tmem_base + (uint32_t)(P::kSfBase + slot * L::kSfCols);
  #pragma unroll
          for (int h = 0; h < MH; ++h)
            tc_cp_32x128b_warpx4(sft + 4 * h, smem_desc_sf_chunk(smem_u32(buf + L::kCpA + h * 512)));
  #pragma unroll
          for (int c = 0; c < L::kSfbChunks; ++c)
            tc_cp_32x128b_warpx4(sft + 4 * MH + 4 * c,
                                 smem_desc_sf_chunk(smem_u32(buf + L::kCpB + c * 512)));
          tc_commit(sfready(slot));
        }
        ++n_laid;
        lay.advance();
      }
      // Drain: scale loads issued but not laid out (abort path) land before exit,
      // and this warp's TMEM copies complete before TMEM can be freed.
      if (lane == 0) {
        for (uint32_t q = n_laid; q < n_loaded; ++q)
          wait_drain<EPI8>(sffull((int)(q % kSfSlots)), (q / kSfSlots) & 1u, tmo, err, kSiteProducerDrain);
        if (n_laid > 0)
          wait_drain<EPI8>(sfready((int)((n_laid - 1) % kSfSlots)), ((n_laid - 1) / kSfSlots) & 1u, tmo, err,
                     kSiteDrain);
      }
      __syncwarp();
    }
  } else if constexpr (EPI8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs) : "memory");
    // ------------------------------------------------------------ epilogue, eight warps
    // Warp w >= 4 drains lane quarter (w & 3) of 128-row half (w - 4) / 4:
    // the lane's whole row of BN columns is read from TMEM, C (fetched
    // before the accumulator is ready) added and the sum rounded to BF16 in
    // registers; TMEM goes back to the MMA as soon as all eight warps have
    // read their rows, and only then are the chunks staged and TMA-stored.
    if constexpr (MODE == kKGrouped) {
      // K-grouped 128 x 256 FP32 tiles: warp w drains lane quarter (w & 3),
      // columns [(w - 4) / 4 * 128, +128): four TMEM loads into 128 registers,
      // TMEM goes back to the MMA, then the columns (+ C) are stored, each
      // 16 x 32 box through the warp's staging chunk.  A quarter whose rows
      // cross M (into the next expert's rows) is stored row by row.
      if (warp >= 4) {
        const int quarter = warp & 3;
        const int chalf = (warp - 4) >> 2;
        uint8_t* ebuf = epi_smem + (warp - 4) * kEpiBuf;
        const uint32_t my_row_off = (uint32_t)lane * 64u;
        const uint32_t my_swz = ((uint32_t)lane >> 1) & 3u;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int it = 0;; ++it) {
          Tile tile;
          int tkb0, tkb1;
          const int st_it = sched.item(it, tile, tkb0, tkb1);
          if (st_it < 0) break;
          if (st_it == 0) continue;
          const int row0 = tile.mb * kBlockM + quarter * 32;
          const int row = row0 + lane;
          const bool row_ok = row < args.m;
          const int64_t out_row0 = (int64_t)tile.g * args.m + row0;
          const bool k_empty = tkb0 >= tkb1;
          const int ncol0 = tile.nb * BN + chalf * 128;
          const bool live = row0 < args.m && ncol0 < args.n;
          DG_CHECK(err, tile.nb >= 0 && tile.nb * BN < args.n && tile.g >= 0 && tile.g < args.num_groups,
                   kSiteCheckStore);
          if (!warp_wait<kSuspendHintNs, EPI8>(tfull(acc), acc_phase, abort_flag, tmo, err, kSiteEpilogueTmemFull))
            break;
          tc_fence_after();
          uint32_t hv[4][32];
          if (live && !k_empty) {
            const uint32_t taddr =
                tmem_base + (uint32_t)(acc * BN + chalf * 128) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
            for (int c = 0; c < 4; ++c) tc_ld_32x32b_x32(taddr + c * 32, hv[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tc_wait_ld_regs(hv[c]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty(acc));
          if (++acc == NUM_ACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
          if (!live) continue;
          float* const drow32 = args.d_f32 + (out_row0 + lane) * args.n;
          const float* const crow32 = args.c_f32 ? args.c_f32 + (out_row0 + lane) * args.n : nullptr;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col0 = ncol0 + c * 32;
            if (col0 >= args.n) break;
            if (row0 + 32 <= args.m) {
              uint32_t(&f)[32] = hv[c];  // FP32 bits, + C in place
              if (k_empty) {
#pragma unroll
                for (int i = 0; i < 32; ++i) f[i] = 0u;
              }
              if (crow32) {
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                  if (col0 + 4 * p < args.n) {
                    const float4 c4 = *reinterpret_cast<const float4*>(crow32 + col0 + 4 * p);
                    f[4 * p] = __float_as_uint(__uint_as_float(f[4 * p]) + c4.x);
                    f[4 * p + 1] = __float_as_uint(__uint_as_float(f[4 * p + 1]) + c4.y);
                    f[4 * p + 2] = __float_as_uint(__uint_as_float(f[4 * p + 2]) + c4.z);
                    f[4 * p + 3] = __float_as_uint(__uint_as_float(f[4 * p + 3]) + c4.w);
                  }
                }
              }
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if (col0 + 16 * h >= args.n) break;
                if (lane == 0) bulk_wait_group_read<0>();  // the staging chunk's previous store has read it
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  *reinterpret_cast<uint4*>(ebuf + my_row_off + 16u * ((uint32_t)j ^ my_swz)) =
                      make_uint4(f[16 * h + 4 * j], f[16 * h + 4 * j + 1], f[16 * h + 4 * j + 2],
                                 f[16 * h + 4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store_2d(&tm_d, smem_u32(ebuf), col0 + 16 * h, (int32_t)out_row0);
                  bulk_commit_group();
                }
              }
            } else if (row_ok) {
              store_row_chunk_f32(hv[c], drow32 + col0, crow32 ? crow32 + col0 : nullptr, args.n - col0,
                                  k_empty);
            }
          }
        }
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
      }
    } else {
      if (warp >= 4) {
        const int quarter = warp & 3;
        const int hh = (warp - 4) >> 2;
        uint8_t* ebuf = epi_smem + (warp - 4) * kEpiBuf;  // one staging chunk per warp
        constexpr int NCH = BN / 32;
        uint32_t pk[NCH][16];
        int acc = 0;
        uint32_t acc_phase = 0;
        // 32 columns of C of one row (this lane's) as BF16 pairs, 0 past M or N
        auto load_c = [&](uint32_t(&dst)[16], int crow, int col0) { load_c_row32(dst, args, crow, col0); };
        int c_ready_it = -1;  // the item whose C pk already holds (fetched during the stores before it)
        for (int it = 0;; ++it) {
          Tile tile;
          int tkb0, tkb1;
          const int st_it = sched.item(it, tile, tkb0, tkb1);
          if (st_it < 0) break;
          if (st_it == 0) continue;
          const int row0 = tile.mb * BM + hh * kBlockM + quarter * 32;
          const int row = row0 + lane;
          const bool part = SK && tile.kind == kItemPart;  // stream-K: a partial sum for another CTA
          // the tile's columns start inside N on an 8-column boundary; a
          // stream-K CTA's slot and flags lie inside the workspace (1024 CTAs
          // at most) and its K blocks inside the tile's
          DG_CHECK(err, tile.nb >= 0 && tile.nb * BN < args.n && ((tile.nb * BN) & 7) == 0 && tile.mb >= 0,
                   kSiteCheckStore);
          if constexpr (SK)
            DG_CHECK(err, gridDim.x <= 1024u && tkb0 >= 0 && tkb0 < tkb1 && tkb1 <= args.k_blocks,
                     kSiteCheckStreamK);
          // stream-K slot of CTA c for this warp's rows: 32 lanes x BN columns,
          // 16 bytes (4 columns) of a lane at ((col / 4) * 32 + lane) * 4 floats
          auto slot = [&](int c) {
            return args.sk_part + (size_t)c * (size_t)(2 * 4 * BN * 32) + (size_t)(hh * 4 + quarter) * (BN * 32);
          };
          uint32_t* const my_flags = args.sk_flags;  // [grid][8]
          if (args.c != nullptr && !part && c_ready_it != it) {
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) load_c(pk[ch], row, tile.nb * BN + ch * 32);
          }
          if (!warp_wait<kSuspendHintNs, EPI8>(tfull(acc), acc_phase, abort_flag, tmo, err, kSiteEpilogueTmemFull)) break;
          tc_fence_after();
          const bool live = row0 < args.m;
          if constexpr (SK) if (part) {
            // contributor: the FP32 partial goes to this CTA's slot as is
            if (live) {
              const uint32_t taddr =
                  tmem_base + (uint32_t)((acc * MH + hh) * BN) + ((uint32_t)(quarter * 32) << 16);
              float* dst = slot(blockIdx.x);
              uint32_t va[32], vb[32];
              tc_ld_32x32b_x32(taddr, va);
#pragma unroll
              for (int ch = 0; ch < NCH; ++ch) {
                uint32_t(&cur)[32] = (ch & 1) ? vb : va;
                uint32_t(&nxt)[32] = (ch & 1) ? va : vb;
                tc_wait_ld_regs(cur);
                if (ch + 1 < NCH) tc_ld_32x32b_x32(taddr + (ch + 1) * 32, nxt);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  *reinterpret_cast<float4*>(dst + ((ch * 8 + j) * 32 + lane) * 4) =
                      make_float4(__uint_as_float(cur[4 * j]), __uint_as_float(cur[4 * j + 1]),
                                  __uint_as_float(cur[4 * j + 2]), __uint_as_float(cur[4 * j + 3]));
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
            if (live) {
              // every lane's stores are ordered before the flag the owner acquires
              __threadfence();
              __syncwarp();
              if (lane == 0) st_release_gpu(my_flags + blockIdx.x * 8 + (warp - 4), 1u);
            }
            if (++acc == NUM_ACC) {
              acc = 0;
              acc_phase ^= 1u;
            }
            continue;
          }
          // owner: the CTAs holding the tile's later K blocks (each a
          // contiguous share of stream-K units starting inside the tile)
          int c_end = (int)blockIdx.x + 1;
          if constexpr (SK) if (tile.kind == kItemOwner && live) {
            const uint32_t tend = (uint32_t)(tile.sk + 1) * (uint32_t)args.k_blocks;
            bool ok = true;
            for (; c_end < (int)gridDim.x; ++c_end) {
              uint32_t lo, hi;
              sched.sk_range(c_end, lo, hi);
              if (lo >= tend) break;
              int got = 1;
              if (lane == 0 && lo < hi)
                got = wait_flag_gpu(my_flags + c_end * 8 + (warp - 4), abort_flag, tmo, err,
                                    kSiteStreamKPartial) ? 1 : 0;
              if (!__shfl_sync(0xffffffffu, got, 0)) {
                ok = false;
                break;
              }
            }
            if (!ok) break;
            __threadfence();  // acquire side: the partials are read after the flags
          }
          if (live) {
            const uint32_t taddr =
                tmem_base + (uint32_t)((acc * MH + hh) * BN) + ((uint32_t)(quarter * 32) << 16);
            uint32_t va[32], vb[32];
            tc_ld_32x32b_x32(taddr, va);
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              uint32_t(&cur)[32] = (ch & 1) ? vb : va;
              uint32_t(&nxt)[32] = (ch & 1) ? va : vb;
              tc_wait_ld_regs(cur);
              // owner: the contributors' partials of these 32 columns, in K
              // order (added before the next TMEM load is issued, so their
              // registers and that load's are never live together)
              if constexpr (SK) for (int c = (int)blockIdx.x + 1; c < c_end; ++c) {
                const float* src = slot(c);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 w = __ldcg(reinterpret_cast<const float4*>(src + ((ch * 8 + j) * 32 + lane) * 4));
                  cur[4 * j] = __float_as_uint(__uint_as_float(cur[4 * j]) + w.x);
                  cur[4 * j + 1] = __float_as_uint(__uint_as_float(cur[4 * j + 1]) + w.y);
                  cur[4 * j + 2] = __float_as_uint(__uint_as_float(cur[4 * j + 2]) + w.z);
                  cur[4 * j + 3] = __float_as_uint(__uint_as_float(cur[4 * j + 3]) + w.w);
                }
              }
              if (ch + 1 < NCH) tc_ld_32x32b_x32(taddr + (ch + 1) * 32, nxt);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float lo = __uint_as_float(cur[2 * i]), hi = __uint_as_float(cur[2 * i + 1]);
                if (args.c) {
                  lo += __uint_as_float(pk[ch][i] << 16);
                  hi += __uint_as_float(pk[ch][i] & 0xFFFF0000u);
                }
                pk[ch][i] = pack_bf16x2(lo, hi);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty(acc));
          // The next item's C is fetched chunk by chunk into the registers
          // each chunk of this tile leaves once staged, so its loads run
          // under the next tile's MMAs instead of after this tile's stores.
          Tile nt;
          int nit = it + 1, nkb0, nkb1, nst = -1;
          if (args.c != nullptr)
            for (;; ++nit)
              if ((nst = sched.item(nit, nt, nkb0, nkb1)) != 0) break;
          const bool prefetch = nst > 0 && !(SK && nt.kind == kItemPart);
          const int nrow = prefetch ? nt.mb * BM + hh * kBlockM + quarter * 32 + lane : 0;
          if (live) {
            // the contributors' flags go back to zero for the next launch
            if constexpr (SK)
              if (lane == 0)
                for (int c = (int)blockIdx.x + 1; c < c_end; ++c) st_relaxed_gpu(my_flags + c * 8 + (warp - 4), 0u);
          }
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            const int col0 = tile.nb * BN + ch * 32;
            if (live && col0 < args.n) {
              if (lane == 0) bulk_wait_group_read<0>();  // the staging chunk's previous store has read it
              __syncwarp();
              emit_packed_tma(pk[ch], ebuf, &tm_d, col0, row0, lane);
            }
            if (prefetch) load_c(pk[ch], nrow, nt.nb * BN + ch * 32);
          }
          if (prefetch) c_ready_it = nit;
          if (++acc == NUM_ACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    // staging: 16-byte piece j of chunk row r at r * 64 + 16 * (j ^ ((r >> 1) & 3)),
    // the layout of CU_TENSOR_MAP_SWIZZLE_64B
    uint8_t* ebuf = epi_smem + (warp - 3) * 2 * kEpiBuf;
    uint32_t nchunk = 0;  // chunks staged so far (buffer = nchunk & 1)
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t n_xchg = 0;  // split-K exchanges of this quarter so far (barrier phases)
    // C of the tile being drained (see below); with 128 x 256 dense tiles
    // (one accumulator) the next tile's C is fetched into these registers
    // chunk by chunk as this tile's chunks are staged, so it lands under the
    // next tile's MMAs.  (With two accumulators the MMA already runs a tile
    // ahead; fetching the next C during the stores there measured slower:
    // 128 x 224 with C on N = 24576, K = 1536, 151 -> 182 us.)
    constexpr bool kRegHeld = MH == 2 || (NUM_ACC == 1 && MODE != kKGrouped && KSPLIT == 1);
    constexpr int kPreHalves = (MODE == kDense && MH == 2 && BN == 192) ? 2 : 1;
    uint4 cpre[BN / 32][4];
    uint32_t cpk[kPreHalves][BN / 32][16];
    int c_ready_it = -1;  // the item whose C is already in cpre / cpk
    for (int it = 0;; ++it) {
      Tile tile;
      int tkb0, tkb1;
      const int st_it = sched.item(it, tile, tkb0, tkb1);
      if (st_it < 0) break;
      if (st_it == 0) continue;
      // C of dense tiles is fetched while the accumulator is still being
      // computed, so the epilogue never waits for a load from HBM.  128-row
      // tiles with two accumulators (no split): this quarter's whole C tile,
      // coalesced (BN / 32 chunks, 16 registers each).  Register-held
      // epilogues (one accumulator): this lane's row of C as BF16 pairs, for
      // the first 128-row half (both halves of a 256 x 192 tile); the
      // epilogue adds the accumulator in place.
      const bool c_ahead =
          is_dense_mode(MODE) && MH == 1 && KSPLIT == 1 && NUM_ACC == 2 && args.c != nullptr;
      if (c_ahead && c_ready_it != it) {
        const int crow0 = tile.mb * BM + quarter * 32;
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch) load_c_chunk(cpre[ch], args, tile.nb * BN + ch * 32, crow0, crow0, lane);
      }
      // the next item, whose C the 128 x 256 dense epilogue fetches during
      // this tile's stores (into cpk[0][ch] once chunk ch is staged)
      const bool c_next = is_dense_mode(MODE) && MH == 1 && KSPLIT == 1 && args.c != nullptr && kRegHeld;
      Tile nt;
      int nit = it + 1, nst = -1;
      if (c_next) {
        int nkb0, nkb1;
        for (;; ++nit)
          if ((nst = sched.item(nit, nt, nkb0, nkb1)) != 0) break;
      }
      const bool prefetch = c_next && nst > 0;
      const int nrow0 = prefetch ? nt.mb * BM + quarter * 32 : 0;
      auto prefetch_c = [&](int ch) {
        if (!prefetch) return;
        load_c_row32(cpk[0][ch], args, nrow0 + lane, nt.nb * BN + ch * 32);
      };
      if (kRegHeld && is_dense_mode(MODE) && args.c != nullptr && c_ready_it != it) {
#pragma unroll
        for (int hh = 0; hh < kPreHalves; ++hh) {
          const int crow = tile.mb * BM + hh * kBlockM + quarter * 32 + lane;
#pragma unroll
          for (int ch = 0; ch < BN / 32; ++ch) load_c_row32(cpk[hh][ch], args, crow, tile.nb * BN + ch * 32);
        }
      }
      if (!warp_wait<kSuspendHintNs, EPI8>(tfull(acc), acc_phase, abort_flag, tmo, err, kSiteEpilogueTmemFull)) break;
      tc_fence_after();
      bool stop = false;
      bool both_halves = false;  // the first half's pass stored both (256 x 192 dense)
      // the tile's 128-row halves in turn; TMEM goes back after the last one
      for (int h = 0; h < MH; ++h) {
        if (both_halves) break;
        const bool last_half = h == MH - 1;
        // contiguous 256-row tiles: the halves are the pair's blocks; the
        // second half of a half-empty pair stores nothing
        constexpr bool kPairs = MODE == kContiguous && BM == 2 * kBlockM;
        const bool half_dead = kPairs && h == 1 && tile.b1 < 0;
        const int row0 = kPairs ? (h == 0 || half_dead ? tile.b0 : tile.b1) * kBlockM + quarter * 32
                                : tile.mb * BM + h * kBlockM + quarter * 32;
        const int row = row0 + lane;
        bool row_ok;
        int64_t out_row0;
        if (is_dense_mode(MODE)) {
          row_ok = row < args.m;
          out_row0 = row0;
        } else if (MODE == kContiguous) {
          const int gi = row < args.m ? __ldg(args.m_indices + row) : -1;
          row_ok = gi == tile.g;
          if (gi >= 0 && gi != tile.g) record_error(err, DG_ERR_DEVICE_BAD_INDEX, kSiteContiguousIndex);
          out_row0 = row0;
        } else if (MODE == kKGrouped) {
          row_ok = row < args.m;
          out_row0 = (int64_t)tile.g * args.m + row0;
        } else {
          row_ok = row < group_valid[tile.g];
          out_row0 = (int64_t)tile.g * args.m + row0;
        }
        if constexpr (DG_DEBUG_CHECKS) {
          // rows written lie inside D (G x M rows when grouped); the tile's
          // columns start inside N on an 8-column boundary
          const int64_t rows = (MODE == kMasked || MODE == kKGrouped) ? (int64_t)args.num_groups * args.m
                                                                      : (int64_t)args.m;
          const bool ok = tile.nb >= 0 && tile.nb * BN < args.n && ((tile.nb * BN) & 7) == 0 &&
                          (!row_ok || (out_row0 + lane >= 0 && out_row0 + lane < rows));
          if (!ok) {
            DG_CHECK(err, false, kSiteCheckStore);
            row_ok = false;
          }
        }
        // The TMA store clips at M and N, so dense quarters always use it; a
        // grouped quarter uses it only when every one of its rows is written.
        const bool use_tma = is_dense_mode(MODE)   ? true
                             : (MODE == kKGrouped) ? false
                                                   : (__all_sync(0xffffffffu, row_ok) != 0);
        __nv_bfloat16* drow = args.d + (out_row0 + lane) * args.ldd;
        const __nv_bfloat16* crow = args.c ? args.c + (out_row0 + lane) * args.ldc : nullptr;
        // K-grouped: FP32 rows of D[g] / C[g]; a tile without K blocks writes C (or 0)
        float* drow32 = MODE == kKGrouped ? args.d_f32 + (out_row0 + lane) * args.n : nullptr;
        const float* crow32 =
            (MODE == kKGrouped && args.c_f32) ? args.c_f32 + (out_row0 + lane) * args.n : nullptr;
        const bool k_empty = MODE == kKGrouped && tkb0 >= tkb1;
        // A quarter none of whose rows is written hands its accumulator back
        // unread: no TMEM load, no exchange, no store.  For dense and K-grouped
        // tiles the test (first row past M) is the same in every CTA of a
        // split-K cluster, so all of them skip the same quarters.
        const bool quarter_live = (is_dense_mode(MODE) || MODE == kKGrouped)
                                      ? row0 < args.m
                                      : (__any_sync(0xffffffffu, row_ok) != 0 && !half_dead);
        if (!quarter_live) {
          if (last_half) {
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
          }
#pragma unroll
          for (int ch = 0; ch < BN / 32; ++ch) prefetch_c(ch);
          continue;
        }
        const uint32_t taddr =
            tmem_base + (uint32_t)((acc * MH + h) * BN) + ((uint32_t)(quarter * 32) << 16);
        constexpr int NCH = BN / 32;
        if constexpr (KSPLIT > 1) {
          // Split-K exchange (dense tiles only).  Every CTA owns one column
          // slice of this quarter: it sends the other slices of its partial to
          // their owners, then adds the partials of its own slice in CTA-rank
          // order (the same result whatever the timing) and stores them.
          constexpr int SCH = P::kSlice / 32;  // chunks per slice
          const uint32_t kpar = n_xchg & 1u;
          const int ncol0 = tile.nb * BN;
          // every owner has read what this warp sent it for the previous tile
          if (n_xchg > 0 &&
              !warp_wait_cluster(recv_free(quarter), kpar ^ 1u, abort_flag, tmo, err, kSiteSplitFree)) {
            stop = true;
            break;
          }
          // chunks sent to other CTAs; the next one's TMEM load overlaps the
          // current one's remote stores (conditions are warp-uniform)
          auto sent = [&](int ch) { return ch / SCH != (int)krank && ncol0 + ch * 32 < args.n; };
          uint32_t va[32], vb[32];
          if (sent(0)) tc_ld_32x32b_x32(taddr, va);
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            uint32_t(&cur)[32] = (ch & 1) ? vb : va;
            uint32_t(&nxt)[32] = (ch & 1) ? va : vb;
            const bool here = sent(ch);
            if (here) tc_wait_ld_regs(cur);
            if (ch + 1 < NCH && sent(ch + 1)) tc_ld_32x32b_x32(taddr + (ch + 1) * 32, nxt);
            if (!here) continue;
            const int o = ch / SCH;
            const int sslot = (int)krank < o ? (int)krank : (int)krank - 1;
            const uint32_t dst = mapa_shared(
                smem_u32(recv + (quarter * (KSPLIT - 1) + sslot) * P::kXSlot + (ch % SCH) * 4096 + lane * 16),
                (uint32_t)o);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st_shared_cluster_v4(dst + j * 512, cur[4 * j], cur[4 * j + 1], cur[4 * j + 2], cur[4 * j + 3]);
          }
          __syncwarp();
          if (lane == 0)
            for (int o = 0; o < KSPLIT; ++o)
              if (o != (int)krank) mbar_arrive_cluster(mapa_shared(recv_full(quarter), (uint32_t)o));
          // the first chunk of the own slice is read from TMEM while waiting
          if (ncol0 + (int)krank * P::kSlice < args.n) tc_ld_32x32b_x32(taddr + (int)krank * P::kSlice, va);
          if (!warp_wait_cluster(recv_full(quarter), kpar, abort_flag, tmo, err, kSiteSplitFull)) {
            stop = true;
            break;
          }
#pragma unroll
          for (int c = 0; c < SCH; ++c) {
            const int ch = (int)krank * SCH + c;
            const int col0 = ncol0 + ch * 32;
            if (col0 >= args.n) break;
            uint32_t(&v)[32] = va;
            if (c > 0) tc_ld_32x32b_x32(taddr + ch * 32, v);
            tc_wait_ld_regs(v);
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = 0.0f;
#pragma unroll
            for (int rr = 0; rr < KSPLIT; ++rr) {
              if (rr == (int)krank) {
#pragma unroll
                for (int i = 0; i < 32; ++i) f[i] += __uint_as_float(v[i]);
              } else {
                const int sslot = rr < (int)krank ? rr : rr - 1;
                const uint8_t* src = recv + (quarter * (KSPLIT - 1) + sslot) * P::kXSlot + c * 4096 + lane * 16;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 w = *reinterpret_cast<const float4*>(src + j * 512);
                  f[4 * j] += w.x;
                  f[4 * j + 1] += w.y;
                  f[4 * j + 2] += w.z;
                  f[4 * j + 3] += w.w;
                }
              }
            }
            uint8_t* buf = ebuf + (nchunk & 1u) * kEpiBuf;
            if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
            __syncwarp();
            emit_chunk_tma(f, buf, &tm_d, args, col0, out_row0, row0, true, lane);
            ++nchunk;
          }
          // all of this accumulator's columns have been read; the received
          // partials have been consumed.  After the CTA's last tile nobody
          // waits for the buffers again (a remote release-arrive costs ~0.5 us).
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(tempty(acc));
            if (sched.has_next(it))
              for (int o = 0; o < KSPLIT; ++o)
                if (o != (int)krank) mbar_arrive_cluster(mapa_shared(recv_free(quarter), (uint32_t)o));
          }
          ++n_xchg;
          continue;
        }
        if constexpr (MODE == kDense && MH == 2 && NCH == 6) {
          // 256 x 192 dense tile: both halves (2 x 96 words of BF16 pairs,
          // + C) are read into registers before any store, so TMEM goes back
          // to the MMA after 12 TMEM loads rather than after half the stores
          const int row0b = row0 + kBlockM;
          // C of both halves is already in cpk (fetched before the wait)
          uint32_t(&pa)[NCH][16] = cpk[0];
          uint32_t(&pb)[NCH][16] = cpk[kPreHalves - 1];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              uint32_t v[32];
              tc_ld_32x32b_x32(taddr + hh * BN + ch * 32, v);
              tc_wait_ld_regs(v);
              uint32_t(&pk)[16] = hh ? pb[ch] : pa[ch];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float lo = __uint_as_float(v[2 * i]), hi = __uint_as_float(v[2 * i + 1]);
                if (args.c) {
                  lo += __uint_as_float(pk[i] << 16);
                  hi += __uint_as_float(pk[i] & 0xFFFF0000u);
                }
                pk[i] = pack_bf16x2(lo, hi);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty(acc));
          both_halves = true;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (hh == 1 && row0b >= args.m) break;
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              const int col0 = tile.nb * BN + ch * 32;
              if (col0 >= args.n) continue;
              uint8_t* buf = ebuf + (nchunk & 1u) * kEpiBuf;
              if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
              __syncwarp();
              emit_packed_tma(hh ? pb[ch] : pa[ch], buf, &tm_d, col0, out_row0 + hh * kBlockM, lane);
              ++nchunk;
            }
          }
          continue;
        }
        if constexpr (MH == 2 || (NUM_ACC == 1 && MODE != kKGrouped && KSPLIT == 1)) {
          {
            // A single accumulator (256-row tiles, or 256 columns): the whole
            // half (the whole row of 256 columns) is read from TMEM, C added
            // and the sum rounded to BF16 in registers first, so TMEM goes
            // back to the MMA before the (second half's) stores instead of
            // after.  pk first holds this lane's row of C: the first half's
            // was fetched before the wait; the second half's chunk c is
            // fetched into pk[c] as soon as the first half's chunk c has been
            // staged for its store (dense 256-row tiles).
            uint32_t(&pk)[NCH][16] = cpk[0];
            if (args.c && h > 0 && !(is_dense_mode(MODE) && MH == 2)) {
#pragma unroll
              for (int ch = 0; ch < NCH; ++ch) {
                const int col0 = tile.nb * BN + ch * 32;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  uint4 v = make_uint4(0u, 0u, 0u, 0u);
                  if (row_ok && col0 + 8 * q < args.n) v = __ldg(reinterpret_cast<const uint4*>(crow + col0 + 8 * q));
                  pk[ch][4 * q] = v.x;
                  pk[ch][4 * q + 1] = v.y;
                  pk[ch][4 * q + 2] = v.z;
                  pk[ch][4 * q + 3] = v.w;
                }
              }
            }
            uint32_t va[32], vb[32];
            tc_ld_32x32b_x32(taddr, va);
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              uint32_t(&cur)[32] = (ch & 1) ? vb : va;
              uint32_t(&nxt)[32] = (ch & 1) ? va : vb;
              tc_wait_ld_regs(cur);
              if (ch + 1 < NCH) tc_ld_32x32b_x32(taddr + (ch + 1) * 32, nxt);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float lo = __uint_as_float(cur[2 * i]), hi = __uint_as_float(cur[2 * i + 1]);
                if (args.c) {
                  lo += __uint_as_float(pk[ch][i] << 16);
                  hi += __uint_as_float(pk[ch][i] & 0xFFFF0000u);
                }
                pk[ch][i] = pack_bf16x2(lo, hi);
              }
            }
            if (last_half) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(tempty(acc));
            }
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              const int col0 = tile.nb * BN + ch * 32;
              if (col0 >= args.n) {
                prefetch_c(ch);
                continue;
              }
              if (!use_tma) {
                // a contiguous quarter with rows of other groups or padding
                if (row_ok) store_packed_row(pk[ch], drow + col0, args.n - col0);
                continue;
              }
              uint8_t* buf = ebuf + (nchunk & 1u) * kEpiBuf;
              if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
              __syncwarp();
              emit_packed_tma(pk[ch], buf, &tm_d, col0, out_row0, lane);
              ++nchunk;
              prefetch_c(ch);
              if (is_dense_mode(MODE) && MH == 2 && h == 0 && args.c) {
                // the second half's C of these columns, into the registers just staged
                const int row1 = row + kBlockM;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  uint4 v = make_uint4(0u, 0u, 0u, 0u);
                  if (row1 < args.m && col0 + 8 * q < args.n)
                    v = __ldg(reinterpret_cast<const uint4*>(args.c + (int64_t)row1 * args.ldc + col0 + 8 * q));
                  pk[ch][4 * q] = v.x;
                  pk[ch][4 * q + 1] = v.y;
                  pk[ch][4 * q + 2] = v.z;
                  pk[ch][4 * q + 3] = v.w;
                }
              }
            }
            continue;
          }
        }
        // K-grouped: FP32 rows of D[g] (+ C[g]).  A quarter whose 32 rows all
        // lie inside M goes through the TMA store; one that crosses M (into
        // the next expert's rows) does not.
        auto kgrouped_chunk = [&](const uint32_t(&cur)[32], int col0) {
          if (row0 + 32 <= args.m) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = k_empty ? 0.0f : __uint_as_float(cur[i]);
            if (crow32) {
#pragma unroll
              for (int p = 0; p < 8; ++p) {
                if (col0 + 4 * p < args.n) {
                  const float4 c4 = *reinterpret_cast<const float4*>(crow32 + col0 + 4 * p);
                  f[4 * p] += c4.x;
                  f[4 * p + 1] += c4.y;
                  f[4 * p + 2] += c4.z;
                  f[4 * p + 3] += c4.w;
                }
              }
            }
            emit_chunk_tma_f32(f, ebuf, nchunk, &tm_d, col0, args.n, out_row0, lane);
          } else if (row_ok) {
            store_row_chunk_f32(cur, drow32 + col0, crow32 ? crow32 + col0 : nullptr, args.n - col0,
                                k_empty);
          }
        };
        if constexpr (MODE == kKGrouped && NUM_ACC == 1 && NCH == 8) {
          // single 256-column accumulator: each 128-column half is read from
          // TMEM in full before it is stored, so TMEM goes back to the MMA
          // once the second half is read rather than once it is stored
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t hv[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc_ld_32x32b_x32(taddr + (hh * 4 + c) * 32, hv[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tc_wait_ld_regs(hv[c]);
            if (hh == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(tempty(acc));
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int col0 = tile.nb * BN + (hh * 4 + c) * 32;
              if (col0 < args.n) kgrouped_chunk(hv[c], col0);
            }
          }
          continue;
        }
        uint32_t ra[32], rb[32];
        tc_ld_32x32b_x32(taddr, ra);
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          uint32_t(&cur)[32] = (ch & 1) ? rb : ra;
          uint32_t(&nxt)[32] = (ch & 1) ? ra : rb;
          tc_wait_ld_regs(cur);
          if (ch + 1 < NCH) {
            tc_ld_32x32b_x32(taddr + (ch + 1) * 32, nxt);
          } else if (last_half) {
            // every column of this accumulator is in registers: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
          }
          const int col0 = tile.nb * BN + ch * 32;
          if (col0 >= args.n) {
            prefetch_c(ch);
            continue;
          }
          if (MODE == kKGrouped) {
            kgrouped_chunk(cur, col0);
            continue;
          }
          if (use_tma) {
            uint8_t* buf = ebuf + (nchunk & 1u) * kEpiBuf;
            if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
            __syncwarp();
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(cur[i]);
            if (c_ahead) emit_chunk_tma_c(f, cpre[ch], buf, &tm_d, col0, out_row0, lane);
            else emit_chunk_tma(f, buf, &tm_d, args, col0, out_row0, row0, is_dense_mode(MODE), lane);
            ++nchunk;
            prefetch_c(ch);
          } else if (row_ok) {
            store_row_chunk(cur, drow + col0, crow ? crow + col0 : nullptr, args.n - col0);
          }
        }
      }  // halves
      if (stop) break;
      if (prefetch) c_ready_it = nit;
      if (++acc == NUM_ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // every TMA store issued here has read its staging buffer before the CTA
    // exits (the writes themselves complete before the grid does)
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }

  __syncthreads();
  // No CTA leaves while others may still reach its shared memory.
  if constexpr (CL > 1) {
    // Clean path: every exchange into this CTA has completed (its mbarrier
    // waits acquired it: split-K partials, and with multicast pairs the
    // peer's halves of B), and the peer's MMA commits that arrive on this
    // CTA's barriers completed before the peer's MMA thread finished its
    // drain, so the barrier needs no release (a release would also wait for
    // this CTA's outstanding global writes).  After an abort
    // that no longer holds: a CTA that gave up on a wait never acquired what
    // its peers sent it, and their remote stores and arrivals may still be in
    // flight.  An aborted CTA therefore marks every peer before the barrier
    // (its fence orders those marks and its own remote stores before the
    // arrival; the waits acquire them), so that every CTA of the cluster sees
    // the abort and all of them take a second, release/acquire barrier, which
    // orders every thread's remote accesses before any CTA exits.  abort_flag
    // is final here (only the roles above raise it), so the choice is the same
    // in every CTA.
    if (*abort_flag) {
      if (threadIdx.x == 0)
        for (uint32_t r = 0; r < (uint32_t)CL; ++r)
          if (r != krank) st_shared_cluster_u32(mapa_shared(smem_u32((const void*)peer_abort), r), 1u);
      fence_acq_rel_cluster();
    }
    cluster_arrive_relaxed_wait_acquire();
    if (*abort_flag || *peer_abort) cluster_sync_all();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Raises the kernel's dynamic shared-memory limit once per device (host-side
// setup kept out of the launch path, e.g. of a CUDA-graph capture).  `Tag`
// makes one set of flags per kernel instantiation (kernels share a signature).
template <int BN, int STAGES, int MODE, int KSPLIT, int CTAS>
struct KernelTag {};

template <class Tag, class Kern>
static cudaError_t set_smem_once(Kern kern, size_t smem) {
  // host threads may launch concurrently: the flags are atomic (setting the
  // attribute twice is harmless)
  static std::atomic<bool> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return e;
}

template <int BN, int STAGES, int MODE, int KSPLIT = 1, int BM = kBlockM, bool EPI8 = false, bool SK = false,
          bool MC = false>
static cudaError_t gemm_launch_impl(const CUtensorMap& a, const CUtensorMap& b,
                                    const CUtensorMap& sfa, const CUtensorMap& sfb,
                                    const CUtensorMap& d, const GemmArgs& args, int grid,
                                    cudaStream_t stream) {
  using Plan = GemmPlan<BN, STAGES, KSPLIT, BM>;
  static_assert(Plan::smem_bytes(MODE) <= (size_t)kSmemLimit, "shared memory over the per-CTA limit");
  auto kern = fp8_gemm_kernel<BN, STAGES, MODE, KSPLIT, BM, EPI8, SK, MC>;
  const size_t smem = Plan::smem_bytes(MODE);
  constexpr int CL = MC ? 2 : KSPLIT;
  cudaError_t e = set_smem_once<
      KernelTag<BN, STAGES, MODE, KSPLIT, MC ? 7 : SK ? 6 : EPI8 ? 5 : (BM == kBlockM ? 1 : (BM > kBlockM ? 3 : 4))>>(
      kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[3];
  unsigned n_attr = 0;
  if (SK) {
    // stream-K owners wait for partial sums of other CTAs: all co-resident
    attr[n_attr].id = cudaLaunchAttributeCooperative;
    attr[n_attr].val.cooperative = 1;
    ++n_attr;
  }
  if (CL > 1) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = CL;
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
  cfg.blockDim = dim3(EPI8 ? kGemmThreadsEpi8 : kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  return cudaLaunchKernelEx(&cfg, kern, a, b, sfa, sfb, d, args);
}

// Largest number of co-resident KSPLIT-CTA clusters of a split-K configuration.
template <int BN, int STAGES, int KSPLIT>
static int gemm_splitk_max_clusters_impl() {
  auto kern = fp8_gemm_kernel<BN, STAGES, kDense, KSPLIT>;
  const size_t smem = GemmPlan<BN, STAGES, KSPLIT>::smem_bytes(kDense);
  if (set_smem_once<KernelTag<BN, STAGES, kDense, KSPLIT, 1>>(kern, smem) != cudaSuccess) return 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = KSPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(KSPLIT, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

template <int BN, int STAGES>
static cudaError_t gemm_launch_modes(int mode, const CUtensorMap& a, const CUtensorMap& b,
                                     const CUtensorMap& sfa, const CUtensorMap& sfb,
                                     const CUtensorMap& d, const GemmArgs& args, int grid,
                                     cudaStream_t stream) {
  switch (mode) {
    case kDense: return gemm_launch_impl<BN, STAGES, kDense>(a, b, sfa, sfb, d, args, grid, stream);
    case kContiguous: return gemm_launch_impl<BN, STAGES, kContiguous>(a, b, sfa, sfb, d, args, grid, stream);
    case kMasked: return gemm_launch_impl<BN, STAGES, kMasked>(a, b, sfa, sfb, d, args, grid, stream);
    // MN-major B tiles are whole 128-column boxes; the other layouts are
    // compiled at the widths 128 and 256 only
    case kKGrouped:
      if constexpr (BN % 128 == 0)
        return gemm_launch_impl<BN, STAGES, kKGrouped>(a, b, sfa, sfb, d, args, grid, stream);
      return cudaErrorInvalidValue;
    case kDenseNN:
      if constexpr (BN % 128 == 0)
        return gemm_launch_impl<BN, STAGES, kDenseNN>(a, b, sfa, sfb, d, args, grid, stream);
      return cudaErrorInvalidValue;
    case kDenseTN:
      if constexpr (BN % 128 == 0)
        return gemm_launch_impl<BN, STAGES, kDenseTN>(a, b, sfa, sfb, d, args, grid, stream);
      return cudaErrorInvalidValue;
    case kDenseTT:
      if constexpr (BN % 128 == 0)
        return gemm_launch_impl<BN, STAGES, kDenseTT>(a, b, sfa, sfb, d, args, grid, stream);
      return cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

}  // namespace dg

// Defines the launch entry of one tile width (one translation unit each).
#define DG_DEFINE_GEMM_BN(BN, STAGES)                                                        \
  namespace dg {                                                                           \
  cudaError_t gemm_launch_bn##BN(int mode, const CUtensorMap& a, const CUtensorMap& b,     \
                                 const CUtensorMap& sfa, const CUtensorMap& sfb,           \
                                 const CUtensorMap& d, const GemmArgs& args, int grid,     \
                                 cudaStream_t stream) {                                    \
    return gemm_launch_modes<BN, STAGES>(mode, a, b, sfa, sfb, d, args, grid, stream);     \
  }                                                                                        \
  int gemm_stages_bn##BN() { return STAGES; }                                              \
  }
