/*
 * dg.h - C ABI of libdg.so: FP8 GEMM with fine-grained scaling for NVIDIA
 * GB300 (sm_103a), in the dense NT form and the two M-grouped MoE layouts.
 *
 * Operation (all GEMM entry points):   D = C + A @ B.T
 *   "DeepGEMM: kernels GEMM FP8 limpos e eficientes por meio de scaling
 *   granular" (pt.news.hada.io), section "Interface GEMM e restrições de
 *   layout": the naming convention D = C + A @ B with NT as the reference
 *   layout, fp8_gemm_nt computing D = C + A @ B.T.
 *   A is E4M3 [M, K] with one scale per 1x128 row group, B is E4M3 [N, K]
 *   (K-major, i.e. row-major [N, K]) with one scale per 128x128 block,
 *   accumulation is FP32 and D (and the optional C) is BF16.
 *
 * Scale factors.  The GEMMs take the packed UE8M0 layout the same section
 * gives for SM100: four 8-bit exponents per 32-bit word, transposed
 * ("MN-major") and TMA-aligned:
 *   sf[j, r] (int32, [ceil(K/512), align(MN, 4)]) holds in byte t (least
 *   significant first) the biased exponent e + 127 of K block 4j + t for
 *   row r; the scale is 2^e.  For B the 128x128 block exponent is repeated on
 *   each of the block's 128 rows.  Rows in [MN, align(MN, 4)) and bytes past
 *   the last K block are ignored.  Grouped tensors add a leading group
 *   dimension: [G, ceil(K/512), align(MN, 4)].
 *   dg_transform_sf converts plain FP32 scales (the SM90 format of the same
 *   section) into this layout; dg_quantize_fp8 writes either format.
 *
 * Common conventions.
 *   - Every pointer argument that names tensor data is a DEVICE pointer on
 *     the current CUDA device unless stated otherwise; `stream` is a
 *     cudaStream_t (NULL = legacy default stream).  The caller owns all memory
 *     and the stream.  The library never allocates device memory, never
 *     synchronises the stream (except dg_get_device_error) and keeps no
 *     pointer after a call returns.  Work is enqueued asynchronously.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     failed check returns its status and enqueues nothing.  Checks: non-null
 *     pointers for non-empty tensors, K % 128 == 0, 16-byte aligned data
 *     pointers and row strides, N % 8 == 0 (16-byte BF16 output rows), sizes
 *     within the 32-bit coordinate range of TMA, a device of compute
 *     capability 10.3.  An empty problem (M, N, m_sum or num_groups equal to
 *     0) is a no-op returning DG_OK.
 *   - Kernel launch failures return DG_ERR_CUDA.  Conditions found on the
 *     device (a bounded wait that ran out, a group index out of range, a scale
 *     that is not a power of two) never trap: the kernel records the first
 *     such condition in a device error word and completes; read it with
 *     dg_get_device_error.
 *   - Entry points may be called from several host threads; calls on the
 *     same stream execute in order.
 */
#ifndef DG_H_
#define DG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dg_status {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum value */
  DG_ERR_ALIGNMENT = 2,         /* K % 128, N % 8, pointer or stride alignment */
  DG_ERR_UNSUPPORTED_ARCH = 3,  /* current device is not compute capability 10.3 */
  DG_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed */
  DG_ERR_DEVICE_TIMEOUT = 5,    /* device: a pipeline wait exceeded its limit */
  DG_ERR_DEVICE_BAD_INDEX = 6,  /* device: m_indices >= num_groups, masked_m outside [0, max_m],
                                   or a contiguous 128-row block mixing experts */
  DG_ERR_TOO_LARGE = 7,         /* a size beyond the supported range */
  DG_ERR_DEVICE_BAD_SCALE = 8,  /* device: an FP32 scale that is not a positive power of two */
  DG_ERR_DEVICE_CHECK = 9       /* device: a bound checked by the debug library failed */
} dg_status;

typedef enum dg_sf_format {
  DG_SF_FP32 = 0,         /* float, [G, ceil(MN/block_rows), K/128], K blocks innermost */
  DG_SF_UE8M0_PACKED = 1  /* int32, [G, ceil(K/512), align(MN, 4)], the layout described above */
} dg_sf_format;

/* ------------------------------------------------------------------------ */
/* GEMMs                                                                     */
/* ------------------------------------------------------------------------ */

/* Dense NT:  D[m, n] = C[m, n] + sum_k A[m, k] * B[n, k]  (dequantised).
 *   a    E4M3 [m, k], row stride lda elements (lda >= k, lda % 16 == 0)
 *   sfa  packed UE8M0 [ceil(k/512), align(m, 4)]  (1x128 row groups of A)
 *   b    E4M3 [n, k], row stride ldb (ldb >= k, ldb % 16 == 0)
 *   sfb  packed UE8M0 [ceil(k/512), align(n, 4)]  (128x128 blocks of B, per row)
 *   c    BF16 [m, n], row stride ldc (ldc % 8 == 0), or NULL for C = 0;
 *        c may equal d (in-place accumulate) when ldc == ldd
 *   d    BF16 [m, n], row stride ldd (ldd >= n, ldd % 8 == 0)
 * Cited: "DeepGEMM: kernels GEMM FP8 limpos e eficientes por meio de scaling
 * granular", sections "Interface GEMM e restrições de layout" and "GEMM denso
 * e grouped" (fp8_gemm_{nt, nn, tn, tt}; the other three layouts below). */
dg_status dg_fp8_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream);

/* Dense NT with a caller-provided workspace (scratch device memory), which
 * lets the call split the K blocks of the output tiles of its last waves
 * between SMs ("stream-K") when the tile count leaves the last wave mostly
 * empty, e.g. M = 4096, N = 2112, K = 7168 on 152 SMs.  Same operation,
 * arguments, layouts and checks as dg_fp8_gemm_nt, plus:
 *   workspace        device pointer, 16-byte aligned, or NULL (then the call
 *                    is exactly dg_fp8_gemm_nt)
 *   workspace_bytes  its size; when it is below
 *                    dg_fp8_gemm_nt_workspace_size for this problem the call
 *                    runs without stream-K (no error)
 * The workspace starts with 32 KiB of flags (one 32-bit word per SM and
 * epilogue warp, for up to 1024 SMs), which must be zero before the first
 * use; one FP32 partial-sum slot of 256 x block_n values per SM follows and
 * needs no initialisation.  Every launch leaves the flags zero
 * again, so the same buffer serves any number of later calls, also inside a
 * CUDA graph.
 * Calls that can overlap on the device (other streams, concurrent graphs)
 * need separate workspaces.  After a DG_ERR_DEVICE_TIMEOUT the flags may be
 * left set: zero the buffer again before reusing it.  Results are
 * deterministic (the partial sums of a tile are added in K order) but may
 * differ from dg_fp8_gemm_nt's in the last bit (another FP32 summation order).
 * Cited: the same pages as dg_fp8_gemm_nt for the operation; splitting K
 * between SMs to balance the last wave is this library's addition. */
dg_status dg_fp8_gemm_nt_ws(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                            const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                            int64_t ldb, int64_t ldc, int64_t ldd, void* workspace,
                            uint64_t workspace_bytes, void* stream);

/* dg_fp8_gemm_nt_ws for callers that cannot allocate device memory: a
 * runtime that reserves all its memory at start-up and forbids allocation
 * afterwards, a plugin whose host hands it no scratch buffer, or code that
 * must not call cudaMalloc because it would synchronise the device or is not
 * allowed where it runs.  The workspace is a 32 MiB array of this library in
 * device memory, present on every device from the moment libdg.so is loaded
 * until the process exits (whether or not this function is ever called).
 * Nothing is allocated or freed: no cudaMalloc, cudaFree or other allocating
 * routine is called.  Same operation, arguments, layouts and checks as
 * dg_fp8_gemm_nt; the tile plan is dg_fp8_gemm_nt_ws's for a 32 MiB
 * workspace.
 *   - A problem whose plan needs more scratch than the array holds (see
 *     dg_fp8_gemm_nt_workspace_size; e.g. stream-K with 224-column tiles on
 *     more than 145 SMs) is rejected with DG_ERR_TOO_LARGE before anything
 *     is enqueued; dg_fp8_gemm_nt needs no scratch at all.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one array and leaves its last
 *     contents in it; each call clears the part that must start at zero (the
 *     flags) on its stream before its kernel.  Calls whose execution can
 *     overlap on the device (other streams, other host threads) race on it:
 *     serialise them.
 * No counterpart on the pages: this entry point exists for callers of this
 * library that cannot provide a workspace. */
dg_status dg_fp8_gemm_nt_static_ws(const void* a, const int32_t* sfa, const void* b,
                                   const int32_t* sfb, const void* c, void* d, int64_t m,
                                   int64_t n, int64_t k, int64_t lda, int64_t ldb, int64_t ldc,
                                   int64_t ldd, void* stream);

/* Bytes of workspace dg_fp8_gemm_nt_ws needs to use stream-K for an
 * M x N x K problem (with C when has_c != 0) on num_sms SMs (the device's
 * count, or the dg_set_num_sms limit); 0 when it would not use stream-K.
 * Pure host arithmetic.  Errors as dg_plan_fp8_gemm_nt. */
dg_status dg_fp8_gemm_nt_workspace_size(int64_t m, int64_t n, int64_t k, int32_t has_c,
                                        int32_t num_sms, uint64_t* bytes);

/* Dense NT with arbitrary FP32 scales (no power-of-two requirement):
 *   D[m, n] = C[m, n] + sum_kb (sum_{k in kb} A[m, k] B[n, k]) * sfa[kb][m] * sfb[n/128][kb]
 *   sfa  float [ceil(k/128), align(m, 4)]: one scale per 1x128 group of A,
 *        K-block-major ("transposed") and padded to 16 bytes per K block
 *   sfb  float [ceil(n/128), k/128]: one scale per 128x128 block of B
 *   a, b, c, d, strides and checks as dg_fp8_gemm_nt; sfa, sfb 4-byte aligned.
 * The tensor core produces each 128-wide K block's FP32 partial sum in TMEM;
 * it is scaled and accumulated in FP32 on the CUDA cores (two-level
 * accumulation), so any finite scale is honoured exactly as the FP32
 * product sfa * sfb.  128-column tiles.
 * Cited: same page, section "Interface GEMM e restrições de layout" (FP32
 * scale factors; LHS scales TMA-aligned and transposed); launch report on
 * feifmx.com (Feb 2025), two-level accumulation with CUDA-core promotion. */
dg_status dg_fp8_gemm_nt_fp32_sf(const void* a, const float* sfa, const void* b, const float* sfb,
                                 const void* c, void* d, int64_t m, int64_t n, int64_t k,
                                 int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, void* stream);

/* Dense GEMM in the other three operand layouts ("D = C + A @ B" with A
 * logically [m, k] and B logically [k, n]; "n" = stored as is, "t" = stored
 * transposed).  Scales, C, D, their layouts and all checks are as for
 * dg_fp8_gemm_nt; only the storage of A and B differs:
 *   nn:  a E4M3 [m, k] row stride lda >= k;  b E4M3 [k, n] row stride ldb >= n
 *   tn:  a E4M3 [k, m] row stride lda >= m;  b E4M3 [k, n] row stride ldb >= n
 *   tt:  a E4M3 [k, m] row stride lda >= m;  b E4M3 [n, k] row stride ldb >= k
 * (lda, ldb % 16 == 0).  sfa is packed per row m, sfb per row n, exactly as
 * for NT (the scale groups follow K whatever the storage).
 * Cited: same page, section "GEMM denso e grouped" (fp8_gemm_{nt, nn, tn, tt})
 * and section "Interface GEMM e restrições de layout" (the SM100 path supports
 * the NT, TN, NN and TT memory layouts). */
dg_status dg_fp8_gemm_nn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream);
dg_status dg_fp8_gemm_tn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream);
dg_status dg_fp8_gemm_tt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                         const void* c, void* d, int64_t m, int64_t n, int64_t k, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t ldd, void* stream);

/* M-grouped, contiguous layout.  The token rows of all experts are
 * concatenated along M, each expert's segment padded to a multiple of 128 rows
 * (dg_get_mk_alignment_for_contiguous_layout); N and K are shared.
 *   a          E4M3 [m_sum, k] (contiguous rows), m_sum % 128 == 0
 *   sfa        packed UE8M0 [ceil(k/512), align(m_sum, 4)]
 *   b          E4M3 [num_groups, n, k] (contiguous)
 *   sfb        packed UE8M0 [num_groups, ceil(k/512), align(n, 4)]
 *   d          BF16 [m_sum, n] (contiguous)
 *   m_indices  int32 [m_sum] on the device: the expert of each row, -1 for a
 *              padding row.  Row r of D is written iff m_indices[r] >= 0; other
 *              rows are left untouched.  Each 128-row block must hold rows of
 *              one expert followed only by -1 rows; a block whose first row
 *              is -1 is skipped.  Violations (index >= num_groups, a second
 *              expert inside a block) leave those rows unwritten and set
 *              DG_ERR_DEVICE_BAD_INDEX.
 * m_indices is never read on the host.
 * Cited: same page, section "GEMM denso e grouped" (contiguous layout:
 * M-axis grouping, fixed N and K, segments aligned to the GEMM M block). */
dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b,
                                              const int32_t* sfb, void* d,
                                              const int32_t* m_indices, int64_t m_sum, int64_t n,
                                              int64_t k, int32_t num_groups, void* stream);

/* M-grouped, masked layout (decode under CUDA graphs: the host does not know
 * the per-expert token counts).
 *   a         E4M3 [num_groups, max_m, k] (contiguous)
 *   sfa       packed UE8M0 [num_groups, ceil(k/512), align(max_m, 4)]
 *   b         E4M3 [num_groups, n, k]
 *   sfb       packed UE8M0 [num_groups, ceil(k/512), align(n, 4)]
 *   d         BF16 [num_groups, max_m, n]
 *   masked_m  int32 [num_groups] on the device: rows [0, masked_m[g]) of
 *             group g are computed and written; rows at or beyond it are left
 *             untouched.  The 128-row blocks of A that hold no valid row are
 *             never read; inside a block that holds one, the rows past
 *             masked_m[g] are loaded and multiplied like the others, but their
 *             results are never stored (so A's contents there do not matter).
 *             Values outside [0, max_m] are clamped and set
 *             DG_ERR_DEVICE_BAD_INDEX.
 *   expected_m  host hint of the typical masked_m (tile selection only);
 *               0 = unknown.  Never affects results.
 * num_groups <= 512.  masked_m is never read on the host, so the call can
 * be captured in a CUDA graph.
 * Cited: same page, section "GEMM denso e grouped" (masked grouped GEMM,
 * m_grouped_fp8_gemm_nt_masked: with a mask tensor the kernel computes only
 * the valid region). */
dg_status dg_m_grouped_fp8_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b,
                                          const int32_t* sfb, void* d, const int32_t* masked_m,
                                          int32_t num_groups, int64_t max_m, int64_t n, int64_t k,
                                          int64_t expected_m, void* stream);

/* K-grouped, contiguous layout ("TN"), for the weight gradients of MoE
 * experts: the experts' token rows are stacked along K, M and N are shared.
 * Expert g owns rows [off_g, off_g + ks[g]) of A and B (off_g = ks[0] + ... +
 * ks[g-1]) and produces
 *   D[g][m, n] = C[g][m, n] + sum_{k in expert g} A[k, m] * B[k, n]
 * (dequantised, FP32 accumulation, FP32 output).
 *   a    E4M3 [sum_k, m] (contiguous, M innermost), m % 16 == 0
 *   sfa  packed UE8M0 [ceil(sum_k/512), align(m, 4)]: one scale per 128 rows
 *        of each column of A (byte t of word (j, col) = e + 127 of K block 4j+t)
 *   b    E4M3 [sum_k, n] (contiguous, N innermost), n % 16 == 0
 *   sfb  packed UE8M0 [ceil(sum_k/512), align(n, 4)], the same per column of B
 *   c    float [num_groups, m, n] or NULL for C = 0; may equal d
 *   d    float [num_groups, m, n] (contiguous); every element is written
 *   ks   int32 [num_groups] on the device: rows per expert, each a multiple
 *        of 128 (dg_get_mk_alignment_for_contiguous_layout), summing to
 *        sum_k.  An expert with 0 rows gets D[g] = C[g] (or 0).  A size that
 *        is negative or not a multiple of 128 counts as 0, and rows past
 *        sum_k are dropped; both set DG_ERR_DEVICE_BAD_INDEX.
 * sum_k % 128 == 0; num_groups <= 512.  ks is never read on the host.
 * Cited: same page, section "GEMM denso e grouped" (a grouped API along K for
 * the weight backward of MoE, M and N fixed, k_grouped_fp8_gemm_tn_contiguous);
 * the page does not give the operand layout or scale granularity: the
 * reading above ("TN": both operands with the reduction axis outermost; the
 * fine-grained 128-element scale groups taken along K) is this library's. */
dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void* a, const int32_t* sfa, const void* b,
                                              const int32_t* sfb, const float* c, float* d,
                                              const int32_t* ks, int64_t m, int64_t n,
                                              int64_t sum_k, int32_t num_groups, void* stream);

/* ------------------------------------------------------------------------ */
/* Quantisation and scale layout                                             */
/* ------------------------------------------------------------------------ */

/* FP32 -> E4M3 with fine-grained power-of-two scales.
 *   x   float [groups, rows, cols] (contiguous), cols % 128 == 0
 *   q   E4M3 [groups, rows, cols] (contiguous)
 *   sf  block_rows == 1:   one scale per 1x128 row group (activations)
 *       block_rows == 128: one scale per 128x128 block (weights; a partial
 *                          last block covers the rows that exist)
 *       sf_format DG_SF_FP32: float [groups, ceil(rows/block_rows), cols/128]
 *       sf_format DG_SF_UE8M0_PACKED: int32 [groups, ceil(cols/512), align(rows, 4)]
 *       (rows in the alignment padding and unused bytes are written as 0).
 * Scale rule: s = 2^e, e the smallest integer with 448 * 2^e >= amax of the
 * group (e clamped to [-127, 127]; an all-zero group gets e = 0), then
 * q = E4M3(x / s), rounding to nearest even and saturating at +-448.
 * Cited: same page, section "Interface GEMM e restrições de layout" (casting
 * to FP8 is left to the user; the library offers simple utilities). */
dg_status dg_quantize_fp8(const float* x, void* q, void* sf, int64_t groups, int64_t rows,
                          int64_t cols, int32_t block_rows, int32_t sf_format, void* stream);

/* FP32 -> E4M3 with one power-of-two scale per 128 rows of each column, the
 * grouping of operands whose reduction axis is the row axis (A and B of
 * dg_k_grouped_fp8_gemm_tn_contiguous).
 *   x   float [rows, cols] (contiguous), rows % 128 == 0, cols % 4 == 0
 *   q   E4M3 [rows, cols] (contiguous)
 *   sf  sf_format DG_SF_FP32: float [rows/128, cols]
 *       sf_format DG_SF_UE8M0_PACKED: int32 [ceil(rows/512), align(cols, 4)],
 *       byte t of word (j, col) = e + 127 of the 128-row block 4j+t (unused
 *       bytes and padding columns are 0)
 * Same scale rule and cast as dg_quantize_fp8.  Cited: same page, section
 * "Interface GEMM e restrições de layout" (fine-grained scaling; casting is
 * the user's job, the library offers utilities), applied along K for the
 * K-grouped layout of section "GEMM denso e grouped". */
dg_status dg_quantize_fp8_cols(const float* x, void* q, void* sf, int64_t rows, int64_t cols,
                               int32_t sf_format, void* stream);

/* FP32 scales -> packed UE8M0 layout.
 *   sf      float [groups, ceil(mn/block_rows), ceil(k/128)]
 *   packed  int32 [groups, ceil(k/512), align(mn, 4)]
 * Each scale must be a positive power of two (2^-127 .. 2^127).  Any other
 * value is rounded up to the next power of two (non-positive or non-finite
 * values become 1.0) and DG_ERR_DEVICE_BAD_SCALE is recorded.
 * Cited: same page, section "Utilitários e variáveis de ambiente"
 * (transform_sf_into_required_layout). */
dg_status dg_transform_sf(const float* sf, int32_t* packed, int64_t groups, int64_t mn, int64_t k,
                          int32_t block_rows, void* stream);

/* ------------------------------------------------------------------------ */
/* Utilities (same page, section "Utilitários e variáveis de ambiente")      */
/* ------------------------------------------------------------------------ */

/* Environment variables read by the library (when the process environment
 * changes, not on every call), all optional, for tuning and diagnosis:
 *   DG_PRINT_CONFIGS=1   print each launch's configuration to stderr;
 *   DG_BLOCK_M=128|256, DG_BLOCK_N=128|192|224|256   force the tile size;
 *   DG_SPLIT_K=1|2|4|8   force the split-K cluster size (8: decode kernel);
 *   DG_CTA_PAIR=1        256-row tiles on 2-CTA pairs (cta_group::2 MMAs);
 *   DG_STREAM_K=0|1      forbid / force stream-K where a workspace allows it;
 *   DG_MULTICAST=0       256-row dense tiles and K-grouped tiles one CTA each
 *                        instead of 2-CTA clusters sharing B by TMA multicast;
 *   DG_TALL_EPI8=0       four epilogue warps for 256-row tiles instead of eight;
 *   DG_DECODE=0          tiled kernels instead of the decode kernel for M <= 128;
 *   DG_RASTER_BAND=n     M blocks per raster band (default 16).
 * Tile sizes and multicast clusters give the same bits: each output element
 * accumulates its K blocks in the same order (tested for 128- against
 * 256-row tiles and for multicast on against off, dense and K-grouped).  Configurations that
 * split K between CTAs (split-K, stream-K, decode clusters) add the partial
 * sums in a fixed order, so their bits are reproducible but may differ from
 * an unsplit launch's within FP32 rounding. */

/* x rounded up so that x * element_size is a multiple of 16 bytes. */
int64_t dg_get_tma_aligned_size(int64_t x, int32_t element_size);

/* Row alignment of each expert segment in the contiguous layouts (the
 * M-grouped contiguous form along M, the K-grouped form along K): 128 unless
 * set.  dg_set_mk_alignment_for_contiguous_layout sets the value the getter
 * returns, process-wide, for callers that lay their segments out by it: a
 * positive multiple of 128 up to 4096 (the kernels work on 128-row blocks,
 * so they accept any such multiple; 256, for instance, lets the contiguous
 * form's 256-row tiles pair every block with one of the same expert),
 * anything else gives DG_ERR_INVALID_ARG and changes nothing.  Cited: same
 * section (get / set_mk_alignment_for_contiguous_layout). */
int32_t dg_get_mk_alignment_for_contiguous_layout(void);
dg_status dg_set_mk_alignment_for_contiguous_layout(int32_t alignment);

/* The tile configuration dg_fp8_gemm_nt chooses for an M x N x K problem,
 * with C (has_c != 0) or without, on a device with num_sms SMs (pass the
 * device's SM count, or the dg_set_num_sms limit when one is set).  Pure host
 * arithmetic: no device, no CUDA call.  The DG_BLOCK_M, DG_BLOCK_N, DG_SPLIT_K
 * and DG_CTA_PAIR environment overrides apply as they do to the call, and
 * DG_DECODE = 0 turns off the decode kernel below.
 * Writes block_m (rows of A per output tile: 64 for the 64-row A slots of a
 * single short M block, 128, or 256), block_n (columns per tile), split_k
 * (CTAs of one cluster sharing each tile's K blocks: 1, 2 or 4) and cta_pair
 * (1 when a 256-row tile spans two CTAs).  For M <= 128 the call normally
 * runs the decode kernel, which swaps the operands' roles: 128 rows of B
 * fill the MMA's 128 lanes and A's rows are its N side; then block_m is the
 * MMA's token width (32, 64 or 128, at least M), block_n 128 and split_k the
 * CTAs of a cluster sharing each 128-column strip's K blocks (1, 2, 4 or 8).
 * All four are 0 for an empty
 * problem.  Errors as dg_fp8_gemm_nt's shape checks; num_sms < 1 or a NULL
 * output gives DG_ERR_INVALID_ARG.  Cited: same page, section "Utilitários e
 * variáveis de ambiente" (DG_PRINT_CONFIGS prints the configuration chosen
 * for a shape); this query returns it instead. */
dg_status dg_plan_fp8_gemm_nt(int64_t m, int64_t n, int64_t k, int32_t has_c, int32_t num_sms,
                              int32_t* block_m, int32_t* block_n, int32_t* split_k,
                              int32_t* cta_pair);

/* The tile configuration dg_fp8_gemm_nt_ws chooses when its workspace is
 * large enough: the outputs of dg_plan_fp8_gemm_nt plus stream_k (1 when the
 * K blocks of the last waves are split between SMs), swap_ab (1 when the
 * decode kernel with swapped operand roles runs; dg_fp8_gemm_nt makes the
 * same choice) and multicast (1 when the 256-row tiles run in clusters of two
 * CTAs on adjacent M blocks and one column block of B, each CTA loading half
 * of the B tile into both with TMA multicast; dg_fp8_gemm_nt makes the same
 * choice; DG_MULTICAST = 0 turns it off).  Same checks. */
dg_status dg_plan_fp8_gemm_nt_ws(int64_t m, int64_t n, int64_t k, int32_t has_c, int32_t num_sms,
                                 int32_t* block_m, int32_t* block_n, int32_t* split_k,
                                 int32_t* cta_pair, int32_t* stream_k, int32_t* swap_ab,
                                 int32_t* multicast);

/* The same query for the two M-grouped forms: the tile configuration
 * dg_m_grouped_fp8_gemm_nt_contiguous / _masked chooses (block_m 256 when a
 * tile pairs two 128-row blocks of one expert, contiguous, or spans a CTA
 * pair, masked).  The per-expert row counts stay on the device, so the masked
 * choice depends on expected_m as the call's does.  Pure host arithmetic; the
 * same checks and overrides as the calls; all outputs 0 for an empty problem.
 * Cited as above. */
dg_status dg_plan_m_grouped_fp8_gemm_nt_contiguous(int64_t m_sum, int64_t n, int64_t k,
                                                   int32_t num_groups, int32_t num_sms,
                                                   int32_t* block_m, int32_t* block_n);
dg_status dg_plan_m_grouped_fp8_gemm_nt_masked(int32_t num_groups, int64_t max_m, int64_t n,
                                               int64_t k, int64_t expected_m, int32_t num_sms,
                                               int32_t* block_m, int32_t* block_n,
                                               int32_t* cta_pair);

/* Upper bound on the SMs the persistent GEMM grid uses; 0 = all SMs of the
 * device.  Process-wide; returns DG_ERR_INVALID_ARG for n < 0. */
dg_status dg_set_num_sms(int32_t n);
int32_t dg_get_num_sms(void);

/* Programmatic dependent launch (PDL), process-wide, off by default.  When on,
 * every kernel of this library is launched with programmatic stream
 * serialisation: it may start while the previous kernel on the stream is
 * finishing, does its set-up (barriers, TMEM allocation, descriptor
 * prefetch), then waits for that kernel's completion before reading global
 * memory; and it lets the next kernel start its own set-up once its set-up is
 * done.  Inside CUDA graphs the dependency becomes a programmatic edge.
 * dg_set_pdl returns DG_ERR_INVALID_ARG for values other than 0 and 1.
 * Cited: same page, section "Utilitários e variáveis de ambiente" (set_pdl /
 * get_pdl). */
dg_status dg_set_pdl(int32_t enable);
int32_t dg_get_pdl(void);

/* Limit of every bounded wait inside the kernels, in nanoseconds (default
 * 2e9).  Process-wide; applies to launches made after the call. */
dg_status dg_set_wait_timeout_ns(uint64_t ns);

/* Synchronises `stream`, then reads and clears the device error words of the
 * current device.  Returns DG_OK or the first recorded DG_ERR_DEVICE_* code.
 * If detail is not NULL it receives the raw word (code in bits 0-7, the
 * recording site in bits 8-23, block index in bits 32-63).  Debug/test use.
 * Sites 40-45 belong to the debug library's checks (A load, B load, scale
 * load, TMEM columns, output rows and columns, stream-K slot and K range).
 * The words are one per device and per process, shared by every launch on
 * every stream: the result is only meaningful when no other work of this
 * library is in flight on the device (a kernel still running on another
 * stream may have its condition cleared here or reported against this call). */
dg_status dg_get_device_error(void* stream, uint64_t* detail);

/* Test hook for failure detection, process-wide, off (0) by default.  With
 * k > 0, the next dense NT launches make CTA 0 arm the pipeline stage of K
 * block k - 1 of its first tile without filling it: that stage never
 * completes, so the kernel's bounded waits must end the launch by themselves
 * and record DG_ERR_DEVICE_TIMEOUT (the result D is then incomplete).  Nothing
 * faults or hangs; the context stays usable.  Pair it with a short
 * dg_set_wait_timeout_ns and reset it to 0 afterwards.  k < 0 gives
 * DG_ERR_INVALID_ARG.  No counterpart on the pages: it exists to test the
 * library's own bounded waits. */
dg_status dg_debug_set_drop_load(int32_t k);

/* Test hook for the device checks of the debug build (libdg_debug.so, built
 * with DG_DEBUG_CHECKS=1), process-wide, off (0) by default.  With on != 0
 * the next single-CTA dense NT launches (no split-K, no CTA pair) evaluate
 * the MMA issuer's TMEM-column check as violated: each records
 * DG_ERR_DEVICE_CHECK at that check's site in the error word (no access
 * changes, D is still computed), which dg_get_device_error then returns.
 * The release library has no checks: there on != 0 gives DG_ERR_INVALID_ARG
 * and on == 0 DG_OK.  No counterpart on the pages: it exists to show that
 * a failed check reaches the caller. */
dg_status dg_debug_plant_check(int32_t on);

/* Static description of a status code. */
const char* dg_status_string(dg_status s);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t dg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DG_H_ */
