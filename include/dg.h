/*
 * dg.h -- C ABI of the GB300 (sm_103a) block-scaled FP8 GEMM library.
 *
 * The library computes D = C + A @ B^T ("NT": A row-major [M,K], B stored as
 * [N,K], both K-contiguous), where A and B are FP8 E4M3 ("fn" flavour), A
 * carries one scale per 1x128 K-group of each row and B one scale per 128x128
 * block, accumulation is FP32 and D is bf16.  Sources: "02 · DeepGEMM 技术解析"
 * (PaperTrace) §1.1, §2, §3, §5 and "DeepSeek V4 源码剖析 第13章 DeepGEMM"
 * §13.3, §13.6.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named a, b, c, d, sfa, sfb, out, grouped_layout, masked_m,
 *    status_dev are DEVICE pointers; the caller owns and allocates all of
 *    them.  The library allocates no device memory on any call.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is asynchronous: it validates its arguments on the host, enqueues
 *    its kernels on `stream` and returns.
 *  - Host-detected errors (bad sizes, strides, alignment, formats, or a
 *    device that is not sm_103) are returned synchronously as a dg_status
 *    before anything is enqueued; nothing is written in that case.
 *  - Device-detected conditions are OR-ed as dg_device_flag bits into
 *    *status_dev (an int32 in device memory, nullable) and are visible
 *    after the stream is synchronised.  Kernels never trap: every wait on the
 *    device has a time limit, after which the kernel sets DG_DEV_TIMEOUT and
 *    returns.
 *  - Scale factors have granularity 128 along K (and 128 along N for B, in
 *    the FP32 form).  sf_k = ceil(K/128), psf_k = ceil(sf_k/4),
 *    align4(x) = ceil(x/4)*4.
 *  - Packed UE8M0 scales (DG_SF_UE8M0_PACKED) are int32 words holding the
 *    exponent bytes of four consecutive K-groups, little-endian by K index,
 *    laid out MN-major: word (row i, slice p) at p*align4(mn) + i, batch
 *    stride psf_k*align4(mn) (PaperTrace §3.1).  B's packed scales are one row
 *    per N index (the 128x128 block scale broadcast along N, §3.2).
 *  - Operand preconditions, unless a call states its own: 16-byte aligned
 *    base pointers; K % 16 == 0; lda, ldb (in elements = bytes) multiples of
 *    16; N % 8 == 0 and ldc, ldd (bf16 elements) multiples of 8.  (FP4
 *    weights, M/N-contiguous operands and FP32 outputs have their own rules,
 *    given with their calls.)
 *  - No split-K: each output element is reduced by one CTA in a fixed K
 *    order, so a row's result does not depend on M or on the other rows of
 *    the batch (batch invariance, §13.1).
 */
#ifndef DG_GB300_H
#define DG_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,   /* a size, pointer or enum value is out of range */
    DG_ERR_ALIGNMENT = 2,     /* a pointer or leading dimension breaks the 16-byte rules */
    DG_ERR_LAYOUT = 3,        /* a scale layout does not match the contract */
    DG_ERR_UNSUPPORTED = 4,   /* valid request outside what the library implements */
    DG_ERR_CUDA = 5,          /* a CUDA runtime call failed (launch, attribute, device) */
    DG_ERR_TIMEOUT = 6,       /* used by helpers that read back the device status */
    DG_ERR_INEXACT_SCALE = 7, /* idem */
    DG_ERR_BAD_GROUP = 8      /* idem */
} dg_status;

/* Bits OR-ed into *status_dev by the kernels. */
typedef enum {
    DG_DEV_TIMEOUT = 1,        /* a bounded device wait ran out; outputs are incomplete */
    DG_DEV_INEXACT_SCALE = 2,  /* an FP32 scale was not a power of two and was truncated */
    DG_DEV_BAD_GROUP = 4       /* an expert id >= num_groups, or masked_m[e] > max_m */
} dg_device_flag;

typedef enum {
    DG_SF_FP32 = 0,          /* FP32 scales in the caller's natural form (see each call) */
    DG_SF_UE8M0_PACKED = 1   /* packed MN-major UE8M0 int32 words (see conventions) */
} dg_sf_format;

/*
 * dg_fp8_gemm_nt -- D[m,n] = C[m,n] + sum_k A[m,k]*sfa(m,k/128) * B[n,k]*sfb(n,k/128)
 * ("DeepSeek V4 源码剖析 第13章" §13.3 interface and pseudocode; PaperTrace §2).
 *
 *   a     [m, lda]  E4M3 codes, row m at a + m*lda, K contiguous.
 *   b     [n, ldb]  E4M3 codes (the "column-major B" of the NT layout).
 *   sfa, sfb formats must match:
 *     DG_SF_UE8M0_PACKED: sfa int32 [psf_k][align4(m)], sfb int32
 *       [psf_k][align4(n)] (one row per N index).  Runs the tcgen05
 *       block-scaled MMA path, exact for power-of-two scales.
 *     DG_SF_FP32: sfa float [m][sf_k] row-major, sfb float [ceil(n/128)][sf_k]
 *       row-major.  Any finite FP32 scale is honoured: each 128-K block is
 *       accumulated on the tensor core and promoted into an FP32 accumulator
 *       as acc += sa*sb*partial (the two-level accumulation of PaperTrace §2.2).
 *   c     bf16 [m, ldc] or NULL (C = 0).  c may equal d (in-place accumulate).
 *   d     bf16 [m, ldd] output.
 *   m, n, k >= 0; m == 0 or n == 0 is a no-op; k == 0 gives D = C.
 *   status_dev: nullable int32 device word receiving dg_device_flag bits.
 */
dg_status dg_fp8_gemm_nt(const void *a, int64_t lda, const void *sfa, int sfa_fmt,
                         const void *b, int64_t ldb, const void *sfb, int sfb_fmt,
                         const void *c, int64_t ldc, void *d, int64_t ldd,
                         int m, int n, int k, int32_t *status_dev, void *stream);

/*
 * dg_transform_sf -- FP32 scales into the MN-major, TMA-aligned layout the GEMMs
 * consume (PaperTrace §3.1-3.2; "DeepSeek V4 源码剖析 第13章" §13.3 constraint 2).
 *
 *   sf      float [batch][mn_rows][sf_k] row-major; row r covers MN indices
 *           r*gran_mn .. r*gran_mn + gran_mn - 1.
 *   gran_mn 1 (activation, 1x128) or 128 (weight, 128x128); mn_rows must equal
 *           ceil(mn / gran_mn).  The output has one row per MN index.
 *   out_fmt DG_SF_UE8M0_PACKED: out int32 [batch][psf_k][align4(mn)]; byte j of
 *             word (p, i) = (bits(sf[i/gran_mn][4p+j]) >> 23) & 0xff, i.e. the
 *             exponent byte: a non-power-of-two scale is truncated (0.75 -> 0.5,
 *             3 -> 2) and DG_DEV_INEXACT_SCALE is set in *status_dev.
 *           DG_SF_FP32: out float [batch][sf_k][align4(mn)] (transpose only).
 *           Bytes past sf_k in the last word and pad rows mn..align4(mn)-1 are 0.
 *   out must not overlap sf.  Size it with dg_packed_sf_words (int32 count) or
 *   batch*sf_k*align4(mn) floats.
 */
dg_status dg_transform_sf(const float *sf, int batch, int mn_rows, int sf_k, int gran_mn, int mn,
                          int out_fmt, void *out, int32_t *status_dev, void *stream);

/*
 * dg_fp8_gemm_nt_f32 -- dg_fp8_gemm_nt with FP32 D and an optional FP32 C
 * ("DeepSeek V4 源码剖析 第13章" §13.3: D = C + A @ B^T; the pages fix no D
 * type, and this form keeps the FP32 accumulator, e.g. to accumulate in place
 * with c == d).  D = C + the FP32 accumulator, added in FP32, no further
 * rounding.
 *
 *   a, sfa, b, sfb, lda, ldb, m, n, k: as for dg_fp8_gemm_nt; only
 *          DG_SF_UE8M0_PACKED scales are accepted (else DG_ERR_UNSUPPORTED).
 *   c      FP32 [m, ldc] or NULL; may alias d.
 *   d      FP32 [m, ldd].
 *   d and c 16-byte aligned, n, ldd and ldc multiples of 4 (else
 *   DG_ERR_ALIGNMENT).  Runs on 256-row CTA pairs for every m.  k == 0 gives D = C
 *   (or 0).
 */
dg_status dg_fp8_gemm_nt_f32(const void *a, int64_t lda, const void *sfa, int sfa_fmt, const void *b,
                             int64_t ldb, const void *sfb, int sfb_fmt, const float *c, int64_t ldc,
                             float *d, int64_t ldd, int m, int n, int k, int32_t *status_dev,
                             void *stream);

/*
 * dg_fp8_gemm_nn / dg_fp8_gemm_tn / dg_fp8_gemm_tt -- the other three operand
 * layouts of "DeepSeek V4 源码剖析 第13章" §13.3 (D = C + A @ B, the two suffix
 * letters giving the transpose state of A and B; the SM100 generation supports
 * all four).  The product and its scales are those of dg_fp8_gemm_nt; only the
 * memory order of A and B changes:
 *
 *   call  A storage            B storage            D[m,n] = C + sum_k ...
 *   nn    [m][lda], K contig.  [k][ldb], N contig.  A[m,k] B[k,n]
 *   tn    [k][lda], M contig.  [k][ldb], N contig.  A[k,m] B[k,n]
 *   tt    [k][lda], M contig.  [n][ldb], K contig.  A[k,m] B[n,k]
 *
 *   Scales: sfa, sfb as for dg_fp8_gemm_nt (one A scale per (m, 128-K block),
 *   one B scale per (128-N block, 128-K block)); only DG_SF_UE8M0_PACKED is
 *   accepted here (DG_SF_FP32 gives DG_ERR_UNSUPPORTED).
 *   Leading dimensions: lda >= k (A K-contiguous) or >= m (M-contiguous);
 *   ldb >= k or >= n likewise; all multiples of 16 (else DG_ERR_ALIGNMENT).
 *   k must be a multiple of 16 when an operand is K-contiguous.
 *   c (bf16 [m, ldc], nullable, may equal d) and d (bf16 [m, ldd]) as for
 *   dg_fp8_gemm_nt; n, ldd, ldc multiples of 8.  Runs on 256x256 CTA-pair tiles.
 *   m == 0 or n == 0 is a no-op; k == 0 gives D = C (or 0).
 */
dg_status dg_fp8_gemm_nn(const void *a, int64_t lda, const void *sfa, int sfa_fmt,
                         const void *b, int64_t ldb, const void *sfb, int sfb_fmt,
                         const void *c, int64_t ldc, void *d, int64_t ldd,
                         int m, int n, int k, int32_t *status_dev, void *stream);
dg_status dg_fp8_gemm_tn(const void *a, int64_t lda, const void *sfa, int sfa_fmt,
                         const void *b, int64_t ldb, const void *sfb, int sfb_fmt,
                         const void *c, int64_t ldc, void *d, int64_t ldd,
                         int m, int n, int k, int32_t *status_dev, void *stream);
dg_status dg_fp8_gemm_tt(const void *a, int64_t lda, const void *sfa, int sfa_fmt,
                         const void *b, int64_t ldb, const void *sfb, int sfb_fmt,
                         const void *c, int64_t ldc, void *d, int64_t ldd,
                         int m, int n, int k, int32_t *status_dev, void *stream);

/*
 * dg_fp8_fp4_gemm_nt -- FP8 activations x FP4 weights ("DeepSeek V4 源码剖析
 * 第13章" §13.1 reason 2 and §13.5: E2M1 weights whose scales run along K, one
 * per 32 elements; the tensor cores take the mixed operands directly):
 *
 *   D[m,n] = C[m,n] + sum_k A[m,k] sa(m, k/128) * B[n,k] sb(n, k/32)
 *
 *   a    E4M3 [m, lda], K contiguous; sfa packed UE8M0 int32 [ceil(k/512)][align4(m)]
 *        (as for dg_fp8_gemm_nt: 4 x 128 K per word).
 *   b    E2M1 codes packed two per byte, row n at b + n*ldb BYTES: element k is
 *        byte k/2, low nibble for even k; b 32-byte aligned, ldb >= k/2 and a
 *        multiple of 32 (else DG_ERR_ALIGNMENT / DG_ERR_INVALID_ARG).
 *   sfb  packed UE8M0 int32 [k/128][align4(n)]: byte j of word (p, i) is the
 *        scale of row i for K elements 128p + 32j .. 128p + 32j + 31; build it
 *        with dg_transform_sf(sfb_fp32 [n][k/32], 1, n, k/32, 1, n, ...).
 *   c    bf16 [m, ldc] or NULL (may equal d); d bf16 [m, ldd].
 *   k a multiple of 128 (DG_ERR_ALIGNMENT otherwise); k == 0 gives D = C.
 *   n, ldc, ldd multiples of 8.  Runs on 256-row CTA pairs; with m <= 128 and
 *   no C, on 128-row CTA pairs (BLOCK_N 32, 96 or 128) instead.  Row i of D is
 *   the same bit for bit whatever m the call has (both tile forms sum each
 *   element's K-blocks in the same order).
 */
dg_status dg_fp8_fp4_gemm_nt(const void *a, int64_t lda, const void *sfa, const void *b, int64_t ldb,
                             const void *sfb, const void *c, int64_t ldc, void *d, int64_t ldd, int m, int n,
                             int k, int32_t *status_dev, void *stream);

/*
 * dg_m_grouped_fp8_fp4_gemm_nt_contiguous / _masked -- the MoE GEMMs grouped
 * along M with FP4 expert weights ("DeepSeek V4 源码剖析 第13章" §13.6: the
 * routed experts run FP8 activations x FP4 weights through
 * m_grouped_fp8_fp4_gemm_nt_{contiguous,masked}).  Layouts, grouped_layout,
 * masked_m and expected_m as for the FP8 calls below; B and its scales as for
 * dg_fp8_fp4_gemm_nt, per expert:
 *   b    E2M1 packed [num_groups][n][ldb bytes] (masked: ldb = k/2), expert
 *        stride n*ldb; 32-byte aligned, ldb a multiple of 32.
 *   sfb  packed int32 [num_groups][k/128][align4(n)] (dg_transform_sf on FP32
 *        [num_groups][n][k/32] with gran_mn 1 and batch num_groups).
 *   sfa  packed as for the FP8 calls ([ceil(k/512)][align4(m_total)], masked:
 *        [num_groups][ceil(k/512)][align4(max_m)]).
 *   k a multiple of 128.  Runs on 256-row CTA pairs only: the contiguous form
 *   takes m_total <= 131072, the masked one at most 512 experts.
 */
dg_status dg_m_grouped_fp8_fp4_gemm_nt_contiguous(const void *a, int64_t lda, const void *sfa, const void *b,
                                                  int64_t ldb, const void *sfb, void *d, int64_t ldd,
                                                  const int32_t *grouped_layout, int m_total, int n, int k,
                                                  int num_groups, int32_t *status_dev, void *stream);
dg_status dg_m_grouped_fp8_fp4_gemm_nt_masked(const void *a, const void *sfa, const void *b, const void *sfb,
                                              void *d, const int32_t *masked_m, int num_groups, int max_m,
                                              int expected_m, int n, int k, int32_t *status_dev, void *stream);

/*
 * dg_m_grouped_fp8_gemm_nt_contiguous -- MoE GEMM grouped along M only
 * (PaperTrace §5.1; "DeepSeek V4 源码剖析 第13章" §13.6): the rows of all
 * experts are concatenated along M, each expert's segment starting on a
 * multiple of dg_get_mk_alignment_for_contiguous_layout() (128) rows.
 *
 *   a      [m_total, lda] E4M3; sfa packed int32 [psf_k][align4(m_total)].
 *   b      [num_groups][n][ldb] E4M3 (expert stride n*ldb);
 *   sfb    packed int32 [num_groups][psf_k][align4(n)].
 *   d      bf16 [m_total, ldd].
 *   grouped_layout int32 [m_total]: expert id of each row, -1 for padding
 *          rows.  Every 128-row block belongs to one expert, taken from its
 *          first row; a block whose first row is -1 is skipped and its D rows
 *          are left unwritten.  D rows marked -1 inside a computed block hold
 *          unspecified values.  An id >= num_groups sets DG_DEV_BAD_GROUP and
 *          the block is skipped.
 *   Only DG_SF_UE8M0_PACKED scales are accepted (else DG_ERR_UNSUPPORTED).
 */
dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void *a, int64_t lda, const void *sfa,
                                              int sfa_fmt, const void *b, int64_t ldb,
                                              const void *sfb, int sfb_fmt, void *d, int64_t ldd,
                                              const int32_t *grouped_layout, int m_total, int n,
                                              int k, int num_groups, int32_t *status_dev,
                                              void *stream);

/*
 * dg_m_grouped_fp8_gemm_nt_contiguous_psum -- the contiguous MoE GEMM with
 * the groups given as prefix sums of their row counts (PaperTrace §5.1: the
 * per-expert prefix sums of received tokens serve as group offsets; §3.1: gap
 * rows lie between groups).  Reading taken: psum[e] = m_0 + ... + m_e (int32,
 * device memory, non-decreasing); expert e's rows are [S_e, S_e + m_e) with
 * S_0 = 0 and S_{e+1} = S_e rounded up past m_e rows to a multiple of 128.
 *
 *   a, sfa, b, sfb, d, strides: as for dg_m_grouped_fp8_gemm_nt_contiguous.
 *   psum   int32 [num_groups] in device memory (read by the kernel).
 *   D rows [S_e + m_e, S_{e+1}) (gap rows) are written 0; rows at or past
 *   S_E are not written.  A decreasing psum (that count is taken as 0) or
 *   S_E > m_total sets DG_DEV_BAD_GROUP.
 *   num_groups <= 255 and m_total <= 131072 (the layout runs on 256-row CTA
 *   pairs only; DG_DEBUG_SINGLE_CTA does not apply), else DG_ERR_UNSUPPORTED.
 *   Only DG_SF_UE8M0_PACKED scales are accepted.
 */
dg_status dg_m_grouped_fp8_gemm_nt_contiguous_psum(const void *a, int64_t lda, const void *sfa,
                                                   int sfa_fmt, const void *b, int64_t ldb,
                                                   const void *sfb, int sfb_fmt, void *d, int64_t ldd,
                                                   const int32_t *psum, int m_total, int n, int k,
                                                   int num_groups, int32_t *status_dev, void *stream);

/*
 * dg_m_grouped_fp8_gemm_nt_masked -- MoE decode GEMM with static shapes
 * (PaperTrace §5.2; "DeepSeek V4 源码剖析 第13章" §13.6): expert e multiplies
 * its first masked_m[e] rows; nothing else of D is read or written.
 *
 *   a      [num_groups][max_m][k] E4M3, dense.
 *   sfa    packed int32 [num_groups][psf_k][align4(max_m)].
 *   b      [num_groups][n][k] E4M3, dense; sfb packed int32 [num_groups][psf_k][align4(n)].
 *   d      bf16 [num_groups][max_m][n], dense.
 *   masked_m int32 [num_groups] in device memory (read by the kernel, so the
 *          call can be captured in a CUDA graph with changing counts); values
 *          are clamped to [0, max_m], and a value > max_m sets DG_DEV_BAD_GROUP.
 *   expected_m  the caller's estimate of the mean valid rows per expert; only
 *          used to choose the tile shape (it never changes a result).
 *   num_groups <= 1024.  Only DG_SF_UE8M0_PACKED scales are accepted.
 */
dg_status dg_m_grouped_fp8_gemm_nt_masked(const void *a, const void *sfa, int sfa_fmt,
                                          const void *b, const void *sfb, int sfb_fmt, void *d,
                                          const int32_t *masked_m, int num_groups, int max_m,
                                          int expected_m, int n, int k, int32_t *status_dev,
                                          void *stream);

/* Row alignment of each expert segment in the contiguous layout (the tile
 * height, PaperTrace §5.1): 128. */
int dg_get_mk_alignment_for_contiguous_layout(void);

/* mn rounded up so that mn * elem_size is a multiple of 16 bytes (the TMA
 * stride rule behind align(mn, 4) for int32, PaperTrace §3.1). */
int64_t dg_get_tma_aligned_size(int64_t mn, int elem_size);

/* Number of int32 words of a packed scale tensor: batch * psf_k * align4(mn)
 * for a K extent of k elements. */
int64_t dg_packed_sf_words(int batch, int mn, int k);

/*
 * K-grouped GEMM for MoE weight gradients (PaperTrace "02 · DeepGEMM 技术解析"
 * §5.2 and §3.3; "DeepSeek V4 源码剖析 第13章" §13.3 for the "tn" naming):
 * M and N are fixed and the groups are concatenated along K.  For each group e
 * with ks[e] rows of K starting at K_e = ks[0] + ... + ks[e-1]:
 *
 *   D[e][m][n] = C[e][m][n] + sum_{k in [K_e, K_e + ks[e])} A[k][m] sa(k/128, m) * B[k][n] sb(k/128, n)
 *
 *   a    E4M3 [K_total][lda], M contiguous (lda >= m, lda % 16 == 0).
 *   b    E4M3 [K_total][ldb], N contiguous (ldb >= n, ldb % 16 == 0).
 *   ks   HOST int array [num_groups]: rows of K per group, each a multiple of
 *        128 (a group stored padded to 128 rows passes its padded size); 0 is
 *        an empty group, whose D is C.  0 <= num_groups <= 255.
 *   ks_dev  the same sizes in device memory (int32 [num_groups]); the kernel
 *        reads its group table from there.  A size there that is negative or
 *        not a multiple of 128 counts as 0 and sets DG_DEV_BAD_GROUP, as does a
 *        total beyond the host sizes' (loads past K_total read zeros).
 *   sfa, sfb  packed UE8M0 int32 [P][m] and [P][n] with
 *        P = dg_k_grouped_packed_sf_rows(ks, num_groups): each group's scale
 *        rows (one per 128 rows of K; per M or N index) packed on their own,
 *        4 per word little-endian by K, the last word of a group zero-filled
 *        past its rows, the groups' packed rows one after another.  Pages'
 *        contract: mn % 4 == 0, no MN padding (else DG_ERR_LAYOUT).  Build them
 *        from FP32 scales with dg_transform_sf_k_grouped.
 *   c    FP32 [num_groups][m][n] contiguous, REQUIRED (the pages make C
 *        mandatory for this layout); may equal d (in-place accumulation).
 *   d    FP32 [num_groups][m][n] contiguous.
 *   c, d, a, b, sfa, sfb 16-byte aligned; m, n multiples of 4.
 *   m == 0, n == 0 or num_groups == 0 is a no-op; all ks 0 gives D = C.
 *   Runs on 256x224 CTA pairs, one persistent launch over all groups.
 */
dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void *a, int64_t lda, const void *sfa, const void *b,
                                              int64_t ldb, const void *sfb, const float *c, float *d, int m,
                                              int n, const int *ks, const int32_t *ks_dev, int num_groups,
                                              int32_t *status_dev, void *stream);

/*
 * dg_transform_sf_k_grouped -- FP32 scales of the K-grouped layout into the
 * packed form above (PaperTrace §3.3).
 *   sf   FP32 [sum_e ks[e]/128][mn], mn contiguous; row r = the scales of the
 *        r-th 128-row K block of the concatenated groups.
 *   ks   HOST int array [num_groups], as for the GEMM.
 *   out  int32 [dg_k_grouped_packed_sf_rows(ks, num_groups)][mn]; byte j of
 *        packed row q of group e = (bits(sf[K_e/128 + 4q + j][i]) >> 23) & 0xff,
 *        0 past the group's rows; a non-power-of-two scale is truncated and
 *        sets DG_DEV_INEXACT_SCALE.
 *   mn % 4 == 0 (else DG_ERR_LAYOUT); ks invalid -> DG_ERR_INVALID_ARG.
 */
dg_status dg_transform_sf_k_grouped(const float *sf, int mn, const int *ks, int num_groups, void *out,
                                    int32_t *status_dev, void *stream);

/*
 * dg_k_grouped_fp8_gemm_tn_contiguous_k32 -- the K-grouped GEMM above with its
 * scales at a K granularity of 32, the form in which the pages' library takes
 * pre-packed int32 scales for this layout (PaperTrace "02 · DeepGEMM 技术解析"
 * §3.3: the int32 path is accepted only at gran_k = 32):
 *
 *   D[e][m,n] = C[e][m,n] + sum over group e's k of A[k,m] sa(k/32, m) * B[k,n] sb(k/32, n)
 *
 *   Arguments as for dg_k_grouped_fp8_gemm_tn_contiguous, except the scales:
 *   sfa, sfb  packed UE8M0 int32 [K_total/128][m] and [K_total/128][n] (no MN
 *        padding, m and n multiples of 4): row r holds, in byte j, the scale of
 *        K rows 128r + 32j .. 128r + 32j + 31 (each group's 32-row scale rows
 *        packed 4 per word on their own; group sizes being multiples of 128, no
 *        word is partial).  Build them from FP32 scales with
 *        dg_transform_sf_k_grouped_k32.
 *   Runs on 256x192 CTA pairs.
 */
dg_status dg_k_grouped_fp8_gemm_tn_contiguous_k32(const void *a, int64_t lda, const void *sfa, const void *b,
                                                  int64_t ldb, const void *sfb, const float *c, float *d, int m,
                                                  int n, const int *ks, const int32_t *ks_dev, int num_groups,
                                                  int32_t *status_dev, void *stream);

/*
 * dg_transform_sf_k_grouped_k32 -- FP32 scales of the K-grouped layout at a K
 * granularity of 32 into the packed form of dg_k_grouped_fp8_gemm_tn_contiguous_k32
 * (PaperTrace §3.3: each group packed on its own, 4 rows per int32, no MN padding).
 *   sf   FP32 [K_total/32][mn], mn contiguous; row r = the scales of K rows
 *        32r .. 32r + 31 of the concatenated groups.
 *   ks   HOST int array [num_groups], multiples of 128.
 *   out  int32 [K_total/128][mn]: byte j of row q of group e =
 *        (bits(sf[K_e/32 + 4q + j][i]) >> 23) & 0xff; a non-power-of-two scale
 *        is truncated and sets DG_DEV_INEXACT_SCALE.
 *   mn % 4 == 0 (else DG_ERR_LAYOUT); ks invalid -> DG_ERR_INVALID_ARG.
 */
dg_status dg_transform_sf_k_grouped_k32(const float *sf, int mn, const int *ks, int num_groups, void *out,
                                        int32_t *status_dev, void *stream);

/* Packed scale rows of the K-grouped layout: sum_e ceil(ks[e] / 512), or -1
 * if ks is invalid (see dg_k_grouped_fp8_gemm_tn_contiguous) or the count
 * exceeds 65535. */
int64_t dg_k_grouped_packed_sf_rows(const int *ks, int num_groups);

/* Number of SMs the persistent kernels use (default: all SMs of the current
 * device).  n <= 0 restores the default. */
void dg_set_num_sms(int n);
int dg_get_num_sms(void);

/* Time limit of every bounded device wait, in milliseconds (default 2000). */
void dg_set_wait_timeout_ms(int ms);

/* Diagnostics.  DG_DEBUG_DROP_ONE_LOAD makes the first CTA of the next GEMM
 * launch skip its first operand load, so its consumer's bounded wait runs
 * out and DG_DEV_TIMEOUT is reported (used by the failure-detection test;
 * the flag clears itself after one launch).  DG_DEBUG_PRINT_CONFIGS prints
 * the chosen tile configuration of each GEMM to stderr.  DG_DEBUG_SINGLE_CTA
 * runs dense GEMMs on single CTAs (128-row tiles) where CTA pairs (256-row
 * tiles) would be chosen; results are bit-identical either way.
 * DG_DEBUG_WIDE_PAIR makes 256-row pair GEMMs without C use 384-column tiles
 * (two MMAs per K step), whatever the tile chooser would pick. */
enum { DG_DEBUG_DROP_ONE_LOAD = 1, DG_DEBUG_PRINT_CONFIGS = 2, DG_DEBUG_SINGLE_CTA = 4, DG_DEBUG_WIDE_PAIR = 8 };
/* Environment, read once per process (tuning and diagnostics only; results are
 * the same for every choice): DG_BLOCK_N forces the single-CTA kernel's tile
 * width, DG_PAIR_BLOCK_N the 256-row pair kernel's, DG_SKINNY_PAIR_BLOCK_N the
 * 128-row pair kernel's for dense GEMMs with m <= 128 and no C (32, 64, 96 or
 * 128; a negative value keeps them on single CTAs), and DG_PRINT_CONFIGS
 * prints each GEMM's tile configuration to stderr.  A DG_PAIR_BLOCK_N width
 * that is not compiled in makes pair launches return DG_ERR_UNSUPPORTED; a
 * DG_BLOCK_N width that is not compiled in is ignored (128 is used), and so
 * is a DG_SKINNY_PAIR_BLOCK_N width (the single-CTA kernel is used). */
void dg_set_debug_flags(uint32_t flags);

/* Human-readable name of a dg_status value. */
const char *dg_status_string(int status);

/* Tile configuration the last GEMM call on this thread launched:
 * out[0]=BLOCK_M, out[1]=BLOCK_N, out[2]=stages, out[3]=grid size,
 * out[4]=kernel kind (0 block-scaled, 1 FP32-promotion, 2 block-scaled on
 * CTA pairs), out[5]=number of
 * kernel launches of that call. */
void dg_get_last_config(int out[6]);

#ifdef __cplusplus
}
#endif

#endif /* DG_GB300_H */
