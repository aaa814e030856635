/*
 * Oracle for the fine-grained block-scaled FP8 GEMM and its scale-factor layout.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously correct CPU
 * restatement of what the GEMM library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Sources (web pages on DeepGEMM and block-scaled quantised matmul):
 *   [P1] "02 · DeepGEMM 技术解析" (PaperTrace), sections 1.1, 2.1-2.2, 3.1-3.2, 5.1-5.2
 *   [P2] "DeepSeek V4 源码剖析 第13章 DeepGEMM", sections 13.3 (interface and
 *        algorithm pseudocode), 13.6 (grouped GEMM)
 *   [P3] "LinearQuant 分块量化矩阵乘法" (lryc.cn), the "what the operator does"
 *        section: expand the block scales to every element, then matmul.
 *
 * Arithmetic: every element of D is the fp64 sum over k of
 *     dec(A[m,k]) * sa[m, k/128]  *  dec(B[n,k]) * sb[n, k/128]
 * taken in increasing k, plus C[m,n] (decoded exactly from bf16), then rounded
 * ONCE, round-to-nearest-even, to bf16.  That is the plain definition of
 * D = C + A @ B^T with 1x128 (A) and 128x128 (B) scales [P1 1.1, P2 13.3,
 * P3]; the two-level promotion of [P1 2.2] is the same sum regrouped.
 *
 * Readings of points the pages leave open:
 *   - "FP8 e4m3" is the OCP E4M3 "fn" flavour (no infinities, S.1111.111 = NaN,
 *     max 448), the torch.float8_e4m3fn type the pages' example code uses [P2 13.11].
 *   - scale groups are fixed at 128 along K and, for B, 128 along N; the group
 *     of element k is k/128 (integer division), so a short last group exists
 *     when K % 128 != 0.
 *   - UE8M0 byte of an FP32 scale = (bits >> 23) & 0xff [P2 13.3]; the value
 *     of byte e is 2^(e-127), and 0xff is NaN [P1 3.1].
 *   - packed layout: 4 consecutive K-groups per int32, little-endian by K
 *     index; MN-major with stride align(mn, 4) int32 per K-slice [P1 3.1];
 *     unused bytes of the last word and pad rows are written 0.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (no -ffast-math: the fp64 sums must
 * be taken in the order written).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits.  Exponent field 0 encodes subnormals m/8 * 2^-6.  Exponent 15 with
 * mantissa 7 is NaN; there is no infinity, so 0x7e (= 448) is the maximum. */
double orc_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xf;
    int m = code & 0x7;
    double v;
    if (e == 0xf && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* OCP MX FP4 E2M1 (the weights' type of the FP8 x FP4 GEMM [P2 13.5]): 1 sign
 * bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0 encodes the
 * subnormal m/2.  No infinity and no NaN: the magnitudes are 0, 0.5, 1, 1.5, 2,
 * 3, 4 and 6.  Only the low 4 bits of `code` are read. */
double orc_e2m1_decode(uint8_t code) {
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return sign ? -v : v;
}

/* UE8M0: 8-bit unsigned exponent, no mantissa, no sign; 2^(e-127); 0xff is
 * NaN [P1 3.1]. */
double orc_ue8m0_decode(uint8_t e) {
    if (e == 0xff) return NAN;
    return ldexp(1.0, (int)e - 127);
}

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* The UE8M0 byte kept when an FP32 scale is packed: its 8 exponent bits
 * [P2 13.3, ">> 23"].  The mantissa and the sign are dropped, so 0.75 -> 0.5
 * and 3 -> 2 (the page's own example). */
uint8_t orc_fp32_to_ue8m0(float s) { return (uint8_t)((f32_bits(s) >> 23) & 0xffu); }

/* A scale is exactly representable as UE8M0 only when it is a positive power
 * of two with a normal exponent: sign 0 and mantissa 0 [P1 3.1, the
 * "(value & 0x807fffff) == 0" assertion]. */
int orc_fp32_is_exact_ue8m0(float s) { return (f32_bits(s) & 0x807fffffu) == 0u; }

double orc_bf16_decode(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value once to bf16 (1 sign, 8 exponent, 7 mantissa bits),
 * round-to-nearest, ties-to-even; overflow goes to +-inf.  Done by scaling
 * to the bf16 quantum of the value's binade (an exact power-of-two scaling),
 * rounding to an integer with nearbyint (default mode = nearest-even), and
 * scaling back. */
uint16_t orc_bf16_from_double(double x) {
    if (isnan(x)) return 0x7fc0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7f80);
    int e;
    (void)frexp(a, &e);       /* a in [2^(e-1), 2^e) */
    int binade = e - 1;
    if (binade < -126) binade = -126; /* subnormals share the quantum 2^-133 */
    double quantum = ldexp(1.0, binade - 7);
    double q = nearbyint(a / quantum);
    double r = q * quantum;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7f80);
    float f = (float)r; /* exact: r has at most 8 significant bits */
    return (uint16_t)(sign | (uint16_t)(f32_bits(f) >> 16));
}

/* ------------------------------------------------------------------------ */
/* Scale-factor layout transform [P1 3.1-3.2, P2 13.3]                      */
/* ------------------------------------------------------------------------ */

static int64_t align4(int64_t x) { return (x + 3) / 4 * 4; }

/*
 * sf:   FP32 [batch][mn_rows][sf_k] row-major; row r covers MN rows
 *       r*gran_mn .. r*gran_mn+gran_mn-1 (gran_mn = 1 for 1x128 activation
 *       scales, 128 for 128x128 weight blocks); the output is broadcast to one
 *       row per MN index (gran_mn becomes 1 [P1 3.2]).
 * out_fmt 1 (packed UE8M0): int32 out[batch][psf_k][align4(mn)],
 *       psf_k = ceil(sf_k/4); byte j of word (b, p, i) is the UE8M0 byte of
 *       K-group 4p+j of MN row i; bytes past sf_k and rows i >= mn are 0.
 * out_fmt 0 (FP32 MN-major): float out[batch][sf_k][align4(mn)], pad 0.
 * Returns the number of scales that were not exact powers of two (they are
 * truncated to their exponent in the packed output).
 */
int64_t orc_transform_sf(const float *sf, int batch, int mn_rows, int sf_k, int gran_mn,
                         int mn, int out_fmt, void *out) {
    int64_t stride = align4(mn);
    int psf_k = (sf_k + 3) / 4;
    int64_t inexact = 0;
    for (int b = 0; b < batch; b++) {
        const float *sfb = sf + (int64_t)b * mn_rows * sf_k;
        if (out_fmt == 1) {
            uint32_t *o = (uint32_t *)out + (int64_t)b * psf_k * stride;
            for (int p = 0; p < psf_k; p++)
                for (int64_t i = 0; i < stride; i++) {
                    uint32_t word = 0;
                    if (i < mn) {
                        int r = (int)(i / gran_mn);
                        for (int j = 0; j < 4; j++) {
                            int k = 4 * p + j;
                            if (k >= sf_k) break;
                            float s = sfb[(int64_t)r * sf_k + k];
                            word |= (uint32_t)orc_fp32_to_ue8m0(s) << (8 * j);
                        }
                    }
                    o[(int64_t)p * stride + i] = word;
                }
        } else {
            float *o = (float *)out + (int64_t)b * sf_k * stride;
            for (int k = 0; k < sf_k; k++)
                for (int64_t i = 0; i < stride; i++)
                    o[(int64_t)k * stride + i] =
                        i < mn ? sfb[(int64_t)(i / gran_mn) * sf_k + k] : 0.0f;
        }
        /* count inexact scales once per input element, not per broadcast row */
        for (int64_t r = 0; r < (int64_t)mn_rows * sf_k; r++)
            if (!orc_fp32_is_exact_ue8m0(sfb[r])) inexact++;
    }
    return inexact;
}

/* Decode a packed MN-major UE8M0 tensor back to fp64 scales
 * out[batch][mn][sf_k] (the inverse view of orc_transform_sf). */
void orc_unpack_sf(const uint32_t *packed, int batch, int mn, int sf_k, double *out) {
    int64_t stride = align4(mn);
    int psf_k = (sf_k + 3) / 4;
    for (int b = 0; b < batch; b++)
        for (int i = 0; i < mn; i++)
            for (int k = 0; k < sf_k; k++) {
                uint32_t word = packed[(int64_t)b * psf_k * stride + (int64_t)(k / 4) * stride + i];
                uint8_t byte = (uint8_t)(word >> (8 * (k % 4)));
                out[((int64_t)b * mn + i) * sf_k + k] = orc_ue8m0_decode(byte);
            }
}

/* Expand 128x128 block scales sb[ceil(N/128)][sf_k] to one row per N index:
 * out[n][kb] = sb[n/128][kb] ([P3]: the scale table is spread over the rows
 * it covers before the matmul). */
void orc_expand_block_rows(const double *sb, int n_rows, int sf_k, double *out) {
    for (int n = 0; n < n_rows; n++)
        for (int k = 0; k < sf_k; k++) out[(int64_t)n * sf_k + k] = sb[(int64_t)(n / 128) * sf_k + k];
}

/* ------------------------------------------------------------------------ */
/* GEMM: D = C + A @ B^T with per-element expanded scales [P2 13.3, P3]     */
/* ------------------------------------------------------------------------ */

/* One output element before rounding: C + sum_k a(m,k) * b(n,k), where
 * a(m,k) = dec(A[m,k]) * sa[m][k/128] and b(n,k) = dec(B[n,k]) * sb[n][k/128].
 * sa is [.][sf_k] for row m, sb is [.][sf_k] for row n (already one row per
 * N index). */
static double dot_element(int K, const uint8_t *arow, const double *sarow, const uint8_t *brow,
                          const double *sbrow, double c) {
    double s = 0.0;
    for (int k = 0; k < K; k++) {
        double a = orc_e4m3_decode(arow[k]) * sarow[k / 128];
        double b = orc_e4m3_decode(brow[k]) * sbrow[k / 128];
        s += a * b;
    }
    return c + s;
}

/*
 * Full GEMM with FP32 C and D (the FP32-output form; same sum as
 * orc_gemm_nt): D[m][n] = fp32_rne(C[m][n] + sum), the products summed in
 * fp64 from 0 in increasing k, then C added (0 if C is NULL), one rounding to
 * FP32 (C's double -> float conversion rounds to nearest even).
 */
void orc_gemm_nt_f32(int M, int N, int K, const uint8_t *A, int64_t lda, const double *sa,
                     const uint8_t *B, int64_t ldb, const double *sb, const float *C, int64_t ldc,
                     float *D, int64_t ldd, int nthreads) {
    int sf_k = (K + 127) / 128;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            double c = C ? (double)C[(int64_t)m * ldc + n] : 0.0;
            double v = dot_element(K, A + (int64_t)m * lda, sa + (int64_t)m * sf_k,
                                   B + (int64_t)n * ldb, sb + (int64_t)n * sf_k, c);
            D[(int64_t)m * ldd + n] = (float)v;
        }
    }
}

/*
 * The FP32-output GEMM with scales every gk elements of K instead of 128 (the
 * K-grouped layout's scales at a K granularity of 32 [P1 3.3]): sa is
 * [M][ceil(K/gk)] (row m, group k/gk), sb is [N][ceil(K/gk)].  Otherwise as
 * orc_gemm_nt_f32: the products summed in fp64 from 0 in increasing k, then C
 * added (0 if NULL), one rounding to FP32.
 */
static double dot_element_gk(int K, int gk, const uint8_t *arow, const double *sarow, const uint8_t *brow,
                             const double *sbrow, double c) {
    double s = 0.0;
    for (int k = 0; k < K; k++) {
        double a = orc_e4m3_decode(arow[k]) * sarow[k / gk];
        double b = orc_e4m3_decode(brow[k]) * sbrow[k / gk];
        s += a * b;
    }
    return c + s;
}

void orc_gemm_nt_f32_gk(int M, int N, int K, int gk, const uint8_t *A, int64_t lda, const double *sa,
                        const uint8_t *B, int64_t ldb, const double *sb, const float *C, int64_t ldc,
                        float *D, int64_t ldd, int nthreads) {
    int sf_k = (K + gk - 1) / gk;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            double c = C ? (double)C[(int64_t)m * ldc + n] : 0.0;
            double v = dot_element_gk(K, gk, A + (int64_t)m * lda, sa + (int64_t)m * sf_k,
                                      B + (int64_t)n * ldb, sb + (int64_t)n * sf_k, c);
            D[(int64_t)m * ldd + n] = (float)v;
        }
    }
}

/* The fp64 product sums (no C, no rounding) of orc_gemm_nt_f32_gk at a list of
 * (row, col) pairs. */
void orc_gemm_nt_gk_pre_sampled(int K, int gk, const uint8_t *A, int64_t lda, const double *sa,
                                const uint8_t *B, int64_t ldb, const double *sb, int64_t nsamples,
                                const int64_t *rows, const int64_t *cols, double *pre, int nthreads) {
    int sf_k = (K + gk - 1) / gk;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (int64_t i = 0; i < nsamples; i++) {
        int64_t m = rows[i], n = cols[i];
        pre[i] = dot_element_gk(K, gk, A + m * lda, sa + m * sf_k, B + n * ldb, sb + n * sf_k, 0.0);
    }
}

/*
 * Full GEMM, NT layout [P2 13.3]: A [M][lda] (K contiguous), B [N][ldb] (K
 * contiguous), sa [M][sf_k], sb [N][sf_k] (per row), C bf16 [M][ldc] or NULL,
 * D bf16 [M][ldd].  pre (optional, [M][N]) receives the fp64 value before
 * the bf16 rounding.  Rows are split across threads; each element's sum is
 * independent of the split.
 */
void orc_gemm_nt(int M, int N, int K, const uint8_t *A, int64_t lda, const double *sa,
                 const uint8_t *B, int64_t ldb, const double *sb, const uint16_t *C, int64_t ldc,
                 uint16_t *D, int64_t ldd, double *pre, int nthreads) {
    int sf_k = (K + 127) / 128;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            double c = C ? orc_bf16_decode(C[(int64_t)m * ldc + n]) : 0.0;
            double v = dot_element(K, A + (int64_t)m * lda, sa + (int64_t)m * sf_k,
                                   B + (int64_t)n * ldb, sb + (int64_t)n * sf_k, c);
            if (pre) pre[(int64_t)m * N + n] = v;
            D[(int64_t)m * ldd + n] = orc_bf16_from_double(v);
        }
    }
}

/* The same elements computed one by one for a list of (row, col) pairs, so
 * that large problems can be checked on samples. */
void orc_gemm_nt_sampled(int K, const uint8_t *A, int64_t lda, const double *sa,
                         const uint8_t *B, int64_t ldb, const double *sb, const uint16_t *C,
                         int64_t ldc, int64_t nsamples, const int64_t *rows, const int64_t *cols,
                         uint16_t *out, double *pre, int nthreads) {
    int sf_k = (K + 127) / 128;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (int64_t i = 0; i < nsamples; i++) {
        int64_t m = rows[i], n = cols[i];
        double c = C ? orc_bf16_decode(C[m * ldc + n]) : 0.0;
        double v = dot_element(K, A + m * lda, sa + m * sf_k, B + n * ldb, sb + n * sf_k, c);
        if (pre) pre[i] = v;
        out[i] = orc_bf16_from_double(v);
    }
}

/*
 * FP8 x FP4 GEMM [P2 13.1 (reason 2), 13.5]: FP8 activations times FP4 weights
 * whose scales run along K with one per 32 elements.
 *   A  E4M3 [M][lda], sa [M][ceil(K/128)] (the activations' 1x128 scales);
 *   B  E2M1 packed two per byte, row n at B + n*ldb bytes: element k of the row
 *      is byte k/2, low nibble for even k, high nibble for odd k;
 *   sb [N][ceil(K/32)]: one scale per row and 32 consecutive K.
 * D[m][n] = bf16_rne(C[m][n] + sum_k dec(A[m,k]) sa[m][k/128] * dec(B[n,k]) sb[n][k/32]),
 * the sum in fp64 in increasing k (C decoded exactly, 0 if NULL).
 */
static double dot_element_fp4(int K, const uint8_t *arow, const double *sarow, const uint8_t *brow,
                              const double *sbrow, double c) {
    double s = 0.0;
    for (int k = 0; k < K; k++) {
        uint8_t byte = brow[k / 2];
        uint8_t code = (k % 2 == 0) ? (uint8_t)(byte & 0xf) : (uint8_t)(byte >> 4);
        double a = orc_e4m3_decode(arow[k]) * sarow[k / 128];
        double b = orc_e2m1_decode(code) * sbrow[k / 32];
        s += a * b;
    }
    return c + s;
}

void orc_gemm_fp8_fp4_nt(int M, int N, int K, const uint8_t *A, int64_t lda, const double *sa,
                         const uint8_t *B, int64_t ldb, const double *sb, const uint16_t *C, int64_t ldc,
                         uint16_t *D, int64_t ldd, double *pre, int nthreads) {
    int sfa_k = (K + 127) / 128, sfb_k = (K + 31) / 32;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            double c = C ? orc_bf16_decode(C[(int64_t)m * ldc + n]) : 0.0;
            double v = dot_element_fp4(K, A + (int64_t)m * lda, sa + (int64_t)m * sfa_k, B + (int64_t)n * ldb,
                                       sb + (int64_t)n * sfb_k, c);
            if (pre) pre[(int64_t)m * N + n] = v;
            D[(int64_t)m * ldd + n] = orc_bf16_from_double(v);
        }
    }
}

/* The same elements one by one for a list of (row, col) pairs. */
void orc_gemm_fp8_fp4_nt_sampled(int K, const uint8_t *A, int64_t lda, const double *sa, const uint8_t *B,
                                 int64_t ldb, const double *sb, int64_t nsamples, const int64_t *rows,
                                 const int64_t *cols, uint16_t *out, int nthreads) {
    int sfa_k = (K + 127) / 128, sfb_k = (K + 31) / 32;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (int64_t i = 0; i < nsamples; i++) {
        int64_t m = rows[i], n = cols[i];
        double v = dot_element_fp4(K, A + m * lda, sa + m * sfa_k, B + n * ldb, sb + n * sfb_k, 0.0);
        out[i] = orc_bf16_from_double(v);
    }
}

/*
 * M-grouped GEMM, contiguous layout [P1 5.1, P2 13.6]: the experts' rows are
 * concatenated along M; grouped_layout[m] is the expert of row m, or -1 for a
 * padding row (left untouched in D).  B is [E][N][ldb], sb [E][N][sf_k].
 */
void orc_m_grouped_contiguous(int M, int N, int K, int num_groups, const uint8_t *A, int64_t lda,
                              const double *sa, const uint8_t *B, int64_t ldb, const double *sb,
                              const int32_t *grouped_layout, uint16_t *D, int64_t ldd,
                              int nthreads) {
    int sf_k = (K + 127) / 128;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int m = 0; m < M; m++) {
        int g = grouped_layout[m];
        if (g < 0 || g >= num_groups) continue;
        const uint8_t *Bg = B + (int64_t)g * N * ldb;
        const double *sbg = sb + (int64_t)g * N * sf_k;
        for (int n = 0; n < N; n++) {
            double v = dot_element(K, A + (int64_t)m * lda, sa + (int64_t)m * sf_k,
                                   Bg + (int64_t)n * ldb, sbg + (int64_t)n * sf_k, 0.0);
            D[(int64_t)m * ldd + n] = orc_bf16_from_double(v);
        }
    }
}

/*
 * M-grouped GEMM, masked layout [P1 5.2, P2 13.6]: A [E][max_m][K], D
 * [E][max_m][N]; only rows m < masked_m[e] of expert e are computed and
 * written; the rest of D is left untouched.
 */
void orc_m_grouped_masked(int num_groups, int max_m, int N, int K, const uint8_t *A,
                          const double *sa, const uint8_t *B, const double *sb,
                          const int32_t *masked_m, uint16_t *D, int nthreads) {
    int sf_k = (K + 127) / 128;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
#endif
    for (int e = 0; e < num_groups; e++) {
        for (int m = 0; m < max_m; m++) {
            if (m >= masked_m[e]) continue;
            int64_t row = (int64_t)e * max_m + m;
            const uint8_t *Be = B + (int64_t)e * N * K;
            const double *sbe = sb + (int64_t)e * N * sf_k;
            for (int n = 0; n < N; n++) {
                double v = dot_element(K, A + row * K, sa + row * sf_k, Be + (int64_t)n * K,
                                       sbe + (int64_t)n * sf_k, 0.0);
                D[row * N + n] = orc_bf16_from_double(v);
            }
        }
    }
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
