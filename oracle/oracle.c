/*
 * oracle.c -- plain CPU oracle for the scaled FP8 / BF16 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only tests/, __graft_entry__.smoke() and the CPU-baseline / reference arm
 * of bench.py load it.  It shares no code, header, table or helper with the
 * CUDA library (fp8_scaled_gemm_sm_gb300/csrc) and includes none of it.
 *
 * What it computes (the plain definition, everything in binary64):
 *
 *   ptpc        R[m,n] = ( sum_k e4m3(A[m,k]) * e4m3(B[n,k]) ) * sa[m] * sb[n]
 *   blockscale  R[m,n] = sum_j ( sum_{k in block j} e4m3(A)*e4m3(B) )
 *                               * sa[j][m] * sb[n/128][j]          (128-wide K blocks)
 *   mxfp8       R[m,n] = sum_j ( sum_{k in block j} e4m3(A)*e4m3(B) )
 *                               * e8m0(sa[j][m]) * e8m0(sb[j][n])  (32-wide K blocks)
 *   bf16        R[m,n] = sum_k bf16(A[m,k]) * bf16(B[n,k])
 *   ref[m,n]    = bf16 round-to-nearest-even of R[m,n], rounded once from binary64.
 *
 * Sources (web pages, read for what the method computes):
 *  - ROCm/mori PR 785 "fix(gemm-ar): drain the peeled tail's producers", Test
 *    section and cost table: the scaled GEMM in ptpc / blockscale / mxfp8
 *    modes, checked element-wise against a bf16-rounded fp32 reference.
 *  - ROCm/aiter PR 6539, Test Plan: the reference function
 *    run_torch(xq, wq, x_scale, w_scale, dtype=bf16), i.e. dequantise, multiply,
 *    scale, round to bf16.
 *  - ROCm/mori PR 809 "Using it": A [M,K] fp8 with a per-row scale, the weight
 *    shard B [N,K] with a per-output-channel scale, bf16 result [M,N]; "Not done
 *    yet": the blockscale / mxfp8 A scale is K-block major.
 *  - deepseek-ai/DeepGEMM PR 453, Reproduction: the plain BF16 GEMM with fp32
 *    accumulation, [4096,1024] x [1024,896].
 * Where the pages are silent (fp8 flavour, block geometry, scale layouts,
 * rounding mode) the readings are the ones listed in the repository's design
 * notes: e4m3fn (OCP OFP8, bias 7, no infinities, S.1111.111 = NaN, max 448);
 * e8m0 = 2^(b-127), 255 = NaN; 1x128 activation / 128x128 weight fp32 blocks;
 * 32-element e8m0 blocks; round-to-nearest-even to bf16.
 *
 * Exactness: every e4m3 x e4m3 product has at most 8 significant bits and lies
 * in [2^-18, 2^17.6], so a K-term binary64 sum is exact for K <= 2^16; the only
 * roundings in ptpc / mxfp8 are the scale products and the final bf16 rounding.
 *
 * Parity pins (all in tests/, run without a GPU): exhaustive decoder tables
 * against torch's float8 / bf16 conversions, bf16 rounding against an exact
 * rational search, integer-valued GEMMs against int64 sums, exact rational brute
 * force on tiny shapes in every mode, one-hot weights, scale invariants and a
 * float64 library matmul.  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define SGO_MODE_BF16 0
#define SGO_MODE_PTPC 1
#define SGO_MODE_BLOCKSCALE 2
#define SGO_MODE_MXFP8 3

/* ---- scalar decoders ------------------------------------------------------ */

/* e4m3fn (OCP OFP8): sign s, 4-bit exponent e (bias 7), 3-bit fraction f.
 * e == 0: subnormal f * 2^-9.  e == 15 && f == 7: NaN.  No infinities.      */
double sgo_dec_e4m3(uint8_t b) {
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int f = b & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp(1.0 + (double)f / 8.0, e - 7);
    return s ? -v : v;
}

/* e8m0 (OCP MX scale): an unsigned biased exponent, value 2^(b-127); 255 = NaN. */
double sgo_dec_e8m0(uint8_t b) {
    if (b == 255) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* bf16: the upper half of an IEEE binary32. */
double sgo_dec_bf16(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a binary64 value to bf16 (8 significant bits, 8 exponent bits, bias
 * 127, subnormals down to 2^-133) with round-to-nearest, ties to even, in one
 * step.  NaN -> 0x7FC0, overflow -> +-inf.                                   */
uint16_t sgo_bf16_rne(double x) {
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 63) << 15);
    int ex = (int)((bits >> 52) & 0x7FF);
    uint64_t frac = bits & ((1ULL << 52) - 1);
    if (ex == 0x7FF) return frac ? (uint16_t)0x7FC0 : (uint16_t)(sign | 0x7F80);
    if (ex == 0) return sign; /* zero or binary64 subnormal: far below 2^-134 */
    uint64_t sig = (1ULL << 52) | frac; /* |x| = sig * 2^(ex-1075) */
    int E = ex - 1023;                   /* |x| in [2^E, 2^(E+1)) */
    int qe = E - 7;                      /* bf16 quantum in this binade */
    if (qe < -133) qe = -133;            /* subnormal bf16 quantum */
    int shift = qe - (ex - 1075);        /* low bits of sig below the quantum */
    uint64_t n;
    if (shift >= 60) {
        n = 0; /* |x| < 2^(qe-6): rounds to zero */
    } else {
        n = sig >> shift;
        uint64_t rem = sig & ((1ULL << shift) - 1);
        uint64_t half = 1ULL << (shift - 1);
        if (rem > half || (rem == half && (n & 1))) n += 1;
    }
    double r = ldexp((double)n, qe); /* exact: n <= 256 */
    if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80);
    float f = (float)r; /* exact: r is a bf16 value */
    uint32_t fb;
    memcpy(&fb, &f, sizeof fb);
    return (uint16_t)(sign | (uint16_t)(fb >> 16));
}

/* ---- shape rules shared by the GEMM entry points ------------------------- */

static int sgo_block_k(int mode) {
    if (mode == SGO_MODE_BLOCKSCALE) return 128;
    if (mode == SGO_MODE_MXFP8) return 32;
    return 0;
}

static int sgo_check(int mode, int64_t M, int64_t N, int64_t K) {
    if (mode < 0 || mode > 3) return -1;
    if (M < 0 || N < 0 || K < 0) return -1;
    int bk = sgo_block_k(mode);
    if (bk && (K % bk) != 0) return -1;
    return 0;
}

static void sgo_decode_row(int mode, const void* X, int64_t row, int64_t K, double* out) {
    if (mode == SGO_MODE_BF16) {
        const uint16_t* p = (const uint16_t*)X + row * K;
        for (int64_t k = 0; k < K; ++k) out[k] = sgo_dec_bf16(p[k]);
    } else {
        const uint8_t* p = (const uint8_t*)X + row * K;
        for (int64_t k = 0; k < K; ++k) out[k] = sgo_dec_e4m3(p[k]);
    }
}

/* One output element from decoded rows a (row m of A) and b (row n of B). */
static double sgo_element(int mode, int64_t M, int64_t N, int64_t K, const double* a,
                          const double* b, const void* sa, const void* sb, int64_t m,
                          int64_t n) {
    if (mode == SGO_MODE_BF16) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];
        return s;
    }
    if (mode == SGO_MODE_PTPC) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];
        return s * (double)((const float*)sa)[m] * (double)((const float*)sb)[n];
    }
    int bk = sgo_block_k(mode);
    int64_t nblk = K / bk;
    double r = 0.0;
    for (int64_t j = 0; j < nblk; ++j) {
        double p = 0.0;
        for (int64_t k = j * bk; k < (j + 1) * bk; ++k) p += a[k] * b[k];
        double s_a, s_b;
        if (mode == SGO_MODE_BLOCKSCALE) {
            s_a = (double)((const float*)sa)[j * M + m];
            s_b = (double)((const float*)sb)[(n / 128) * nblk + j];
        } else {
            s_a = sgo_dec_e8m0(((const uint8_t*)sa)[j * M + m]);
            s_b = sgo_dec_e8m0(((const uint8_t*)sb)[j * N + n]);
        }
        r += p * s_a * s_b;
    }
    return r;
}

/* Rows [m_begin, m_end) of R and ref, each row N wide.  R may be NULL.
 * Returns 0, or -1 on a bad argument, -2 if memory runs out.                 */
int sgo_gemm_rows(int mode, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                  const void* sa, const void* sb, int64_t m_begin, int64_t m_end, double* R,
                  uint16_t* ref) {
    if (sgo_check(mode, M, N, K)) return -1;
    if (m_begin < 0 || m_end > M || m_begin > m_end) return -1;
    if (N == 0 || m_begin == m_end) return 0;
    double* Bd = (double*)malloc((size_t)(N * K > 0 ? N * K : 1) * sizeof(double));
    if (!Bd) return -2;
    for (int64_t n = 0; n < N; ++n) sgo_decode_row(mode, B, n, K, Bd + n * K);
    int failed = 0;
#pragma omp parallel
    {
        double* Ad = (double*)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!Ad) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t m = m_begin; m < m_end; ++m) {
                sgo_decode_row(mode, A, m, K, Ad);
                for (int64_t n = 0; n < N; ++n) {
                    double r = sgo_element(mode, M, N, K, Ad, Bd + n * K, sa, sb, m, n);
                    int64_t o = (m - m_begin) * N + n;
                    if (R) R[o] = r;
                    ref[o] = sgo_bf16_rne(r);
                }
            }
            free(Ad);
        }
    }
    free(Bd);
    return failed ? -2 : 0;
}

/* Individual elements (ms[i], ns[i]) for i < npts, computed one by one.
 * Used to check full-size outputs at sampled positions.                      */
int sgo_gemm_points(int mode, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                    const void* sa, const void* sb, int64_t npts, const int64_t* ms,
                    const int64_t* ns, double* R, uint16_t* ref) {
    if (sgo_check(mode, M, N, K)) return -1;
    for (int64_t i = 0; i < npts; ++i)
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double* a = (double*)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double* b = (double*)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!a || !b) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t i = 0; i < npts; ++i) {
                sgo_decode_row(mode, A, ms[i], K, a);
                sgo_decode_row(mode, B, ns[i], K, b);
                double r = sgo_element(mode, M, N, K, a, b, sa, sb, ms[i], ns[i]);
                if (R) R[i] = r;
                ref[i] = sgo_bf16_rne(r);
            }
        }
        free(a);
        free(b);
    }
    return failed ? -2 : 0;
}

/* Threads OpenMP would use for the calls above (reported with CPU timings). */
int sgo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- quantisation to e4m3 + scales (the step before the GEMM) -----------------
 *
 * ROCm/mori PR 809, "Using it": a_fp8, a_scale = quantize_per_token(x) -- the
 * activations are quantised per row (per token) before the ptpc GEMM; the
 * blockscale and mxfp8 modes take per-block scales (the same PR, "Not done yet":
 * the blockscale / mxfp8 A scale is K-block major).  Definition used here, for
 * a row segment (whole row, 128 or 32 elements) with amax = max |x|:
 *   ptpc / blockscale  s = fp32(amax / 448) (s = 1 if amax == 0);
 *                      q = e4m3_rne_satfinite(fp32(x / s))
 *   mxfp8              e = the least integer with amax <= 448 * 2^e (e = 0 if
 *                      amax == 0); code = clamp(e + 127, 0, 254); s = 2^(code-127);
 *                      q = e4m3_rne_satfinite(fp32(x / s))
 * fp32(.) is one IEEE round-to-nearest-even fp32 operation; e4m3_rne_satfinite
 * rounds to the nearest e4m3fn value (ties to even) and clamps to +-448.       */

/* Nearest e4m3fn code to the binary64 value v, ties to even, saturated to
 * +-448.  NaN -> 0x7F.                                                         */
uint8_t sgo_e4m3_rne_sat(double v) {
    if (v != v) return 0x7F;
    uint8_t sign = (uint8_t)(signbit(v) ? 0x80 : 0x00);
    double a = fabs(v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);              /* a in [2^(ex-1), 2^ex) */
    int E = ex - 1;             /* unbiased exponent of a */
    if (E < -6) E = -6;         /* subnormal range shares the 2^-9 quantum */
    double q = ldexp(1.0, E - 3);
    double n = a / q;           /* exact: q is a power of two */
    double fl = floor(n);
    double rem = n - fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = fl * q;          /* exact: fl <= 16 */
    if (r >= 448.0) return (uint8_t)(sign | 0x7E);
    if (r == 0.0) return sign;
    int ex2;
    frexp(r, &ex2);
    int E2 = ex2 - 1;
    if (E2 < -6) { /* subnormal: r = f * 2^-9, f in 1..7 */
        int f = (int)(r / ldexp(1.0, -9));
        return (uint8_t)(sign | f);
    }
    int f = (int)((r / ldexp(1.0, E2) - 1.0) * 8.0);
    return (uint8_t)(sign | ((E2 + 7) << 3) | f);
}

/* Least integer e with amax <= 448 * 2^e (amax > 0), by exact comparison. */
static int sgo_mx_exponent(double amax) {
    int e = ilogb(amax) - 8;
    while (448.0 * ldexp(1.0, e) < amax) ++e;
    while (448.0 * ldexp(1.0, e - 1) >= amax) --e;
    return e;
}

/* Quantise X [R][C] (x_is_bf16: uint16 bf16 bits, else float32) in `mode`
 * (1 ptpc, 2 blockscale 1x128, 3 mxfp8 1x32) into Q [R][C] e4m3 codes and
 * scales (ptpc float[R]; blockscale float[C/128][R]; mxfp8 uint8[C/32][R]).
 * Returns 0, or -1 on a bad argument.                                        */
int sgo_quantize(int mode, int x_is_bf16, int64_t R, int64_t C, const void* X, uint8_t* Q,
                 void* scale) {
    int64_t blk;
    if (mode == SGO_MODE_PTPC) blk = C;
    else if (mode == SGO_MODE_BLOCKSCALE) blk = 128;
    else if (mode == SGO_MODE_MXFP8) blk = 32;
    else return -1;
    if (R < 0 || C < 0 || (blk > 0 && C % blk != 0)) return -1;
    if (R == 0 || C == 0) return 0;
    int64_t nblk = C / blk;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t j = 0; j < nblk; ++j) {
            float amax = 0.0f;
            for (int64_t k = j * blk; k < (j + 1) * blk; ++k) {
                float x = x_is_bf16 ? (float)sgo_dec_bf16(((const uint16_t*)X)[r * C + k])
                                    : ((const float*)X)[r * C + k];
                float a = fabsf(x);
                if (a > amax) amax = a;
            }
            float s;
            if (mode == SGO_MODE_MXFP8) {
                int e = amax > 0.0f ? sgo_mx_exponent((double)amax) : 0;
                int code = e + 127;
                if (code < 0) code = 0;
                if (code > 254) code = 254;
                ((uint8_t*)scale)[j * R + r] = (uint8_t)code;
                s = (float)ldexp(1.0, code - 127);
            } else {
                volatile float num = amax, den = 448.0f;
                s = amax > 0.0f ? num / den : 1.0f;
                if (mode == SGO_MODE_PTPC)
                    ((float*)scale)[r] = s;
                else
                    ((float*)scale)[j * R + r] = s;
            }
            for (int64_t k = j * blk; k < (j + 1) * blk; ++k) {
                float x = x_is_bf16 ? (float)sgo_dec_bf16(((const uint16_t*)X)[r * C + k])
                                    : ((const float*)X)[r * C + k];
                volatile float y = x / s; /* one fp32 IEEE division */
                Q[r * C + k] = sgo_e4m3_rne_sat((double)y);
            }
        }
    }
    return 0;
}
