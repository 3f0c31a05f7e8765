/*
 * dtc_oracle.c -- plain, slow, obviously correct CPU oracle for the dense GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's CPU-baseline leg
 * load this file's shared library; the CUDA library never calls it, and the two share no
 * source, header, table or helper.
 *
 * What it computes -- the plain definition, written out, with one rounding at the end:
 *
 *   16-bit operands (bf16 or fp16):
 *     C[m,n] = round_out( sum_{k<K} dec(A[m,k]) * dec(Bop[k,n]) )
 *     "NT": B is stored [N,K] and Bop[k,n] = B[n,k]
 *           (TileLang SM100 Support (Preview), "Code Example": B is (N, K) and the gemm uses
 *            trans_B=True; "Compilation and Usage": ref_c = (a.float() @ b.T.float()).to(bf16))
 *     "NN": B is stored [K,N] and Bop[k,n] = B[k,n]
 *           (tilelang (velog), section 1.1 Front-End DSL: B is T.Tensor((K, N)) and
 *            T.gemm(A_shared, B_shared, C_local) with no transpose)
 *     "TN", "TT": as "NN", "NT", with A stored [K,M] and Aop[m,k] = A[k,m] (the first letter is
 *           A's transpose flag, the second B's: the trans_A / trans_B arguments of T.gemm in
 *           TileLang SM100 Support (Preview), "Current Limitations" and "Code Example");
 *           for "NT"/"NN" Aop[m,k] = A[m,k] with A stored [M,K]
 *
 *   MXFP8 block-scaled (both operands e4m3, one E8M0 scale per row per 128 K-elements,
 *   "1d1d" granularity 128 for A and B:
 *   05 Blackwell TCGEN05 GEMM tutorial, section "Advanced (not implemented here)",
 *   gemm_blockscaled with sf_a_granularity_k = sf_b_granularity_k = 128):
 *     C[m,n] = round_bf16( sum_k  e4m3(A[m,k]) * 2^(sfA[m,k/128]-127)
 *                               * e4m3(B[n,k]) * 2^(sfB[n,k/128]-127) )
 *   and the "other block-scaled formats" of the same section read as the OCP MX family the
 *   instruction supports: each operand e4m3, e5m2, e2m3, e3m2 or e2m1, and scale blocks of g =
 *   128 or 32 K-elements (the OCP MX block size), E8M0 scales [rows, ceil(K/g)]; and NVFP4:
 *   e2m1 operands with one UE4M3 scale per 16 K-elements:
 *     C[m,n] = round_bf16( sum_k  fa(A[m,k]) * sa(sfA[m,k/g]) * fb(B[n,k]) * sb(sfB[n,k/g]) )
 *
 * Accumulation is in double. Every product of two bf16/fp16/e4m3 values, times powers of two
 * from the scales, is exact in double; only the sum carries rounding error, which for the
 * sizes used (K <= 8192, |terms| < 2^20) is below 1e-10 relative -- far inside the pages'
 * rtol = atol = 1e-2. The single final rounding is IEEE round-to-nearest-even straight from
 * double to the output format (never double -> float -> 16-bit, which would round twice).
 *
 * Format definitions used by the codecs:
 *   bf16  : the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent, 7 fraction bits).
 *   fp16  : IEEE binary16 (1, 5, 10; bias 15; subnormals; exponent 31 = inf/NaN).
 *   e4m3  : OCP FP8 E4M3 "fn" variant (1, 4, 3; bias 7; no infinities; S.1111.111 = NaN;
 *           largest finite 448; subnormals m/8 * 2^-6).
 *   e5m2  : OCP FP8 E5M2 (1, 5, 2; bias 15; exponent 31 = inf (m = 0) / NaN; subnormals
 *           m/4 * 2^-14; largest finite 57344).
 *   E8M0  : unsigned 8-bit exponent, value 2^(e-127); 0xFF = NaN.
 *   The OCP MX element formats below fp8 (OCP Microscaling Formats (MX) v1.0; none has
 *   infinities or NaNs):
 *   e2m3  : FP6 (1, 2, 3; bias 1; subnormals m/8; largest 7.5).
 *   e3m2  : FP6 (1, 3, 2; bias 3; subnormals m/16; largest 28).
 *   e2m1  : FP4 (1, 2, 1; bias 1; subnormal 0.5; largest 6).
 *   UE4M3 : the scale of NVFP4 (one per 16 elements): an e4m3 code with the sign bit clear.
 *
 * Packed storage of the sub-byte formats: a row of K elements of b bits (b = 4 or 6) is read as a
 * little-endian bit stream, element k in bits [b*k, b*k + b) (fp4: byte k/2, the low nibble for
 * even k; fp6: 4 elements in 3 bytes). A row of fp8 codes is one byte per element.
 *
 *   2:4 structured-sparse A (gemm_sp; 05 Blackwell TCGEN05 GEMM tutorial, "An API-level note",
 *   which names the sparse GEMM among the exported forms without defining it; read as the 2:4
 *   pattern along K): of every group of 4 consecutive K-elements of a row of A, two values are
 *   stored, vals [M, K/2] (16-bit, the group's two values in order), and the group's two
 *   positions (0..3) in meta [M, K/8] bytes: group g's nibble sits at bits 4*(g % 2) of byte g/2,
 *   its bits 0-1 the position of vals[m, 2g] and bits 2-3 that of vals[m, 2g+1]:
 *     C[m,n] = round_out( sum_g sum_{j<2} dec(vals[m,2g+j]) * dec(Bop[4g + pos_j(m,g), n]) )
 *   with Bop as for the dense product ("NT" or "NN"). The two positions of a group differ in the
 *   2:4 pattern; the sum above is defined either way.
 *
 * Degenerate sizes: M == 0 or N == 0 computes nothing; K == 0 gives the empty sum, +0.
 *
 * Threads: rows of C are split across POSIX threads, one per requested worker; the
 * arithmetic for each output element is identical whatever the split.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define DTC_ORACLE_BF16 0
#define DTC_ORACLE_F16 1
#define DTC_ORACLE_NT 0
#define DTC_ORACLE_NN 1
#define DTC_ORACLE_TN 2
#define DTC_ORACLE_TT 3

/* A stored [K,M] (transposed)? B stored [K,N]? */
static int a_is_km(int layout) { return layout == DTC_ORACLE_TN || layout == DTC_ORACLE_TT; }
static int b_is_kn(int layout) { return layout == DTC_ORACLE_NN || layout == DTC_ORACLE_TN; }
static int layout_ok(int layout) { return layout >= DTC_ORACLE_NT && layout <= DTC_ORACLE_TT; }

/* ------------------------------------------------------------------------------------------ */
/* Decoders: code -> exact double value                                                        */
/* ------------------------------------------------------------------------------------------ */

double dtc_oracle_dec_bf16(uint16_t h) {
    /* bf16 is the top half of a binary32: widen and reinterpret. */
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

double dtc_oracle_dec_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

double dtc_oracle_dec_e4m3(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int m = b & 0x7;
    double v;
    if (e == 15 && m == 7) {
        return NAN; /* the only NaN encodings: S.1111.111 */
    } else if (e == 0) {
        v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
    } else {
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

double dtc_oracle_dec_e5m2(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1f;
    int m = b & 0x3;
    double v;
    if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -16); /* subnormal: m/4 * 2^-14 */
    } else {
        v = ldexp((double)(4 + m), e - 17); /* (1 + m/4) * 2^(e-15) */
    }
    return sign ? -v : v;
}

double dtc_oracle_dec_e8m0(uint8_t b) {
    if (b == 0xff) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* FP6 E2M3: sign bit 5, exponent bits 3-4 (bias 1), mantissa bits 0-2. */
double dtc_oracle_dec_e2m3(uint8_t c) {
    int sign = (c >> 5) & 1;
    int e = (c >> 3) & 0x3;
    int m = c & 0x7;
    double v = e == 0 ? ldexp((double)m, -3)            /* subnormal: m/8 * 2^(1-1) */
                      : ldexp((double)(8 + m), e - 4);  /* (1 + m/8) * 2^(e-1) */
    return sign ? -v : v;
}

/* FP6 E3M2: sign bit 5, exponent bits 2-4 (bias 3), mantissa bits 0-1. */
double dtc_oracle_dec_e3m2(uint8_t c) {
    int sign = (c >> 5) & 1;
    int e = (c >> 2) & 0x7;
    int m = c & 0x3;
    double v = e == 0 ? ldexp((double)m, -4)            /* subnormal: m/4 * 2^(1-3) */
                      : ldexp((double)(4 + m), e - 5);  /* (1 + m/4) * 2^(e-3) */
    return sign ? -v : v;
}

/* FP4 E2M1: sign bit 3, exponent bits 1-2 (bias 1), mantissa bit 0. */
double dtc_oracle_dec_e2m1(uint8_t c) {
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int m = c & 0x1;
    double v = e == 0 ? ldexp((double)m, -1)            /* subnormal: m/2 * 2^(1-1) */
                      : ldexp((double)(2 + m), e - 2);  /* (1 + m/2) * 2^(e-1) */
    return sign ? -v : v;
}

/* UE4M3 (NVFP4 scale): an e4m3 code whose sign bit must be clear; NaN otherwise. */
double dtc_oracle_dec_ue4m3(uint8_t b) {
    if (b & 0x80) return NAN;
    return dtc_oracle_dec_e4m3(b);
}

/* ------------------------------------------------------------------------------------------ */
/* Encoders: double -> nearest representable code, ties to even, one rounding                  */
/* ------------------------------------------------------------------------------------------ */

/* Round x to a binary format with p significand bits (implicit bit included), smallest normal
 * exponent emin and largest finite value maxfin. Returns the rounded value as a double (exact:
 * every value of these formats is a double), +-inf on overflow. x must be finite. */
static double round_to_format(double x, int p, int emin, double maxfin) {
    if (x == 0.0) return x;
    int e;
    frexp(fabs(x), &e); /* |x| = f * 2^e with 0.5 <= f < 1, so the leading bit is 2^(e-1) */
    int lead = e - 1;
    if (lead < emin) lead = emin; /* subnormal range keeps the smallest normal's quantum */
    int qexp = lead - (p - 1);    /* weight of the last significand bit */
    double scaled = ldexp(x, -qexp);       /* exact: a power-of-two scaling */
    double r = nearbyint(scaled);          /* default mode: round half to even */
    double y = ldexp(r, qexp);
    if (fabs(y) > maxfin) return x > 0 ? INFINITY : -INFINITY;
    return y;
}

uint16_t dtc_oracle_enc_bf16(double x) {
    if (isnan(x)) return 0x7fc0;
    double y = isinf(x) ? x : round_to_format(x, 8, -126, ldexp(255.0, 120)); /* max (2-2^-7)*2^127 */
    /* y is a bf16 value, hence exactly a binary32 value: its top 16 bits are the code. */
    float f = (float)y;
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(w >> 16);
}

uint16_t dtc_oracle_enc_f16(double x) {
    if (isnan(x)) return 0x7e00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isinf(x)) return sign | 0x7c00;
    double y = round_to_format(x, 11, -14, 65504.0);
    if (isinf(y)) return sign | 0x7c00;
    double a = fabs(y);
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14)) {
        /* subnormal: a = m * 2^-24, 1 <= m <= 1023 */
        return sign | (uint16_t)ldexp(a, 24);
    }
    int e;
    double f = frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> (2f) * 2^(e-1) */
    int biased = (e - 1) + 15;
    uint16_t mant = (uint16_t)(ldexp(f, 11) - 1024.0); /* (2f - 1) * 1024, exact */
    return sign | (uint16_t)(biased << 10) | mant;
}

/* ------------------------------------------------------------------------------------------ */
/* 16-bit GEMM                                                                                 */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    const double* a;  /* decoded A, [M][K] */
    const double* bt; /* decoded Bop, gathered as [N][K] so that Bop[k][n] = bt[n*K + k] */
    int64_t M, N, K;
    int dtype;        /* output format */
    uint16_t* c;      /* [M][N] codes, may be NULL */
    double* s;        /* [M][N] unrounded sums, may be NULL */
    int64_t row0, row1;
} gemm_job;

static void* gemm_rows(void* arg) {
    gemm_job* j = (gemm_job*)arg;
    for (int64_t m = j->row0; m < j->row1; ++m) {
        const double* arow = j->a + m * j->K;
        for (int64_t n = 0; n < j->N; ++n) {
            const double* brow = j->bt + n * j->K;
            double acc = 0.0;
            for (int64_t k = 0; k < j->K; ++k) acc += arow[k] * brow[k];
            if (j->s) j->s[m * j->N + n] = acc;
            if (j->c)
                j->c[m * j->N + n] =
                    j->dtype == DTC_ORACLE_F16 ? dtc_oracle_enc_f16(acc) : dtc_oracle_enc_bf16(acc);
        }
    }
    return NULL;
}

static int run_rows(gemm_job* proto, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((int64_t)nthreads > proto->M) nthreads = (int)(proto->M > 0 ? proto->M : 1);
    pthread_t tids[1024];
    int joined[1024];
    gemm_job jobs[1024];
    int64_t per = (proto->M + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].row0 = t * per < proto->M ? t * per : proto->M;
        jobs[t].row1 = (t + 1) * per < proto->M ? (t + 1) * per : proto->M;
    }
    for (int t = 1; t < nthreads; ++t) {
        joined[t] = pthread_create(&tids[t], NULL, gemm_rows, &jobs[t]) == 0;
        if (!joined[t]) gemm_rows(&jobs[t]); /* could not start a thread: do that share here */
    }
    gemm_rows(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joined[t]) pthread_join(tids[t], NULL);
    return 0;
}

static double dec16(int dtype, uint16_t h) {
    return dtype == DTC_ORACLE_F16 ? dtc_oracle_dec_f16(h) : dtc_oracle_dec_bf16(h);
}

/* Decode Aop to [M][K] doubles and Bop to [N][K] doubles (a gather, no arithmetic). */
static int decode16(int dtype, int layout, const uint16_t* A, const uint16_t* B, int64_t M,
                    int64_t N, int64_t K, double** a_out, double** bt_out) {
    double* a = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double* bt = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a || !bt) {
        free(a);
        free(bt);
        return -1;
    }
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            a[m * K + k] = dec16(dtype, a_is_km(layout) ? A[k * M + m] : A[m * K + k]);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            bt[n * K + k] = dec16(dtype, b_is_kn(layout) ? B[k * N + n] : B[n * K + k]);
    *a_out = a;
    *bt_out = bt;
    return 0;
}

/* Full C. Returns 0 on success, -1 on bad arguments or out of memory. */
int dtc_oracle_gemm16(int dtype, int layout, const uint16_t* A, const uint16_t* B, int64_t M,
                      int64_t N, int64_t K, uint16_t* C, double* S, int nthreads) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (dtype != DTC_ORACLE_BF16 && dtype != DTC_ORACLE_F16) return -1;
    if (!layout_ok(layout)) return -1;
    if (M == 0 || N == 0) return 0;
    double *a, *bt;
    if (decode16(dtype, layout, A, B, M, N, K, &a, &bt) != 0) return -1;
    gemm_job proto = {a, bt, M, N, K, dtype, C, S, 0, 0};
    run_rows(&proto, nthreads);
    free(a);
    free(bt);
    return 0;
}

/* Selected outputs only: out[i] = C[rows[i], cols[i]] (and its unrounded sum). Used at sizes
 * where the full product would take the oracle too long. Decodes only what it touches. */
int dtc_oracle_gemm16_sampled(int dtype, int layout, const uint16_t* A, const uint16_t* B,
                              int64_t M, int64_t N, int64_t K, const int64_t* rows,
                              const int64_t* cols, int64_t count, uint16_t* Cout, double* Sout) {
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    if (dtype != DTC_ORACLE_BF16 && dtype != DTC_ORACLE_F16) return -1;
    if (!layout_ok(layout)) return -1;
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = rows[i], n = cols[i];
        if (m < 0 || m >= M || n < 0 || n >= N) return -1;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            uint16_t a = a_is_km(layout) ? A[k * M + m] : A[m * K + k];
            uint16_t b = b_is_kn(layout) ? B[k * N + n] : B[n * K + k];
            acc += dec16(dtype, a) * dec16(dtype, b);
        }
        if (Sout) Sout[i] = acc;
        if (Cout) Cout[i] = dtype == DTC_ORACLE_F16 ? dtc_oracle_enc_f16(acc) : dtc_oracle_enc_bf16(acc);
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* 2:4 structured-sparse A                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* Position (0..3) of stored value j (0 or 1) of group g of a row of metadata. */
static int sp_position(const uint8_t* meta_row, int64_t g, int j) {
    uint8_t nib = (uint8_t)((meta_row[g / 2] >> (4 * (g % 2))) & 0xf);
    return (nib >> (2 * j)) & 0x3;
}

/* Full C of the sparse product (layouts "NT" and "NN" for B). K must be a multiple of 4. */
int dtc_oracle_gemm_sp(int dtype, int layout, const uint16_t* vals, const uint8_t* meta,
                       const uint16_t* B, int64_t M, int64_t N, int64_t K, uint16_t* C, double* S,
                       int nthreads) {
    if (M < 0 || N < 0 || K < 0 || K % 4) return -1;
    if (dtype != DTC_ORACLE_BF16 && dtype != DTC_ORACLE_F16) return -1;
    if (layout != DTC_ORACLE_NT && layout != DTC_ORACLE_NN) return -1;
    if (M == 0 || N == 0) return 0;
    /* Aop as a dense [M][K] array of doubles: each stored value added at its position. */
    double* a = (double*)calloc((size_t)(M * K > 0 ? M * K : 1), sizeof(double));
    double* bt = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a || !bt) {
        free(a);
        free(bt);
        return -1;
    }
    const int64_t mrow = (K / 4 + 1) / 2; /* metadata bytes per row */
    for (int64_t m = 0; m < M; ++m)
        for (int64_t g = 0; g < K / 4; ++g)
            for (int j = 0; j < 2; ++j)
                a[m * K + 4 * g + sp_position(meta + m * mrow, g, j)] +=
                    dec16(dtype, vals[m * (K / 2) + 2 * g + j]);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const uint16_t code = b_is_kn(layout) ? B[k * N + n] : B[n * K + k]; /* Bop[k][n] */
            bt[n * K + k] = dec16(dtype, code);
        }
    gemm_job proto = {a, bt, M, N, K, dtype, C, S, 0, 0};
    run_rows(&proto, nthreads);
    free(a);
    free(bt);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Block-scaled fp8 GEMM (NT: A [M,K], B [N,K], scales [rows, ceil(K/g)] E8M0)                   */
/* ------------------------------------------------------------------------------------------ */

#define DTC_ORACLE_E4M3 0
#define DTC_ORACLE_E5M2 1
#define DTC_ORACLE_E2M3 2
#define DTC_ORACLE_E3M2 3
#define DTC_ORACLE_E2M1 4
#define DTC_ORACLE_SF_E8M0 0
#define DTC_ORACLE_SF_UE4M3 1

/* Bits per element of an element format; 0 if unknown. */
int dtc_oracle_format_bits(int fmt) {
    switch (fmt) {
    case DTC_ORACLE_E4M3:
    case DTC_ORACLE_E5M2: return 8;
    case DTC_ORACLE_E2M3:
    case DTC_ORACLE_E3M2: return 6;
    case DTC_ORACLE_E2M1: return 4;
    default: return 0;
    }
}

/* Element k of a packed row (see the header comment): the b-bit field at bit b*k. */
static uint8_t row_code(const uint8_t* row, int bits, int64_t k) {
    if (bits == 8) return row[k];
    int64_t bit = k * bits;
    int64_t byte = bit / 8;
    int shift = (int)(bit % 8);
    unsigned v = row[byte];
    if (shift + bits > 8) v |= (unsigned)row[byte + 1] << 8; /* the field spans two bytes */
    return (uint8_t)((v >> shift) & ((1u << bits) - 1u));
}

static double dec_elem(int fmt, uint8_t c) {
    switch (fmt) {
    case DTC_ORACLE_E4M3: return dtc_oracle_dec_e4m3(c);
    case DTC_ORACLE_E5M2: return dtc_oracle_dec_e5m2(c);
    case DTC_ORACLE_E2M3: return dtc_oracle_dec_e2m3(c);
    case DTC_ORACLE_E3M2: return dtc_oracle_dec_e3m2(c);
    default: return dtc_oracle_dec_e2m1(c);
    }
}

static double dec_scale(int sf_kind, uint8_t c) {
    return sf_kind == DTC_ORACLE_SF_UE4M3 ? dtc_oracle_dec_ue4m3(c) : dtc_oracle_dec_e8m0(c);
}

static int bs_args_ok(int fmt_a, int fmt_b, int sf_kind, int block) {
    return dtc_oracle_format_bits(fmt_a) && dtc_oracle_format_bits(fmt_b) &&
           (sf_kind == DTC_ORACLE_SF_E8M0 || sf_kind == DTC_ORACLE_SF_UE4M3) &&
           (block == 16 || block == 32 || block == 128);
}

/* Bytes of one packed row of K elements. */
static int64_t row_bytes(int fmt, int64_t K) { return (K * dtc_oracle_format_bits(fmt) + 7) / 8; }

/* Decode one operand with its scales applied: out[r][k] = f(X[r,k]) * s(sf[r,k/g]). Exact in
 * double (a product of two values with at most 4 significant bits and a power of two, or of an
 * fp8 value and a power of two). */
static double* decode_scaled(int fmt, int sf_kind, int block, const uint8_t* X, const uint8_t* sf,
                             int64_t R, int64_t K) {
    int64_t kb = (K + block - 1) / block;
    int64_t rb = row_bytes(fmt, K);
    int bits = dtc_oracle_format_bits(fmt);
    double* out = (double*)malloc(sizeof(double) * (size_t)(R * K > 0 ? R * K : 1));
    if (!out) return NULL;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = dec_elem(fmt, row_code(X + r * rb, bits, k)) *
                             dec_scale(sf_kind, sf[r * kb + k / block]);
    return out;
}

/* General block-scaled product, NT: A [M,K] and B [N,K] as packed rows of their formats, scales
 * [rows, ceil(K/block)]. Output bf16 codes (and unrounded sums). */
int dtc_oracle_gemm_bs(int fmt_a, int fmt_b, int sf_kind, int block, const uint8_t* A,
                       const uint8_t* B, const uint8_t* sfA, const uint8_t* sfB, int64_t M,
                       int64_t N, int64_t K, uint16_t* C, double* S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || !bs_args_ok(fmt_a, fmt_b, sf_kind, block)) return -1;
    if (M == 0 || N == 0) return 0;
    double* a = decode_scaled(fmt_a, sf_kind, block, A, sfA, M, K);
    double* bt = decode_scaled(fmt_b, sf_kind, block, B, sfB, N, K);
    if (!a || !bt) {
        free(a);
        free(bt);
        return -1;
    }
    gemm_job proto = {a, bt, M, N, K, DTC_ORACLE_BF16, C, S, 0, 0};
    run_rows(&proto, nthreads);
    free(a);
    free(bt);
    return 0;
}

int dtc_oracle_gemm_bs_sampled(int fmt_a, int fmt_b, int sf_kind, int block, const uint8_t* A,
                               const uint8_t* B, const uint8_t* sfA, const uint8_t* sfB, int64_t M,
                               int64_t N, int64_t K, const int64_t* rows, const int64_t* cols,
                               int64_t count, uint16_t* Cout, double* Sout) {
    if (M < 0 || N < 0 || K < 0 || count < 0 || !bs_args_ok(fmt_a, fmt_b, sf_kind, block)) return -1;
    int64_t kb = (K + block - 1) / block;
    int64_t ra = row_bytes(fmt_a, K), rb = row_bytes(fmt_b, K);
    int ba = dtc_oracle_format_bits(fmt_a), bb = dtc_oracle_format_bits(fmt_b);
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = rows[i], n = cols[i];
        if (m < 0 || m >= M || n < 0 || n >= N) return -1;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double av = dec_elem(fmt_a, row_code(A + m * ra, ba, k)) *
                        dec_scale(sf_kind, sfA[m * kb + k / block]);
            double bv = dec_elem(fmt_b, row_code(B + n * rb, bb, k)) *
                        dec_scale(sf_kind, sfB[n * kb + k / block]);
            acc += av * bv;
        }
        if (Sout) Sout[i] = acc;
        if (Cout) Cout[i] = dtc_oracle_enc_bf16(acc);
    }
    return 0;
}

/* The fp8 members of the family (E8M0 scales, blocks of 32 or 128). */
int dtc_oracle_gemm_mx(int fmt_a, int fmt_b, int block, const uint8_t* A, const uint8_t* B,
                       const uint8_t* sfA, const uint8_t* sfB, int64_t M, int64_t N, int64_t K,
                       uint16_t* C, double* S, int nthreads) {
    if (fmt_a > DTC_ORACLE_E5M2 || fmt_b > DTC_ORACLE_E5M2 || block == 16) return -1;
    return dtc_oracle_gemm_bs(fmt_a, fmt_b, DTC_ORACLE_SF_E8M0, block, A, B, sfA, sfB, M, N, K,
                              C, S, nthreads);
}

int dtc_oracle_gemm_mx_sampled(int fmt_a, int fmt_b, int block, const uint8_t* A,
                               const uint8_t* B, const uint8_t* sfA, const uint8_t* sfB, int64_t M,
                               int64_t N, int64_t K, const int64_t* rows, const int64_t* cols,
                               int64_t count, uint16_t* Cout, double* Sout) {
    if (fmt_a > DTC_ORACLE_E5M2 || fmt_b > DTC_ORACLE_E5M2 || block == 16) return -1;
    return dtc_oracle_gemm_bs_sampled(fmt_a, fmt_b, DTC_ORACLE_SF_E8M0, block, A, B, sfA, sfB, M,
                                      N, K, rows, cols, count, Cout, Sout);
}

/* The pages' MXFP8 product: e4m3 x e4m3, scale blocks of 128. */
int dtc_oracle_gemm_mxfp8(const uint8_t* A, const uint8_t* B, const uint8_t* sfA,
                          const uint8_t* sfB, int64_t M, int64_t N, int64_t K, uint16_t* C,
                          double* S, int nthreads) {
    return dtc_oracle_gemm_mx(DTC_ORACLE_E4M3, DTC_ORACLE_E4M3, 128, A, B, sfA, sfB, M, N, K, C,
                              S, nthreads);
}

int dtc_oracle_gemm_mxfp8_sampled(const uint8_t* A, const uint8_t* B, const uint8_t* sfA,
                                  const uint8_t* sfB, int64_t M, int64_t N, int64_t K,
                                  const int64_t* rows, const int64_t* cols, int64_t count,
                                  uint16_t* Cout, double* Sout) {
    return dtc_oracle_gemm_mx_sampled(DTC_ORACLE_E4M3, DTC_ORACLE_E4M3, 128, A, B, sfA, sfB, M, N,
                                      K, rows, cols, count, Cout, Sout);
}

/* Host cores this process may use (what the oracle's default thread count is based on). */
int dtc_oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
