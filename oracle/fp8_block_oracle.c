/*
 * CPU oracle for the W8A8 block-FP8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. The parity tests, the smoke check and the
 * bench's CPU-baseline leg are the only users; the product path never
 * loads this library, and it shares no code, header or table with the
 * CUDA kernels.
 *
 * What it computes (the layer the dual-L20 Qwen3.8-27B-FP8 tuning report
 * calls "W8A8 Block FP8", section 8; the single-RTX-PRO-6000 Qwen3.8-27B
 * optimisation post's "Marlin skips the activation quantisation" in its
 * single-request section implies that this default path quantises the
 * activations at run time). The pages do not spell out the arithmetic; the
 * plainest reading, used here, is:
 *
 *   activation groups 1x128, weight blocks 128x128, G = 128;
 *   s = amax / 448 in fp32 (448 = largest finite E4M3), s = 1 when amax = 0;
 *   code = E4M3(x / s): one IEEE fp32 division, then round to nearest,
 *          ties to even, saturating to +-448, sign of zero kept;
 *   y[m][n] = sum_kb sa[m][kb] * sw[n/G][kb] * sum_{k in kb} dq(q[m][k]) dq(w[n][k]);
 *   out = bf16(y), rounded to nearest even straight from the fp64 value.
 *
 * Every finite E4M3 value is an integer multiple of 2^-9, so each block dot
 * is computed exactly as an int64 sum of (value * 2^9) products and scaled
 * by 2^-18; the scales and the sum over blocks are applied in fp64. The
 * result is the definition up to fp64 rounding (relative ~1e-15), far
 * tighter than any fp32 kernel.
 *
 * Parity of every function here is pinned by tests that do not reuse this
 * file's arithmetic: the E4M3 table against torch's float8_e4m3fn decoder
 * and the format's closed-form landmarks, the encoder against torch's
 * converter and hand-derived ties, the quantisers against exact rational
 * checks, and the GEMM against exact Fraction brute force, one-hot inputs,
 * scale linearity and K permutation. The weight-only GEMM is pinned by
 * Fraction brute force, by its exact reduction to the W8A8 GEMM when the
 * activations are quantised values times powers of two, and by an fp64
 * dequantise-then-matmul.
 *
 * Built with gcc -O2 -fopenmp (no fast-math: IEEE fp32 division and no
 * flush-to-zero are part of the definition).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define G 128
#define E4M3_MAX 448.0f

/* Status codes returned by the entry points. */
#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE 1      /* a size < 0, or K not a multiple of 128 */
#define ORACLE_ERR_NONFINITE 2  /* a NaN or infinite input value          */
#define ORACLE_ERR_NAN_CODE 3   /* an E4M3 NaN code (0x7F / 0xFF) in a GEMM input */

static float e4m3_value[256];
static int32_t e4m3_int[256]; /* value * 2^9, exact for the finite codes */
static int table_ready = 0;

/*
 * E4M3 ("fn" variant: no infinities) decoded from its bit fields:
 * sign = bit 7, exponent e = bits 6..3 (bias 7), mantissa m = bits 2..0.
 * e = 0 encodes subnormals m * 2^-9; otherwise (1 + m/8) * 2^(e-7).
 * The all-ones pattern S.1111.111 is NaN, so the largest finite value is
 * 1.75 * 2^8 = 448 (code 0x7E).
 */
static void build_table(void) {
    if (table_ready) return;
    for (int c = 0; c < 256; ++c) {
        int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
        double v;
        if (e == 0xF && m == 7) {
            v = NAN;
        } else if (e == 0) {
            v = ldexp((double)m, -9);
        } else {
            v = ldexp(1.0 + m / 8.0, e - 7);
        }
        if (s) v = -v;
        e4m3_value[c] = (float)v;
        e4m3_int[c] = isnan(v) ? 0 : (int32_t)ldexp(v, 9);
    }
    table_ready = 1;
}

void oracle_e4m3_table(float out[256]) {
    build_table();
    memcpy(out, e4m3_value, sizeof(e4m3_value));
}

/*
 * Round-to-nearest-even, saturating E4M3 encode of a finite fp32 value.
 * The non-negative finite codes 0x00..0x7E are strictly increasing in value,
 * so the code below |f| is found by bisection over the table; the two
 * neighbours' midpoint (exact in fp64: at most 5 significant bits) decides,
 * and an exact tie goes to the code whose mantissa LSB (bit 0) is 0.
 */
uint8_t oracle_e4m3_encode(float f) {
    build_table();
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    float a = fabsf(f);
    if (a >= E4M3_MAX) return sign | 0x7E; /* satfinite */
    int lo = 0x00, hi = 0x7E;               /* value[lo] <= a < value[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (e4m3_value[mid] <= a) lo = mid; else hi = mid;
    }
    double mid = 0.5 * ((double)e4m3_value[lo] + (double)e4m3_value[hi]);
    int code;
    if ((double)a < mid) code = lo;
    else if ((double)a > mid) code = hi;
    else code = (lo & 1) ? hi : lo;
    return (uint8_t)(sign | code);
}

void oracle_e4m3_encode_array(const float* f, int64_t n, uint8_t* out) {
    build_table();
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(f[i]);
}

static float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/*
 * Quantise one group given by a row-major sub-matrix: rows r0..r1-1,
 * columns c0..c0+G-1 of a [rows, ld] bf16 matrix.
 * amax = max |x| (exact in fp32), s = amax / 448 (one fp32 division),
 * s = 1 if amax = 0, code = E4M3(x / s) with one fp32 division per element.
 */
static int quant_group(const uint16_t* x, int64_t ld, int64_t r0, int64_t r1, int64_t c0,
                       uint8_t* q, float* scale_out) {
    float amax = 0.0f;
    for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c0 + G; ++c) {
            float v = bf16_to_float(x[r * ld + c]);
            if (!isfinite(v)) return ORACLE_ERR_NONFINITE;
            float av = fabsf(v);
            if (av > amax) amax = av;
        }
    float s = (amax == 0.0f) ? 1.0f : amax / E4M3_MAX;
    for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c0 + G; ++c) {
            float v = bf16_to_float(x[r * ld + c]);
            float t = v / s;
            q[r * ld + c] = oracle_e4m3_encode(t);
        }
    *scale_out = s;
    return ORACLE_OK;
}

/*
 * Activation quantisation, one scale per token and 128-wide K group:
 * x bf16 [M, K] (raw uint16 bits, row-major) -> q E4M3 [M, K], sa fp32 [M, K/128].
 */
int oracle_act_quant(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, float* sa) {
    if (M < 0 || K < 0 || K % G) return ORACLE_ERR_SHAPE;
    build_table();
    int64_t KB = K / G;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t kb = 0; kb < KB; ++kb) {
            int st = quant_group(x, K, m, m + 1, kb * G, q, &sa[m * KB + kb]);
            if (st != ORACLE_OK) {
#pragma omp atomic write
                status = st;
            }
        }
    return status;
}

/*
 * Weight quantisation, one scale per 128x128 block:
 * W bf16 [N, K] -> w E4M3 [N, K], sw fp32 [ceil(N/128), K/128].
 * A partial block at the N edge uses the rows that exist.
 */
int oracle_weight_quant(const uint16_t* W, int64_t N, int64_t K, uint8_t* w, float* sw) {
    if (N < 0 || K < 0 || K % G) return ORACLE_ERR_SHAPE;
    build_table();
    int64_t KB = K / G, NB = (N + G - 1) / G;
    int status = ORACLE_OK;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb)
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t r1 = (nb + 1) * G < N ? (nb + 1) * G : N;
            int st = quant_group(W, K, nb * G, r1, kb * G, w, &sw[nb * KB + kb]);
            if (st != ORACLE_OK) {
#pragma omp atomic write
                status = st;
            }
        }
    return status;
}

/*
 * bf16 rounding of an fp64 value, to nearest with ties to even, taken in one
 * step from fp64 (no intermediate fp32 rounding). bf16 keeps 8 significant
 * bits and fp32's exponent range: the quantum at y is 2^(e-8) where
 * 2^(e-1) <= |y| < 2^e, and never below 2^-133 (bf16 subnormals).
 */
uint16_t oracle_bf16_from_double(double y) {
    if (y == 0.0) return signbit(y) ? 0x8000 : 0x0000;
    int e;
    frexp(y, &e);
    int qe = e - 8;
    if (qe < -133) qe = -133;
    double r = ldexp(nearbyint(ldexp(y, -qe)), qe);
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/*
 * Block-scaled GEMM for the listed output rows (rows == NULL: all M rows).
 * Inputs: q E4M3 [M, K], sa fp32 [M, K/128], w E4M3 [N, K], sw fp32
 * [ceil(N/128), K/128], all row-major. For each listed row index i (row
 * m = rows[i]) and each n it writes, at [i, n]:
 *   y     = sum_kb sa*sw*P_kb*2^-18 in fp64, with P_kb the exact int64 block dot;
 *   aabs  = sum_kb |sa*sw*P_kb*2^-18| (the size of the terms, for error floors);
 *   out   = bf16 bits of y (nearest even).
 * Any of y / aabs / out may be NULL.
 */
int oracle_block_gemm_rows(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw,
                           int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                           double* y, double* aabs, uint16_t* out) {
    if (M < 0 || N < 0 || K < 0 || K % G || nrows < 0) return ORACLE_ERR_SHAPE;
    build_table();
    int64_t KB = K / G;
    if (rows == NULL) nrows = M;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        if (m < 0 || m >= M) return ORACLE_ERR_SHAPE;
        for (int64_t k = 0; k < K; ++k)
            if ((q[m * K + k] & 0x7F) == 0x7F) return ORACLE_ERR_NAN_CODE;
    }
    for (int64_t i = 0; i < N * K; ++i)
        if ((w[i] & 0x7F) == 0x7F) return ORACLE_ERR_NAN_CODE;

#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < nrows; ++i)
        for (int64_t n = 0; n < N; ++n) {
            int64_t m = rows ? rows[i] : i;
            const uint8_t* qr = q + m * K;
            const uint8_t* wr = w + n * K;
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                int64_t P = 0;
                for (int64_t k = kb * G; k < (kb + 1) * G; ++k)
                    P += (int64_t)e4m3_int[qr[k]] * (int64_t)e4m3_int[wr[k]];
                double scale = (double)sa[m * KB + kb] * (double)sw[(n / G) * KB + kb];
                double term = scale * ldexp((double)P, -18);
                acc += term;
                acc_abs += fabs(term);
            }
            if (y) y[i * N + n] = acc;
            if (aabs) aabs[i * N + n] = acc_abs;
            if (out) out[i * N + n] = oracle_bf16_from_double(acc);
        }
    return ORACLE_OK;
}

int oracle_block_gemm(const uint8_t* q, const float* sa, const uint8_t* w, const float* sw,
                      int64_t M, int64_t N, int64_t K, double* y, double* aabs, uint16_t* out) {
    return oracle_block_gemm_rows(q, sa, w, sw, M, N, K, NULL, 0, y, aabs, out);
}

/*
 * Weight-only block-FP8 GEMM (W8A16) for the listed output rows: the same
 * E4M3 weights and 128x128 block scales, multiplied by the bf16 activations
 * themselves, with no activation quantisation. This is the job of the
 * weight-only FP8 back-end (Marlin) that the single-RTX-PRO-6000
 * Qwen3.8-27B optimisation post chooses at one request, section "单并发优化",
 * because it skips the activation quantisation. The pages give no formula;
 * the plain reading is the dequantised product:
 *   y[m][n] = sum_kb sw[n/G][kb] * sum_{k in kb} x[m][k] * dq(w[n][k]).
 * x is bf16 bits [M, K]; w, sw, rows, y, aabs, out as in
 * oracle_block_gemm_rows (aabs = sum_kb |sw * block dot|). Each product
 * bf16 * E4M3 has at most 12 significant bits, so the fp64 block dot is
 * exact while one block's products span less than 2^41 in magnitude (true
 * of every test input); the block scales and the sum over blocks are fp64.
 */
int oracle_block_gemm_w8a16_rows(const uint16_t* x, const uint8_t* w, const float* sw, int64_t M, int64_t N,
                                 int64_t K, const int64_t* rows, int64_t nrows, double* y, double* aabs,
                                 uint16_t* out) {
    if (M < 0 || N < 0 || K < 0 || K % G || nrows < 0) return ORACLE_ERR_SHAPE;
    build_table();
    int64_t KB = K / G;
    if (rows == NULL) nrows = M;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        if (m < 0 || m >= M) return ORACLE_ERR_SHAPE;
        for (int64_t k = 0; k < K; ++k)
            if (!isfinite(bf16_to_float(x[m * K + k]))) return ORACLE_ERR_NONFINITE;
    }
    for (int64_t i = 0; i < N * K; ++i)
        if ((w[i] & 0x7F) == 0x7F) return ORACLE_ERR_NAN_CODE;

#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < nrows; ++i)
        for (int64_t n = 0; n < N; ++n) {
            int64_t m = rows ? rows[i] : i;
            const uint16_t* xr = x + m * K;
            const uint8_t* wr = w + n * K;
            const float* sw_row = sw + (n / G) * KB; /* scales of this row's 128-row weight block */
            double sum = 0.0, sum_abs = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                double dot = 0.0;
                for (int64_t k = kb * G; k < (kb + 1) * G; ++k)
                    dot += (double)bf16_to_float(xr[k]) * (double)e4m3_value[wr[k]];
                double t = (double)sw_row[kb] * dot;
                sum += t;
                sum_abs += fabs(t);
            }
            if (y) y[i * N + n] = sum;
            if (aabs) aabs[i * N + n] = sum_abs;
            if (out) out[i * N + n] = oracle_bf16_from_double(sum);
        }
    return ORACLE_OK;
}

/* Threads the OpenMP loops use (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
