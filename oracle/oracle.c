/*
 * Oracle: plain, slow, CPU reference of the quantized GEMV / skinny GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the bench's CPU
 * baseline use it. It shares no code, header, table or constant with the CUDA
 * sources.
 *
 * Every floating-point result is computed in IEEE double from the exact values
 * of the fp16/bf16/E2M1/E8M0 inputs, except the block-32 Hadamard + int8 path,
 * whose integer codes are decided in fp32 (the precision both sides share).
 * Build without -ffast-math and with -ffp-contract=off so each fp32 operation
 * is a single correctly rounded IEEE operation.
 *
 * Sources (page title, section):
 *  [MLXR] "MLX Runner: An Inference Engine You Can Read",
 *         "Architecture: one command buffer per token": affine groups,
 *         weight = scale x code + bias, codes multiplied directly.
 *  [KRILL] "Krill Teardown", "Core mechanisms": one weight read serves many
 *         rows (skinny form).
 *  [K3]   "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin),
 *         "Technical approach / compute" (fused MXFP4 dequant + GEMV, E2M1
 *         16-entry table, E8M0 scale on the exponent) and "How it works"
 *         (router picks the top-16 experts per layer).
 *  [UZU]  Uzu article, "How Uzu optimizes bytes and tokens per pass":
 *         block-diagonal randomized Hadamard, 32-element blocks, random sign
 *         flips before mixing, 8-bit activations on the int8 matrix path.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* IEEE binary16 bit pattern -> double (sign, 5-bit exponent bias 15,
 * 10-bit fraction; exponent 0 = subnormal m * 2^-24). */
double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp(1024.0 + m, e - 25);
    return sign ? -v : v;
}

/* bfloat16 bit pattern -> float: the upper half of an IEEE binary32. */
static float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double oracle_bf16_to_double(uint16_t b) { return (double)bf16_to_float(b); }

/* ------------------------------------------------------------------------
 * W4A16 affine (MLXR): y[m][n] = sum_k (s[n][g] * q[n][k] + b[n][g]) * x[m][k]
 * with g = k / group, q = bits [4(k%8), 4(k%8)+3] of wq[n][k/8].
 * absdot[m][n] = sum_k |w[n][k] * x[m][k]| (the tolerance's scale).
 * One call covers the GEMV (M = 1) and the skinny form (M rows, KRILL).
 * ---------------------------------------------------------------------- */
void oracle_w4a16(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                  const uint16_t *x, int M, int N, int K, int group,
                  double *y, double *absdot, int nthreads) {
    set_threads(nthreads);
    const int words = K / 8, groups = K / group;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                uint32_t word = wq[(size_t)n * words + k / 8];
                int q = (int)((word >> (4 * (k % 8))) & 0xFu);
                double s = oracle_f16_to_double(scales[(size_t)n * groups + k / group]);
                double b = oracle_f16_to_double(biases[(size_t)n * groups + k / group]);
                double w = s * q + b;
                double xv = (double)bf16_to_float(x[(size_t)m * K + k]);
                acc += w * xv;
                aacc += fabs(w * xv);
            }
            y[(size_t)m * N + n] = acc;
            if (absdot) absdot[(size_t)m * N + n] = aacc;
        }
    }
}

/* ------------------------------------------------------------------------
 * Affine quantization at any of the widths MLXR lists (2, 3, 4, 5, 6 or 8
 * bits; groups of 32, 64 or 128): weight = scale x code + bias. The codes of
 * a row form one little-endian bit stream: code k occupies bits
 * [bits*k, bits*k + bits) of the row, bit j of the stream being bit j % 32 of
 * word j / 32 (for 4 bits this is the W4A16 layout above). K is a multiple
 * of 32 and of the group, so every row is a whole number of words
 * (K * bits / 32). y and absdot as in oracle_w4a16.
 * ---------------------------------------------------------------------- */
void oracle_affine(const uint32_t *wq, int bits, const uint16_t *scales, const uint16_t *biases,
                   const uint16_t *x, int M, int N, int K, int group, double *y, double *absdot,
                   int nthreads) {
    set_threads(nthreads);
    const size_t words = (size_t)K * bits / 32;
    const int groups = K / group;
    const uint32_t mask = (1u << bits) - 1u;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint32_t *row = wq + (size_t)n * words;
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                const size_t bit = (size_t)bits * k;
                uint64_t two = row[bit / 32];
                if (bit / 32 + 1 < words) two |= (uint64_t)row[bit / 32 + 1] << 32;
                const int q = (int)((two >> (bit % 32)) & mask);
                const double s = oracle_f16_to_double(scales[(size_t)n * groups + k / group]);
                const double b = oracle_f16_to_double(biases[(size_t)n * groups + k / group]);
                const double w = s * q + b;
                const double xv = (double)bf16_to_float(x[(size_t)m * K + k]);
                acc += w * xv;
                aacc += fabs(w * xv);
            }
            y[(size_t)m * N + n] = acc;
            if (absdot) absdot[(size_t)m * N + n] = aacc;
        }
    }
}

/* Same definition for a list of rows only (sampled checks at full size). */
void oracle_w4a16_rows(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                       const uint16_t *x, int M, int K, int group,
                       const int64_t *rows, int nrows, int64_t row_base,
                       double *y, double *absdot, int nthreads) {
    /* wq/scales/biases point at row row_base; y is [M][nrows] */
    set_threads(nthreads);
    const int words = K / 8, groups = K / group;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < nrows; ++r) {
        int64_t n = rows[r] - row_base;
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                uint32_t word = wq[(size_t)n * words + k / 8];
                int q = (int)((word >> (4 * (k % 8))) & 0xFu);
                double s = oracle_f16_to_double(scales[(size_t)n * groups + k / group]);
                double b = oracle_f16_to_double(biases[(size_t)n * groups + k / group]);
                double w = s * q + b;
                double xv = (double)bf16_to_float(x[(size_t)m * K + k]);
                acc += w * xv;
                aacc += fabs(w * xv);
            }
            y[(size_t)m * nrows + r] = acc;
            if (absdot) absdot[(size_t)m * nrows + r] = aacc;
        }
    }
}

/* ------------------------------------------------------------------------
 * MXFP4 (K3; value sets from the OCP MX v1.0 definition of E2M1 / E8M0).
 * E2M1 code: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Two codes per byte, the even element in the low nibble.
 * ---------------------------------------------------------------------- */
static const double E2M1_VALUE[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double oracle_e2m1(int code) { return E2M1_VALUE[code & 15]; }

double oracle_e8m0(int e) {
    if (e == 255) return NAN;
    return ldexp(1.0, e - 127);
}

static double mxfp4_weight(const uint8_t *codes, const uint8_t *scales, int C,
                           int64_t r, int c) {
    uint8_t byte = codes[(size_t)r * (C / 2) + c / 2];
    int code = (c & 1) ? (byte >> 4) : (byte & 15);
    return E2M1_VALUE[code] * oracle_e8m0(scales[(size_t)r * (C / 32) + c / 32]);
}

/* out[r] = sum_c W[r][c] * v[c]; absout[r] = sum_c |W[r][c] * v[c]|;
 * aw_out[r] = sum_c |W[r][c]| * wv[c] (optional, for error propagation). */
void oracle_mxfp4_gemv(const uint8_t *codes, const uint8_t *scales, int R, int C,
                       const double *v, const double *wv,
                       double *out, double *absout, double *aw_out, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        double acc = 0.0, aacc = 0.0, wacc = 0.0;
        for (int c = 0; c < C; ++c) {
            double w = mxfp4_weight(codes, scales, C, r, c);
            acc += w * v[c];
            aacc += fabs(w * v[c]);
            if (wv) wacc += fabs(w) * wv[c];
        }
        out[r] = acc;
        if (absout) absout[r] = aacc;
        if (aw_out) aw_out[r] = wacc;
    }
}

/* ------------------------------------------------------------------------
 * Block-32 randomized Hadamard + per-token symmetric int8 (UZU).
 * For each row m and 32-block b: v_j = x[m][32b+j] as fp32, negated where bit
 * j of sign_bits[b] is set; then the Walsh-Hadamard butterflies with spans
 * 1, 2, 4, 8, 16: for every pair (i, i+h) with bit h of i clear,
 * (a, c) -> (a + c, a - c), in fp32 (unnormalized H, entries +-1).
 * Then amax_m = max |z|, s_m = amax_m / 127 (fp32 division),
 * q = clamp(rint(z / s_m), -127, 127) with rint = round half to even;
 * amax_m = 0 gives s_m = 0 and q = 0.
 * z_out (optional) receives the transformed row in fp32.
 * ---------------------------------------------------------------------- */
void oracle_hadamard32(const float *in, const uint32_t *sign_bits, int K, float *z) {
    for (int b = 0; b < K / 32; ++b) {
        float v[32];
        for (int j = 0; j < 32; ++j) {
            float t = in[32 * b + j];
            v[j] = ((sign_bits[b] >> j) & 1u) ? -t : t;
        }
        for (int h = 1; h < 32; h *= 2) {
            for (int i = 0; i < 32; ++i) {
                if (i & h) continue;
                float a = v[i], c = v[i + h];
                v[i] = a + c;
                v[i + h] = a - c;
            }
        }
        for (int j = 0; j < 32; ++j) z[32 * b + j] = v[j];
    }
}

/* Per-token symmetric int8 of one transformed row z[K] (fp32 decisions). */
void oracle_quant_i8_row(const float *z, int K, int8_t *q, float *scale) {
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
        float a = fabsf(z[k]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    *scale = s;
    for (int k = 0; k < K; ++k) {
        int8_t code = 0;
        if (s > 0.0f) {
            float r = rintf(z[k] / s);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            code = (int8_t)r;
        }
        q[k] = code;
    }
}

void oracle_hadamard32_quant_i8(const uint16_t *x, const uint32_t *sign_bits, int M, int K,
                                int8_t *q, float *scale, float *z_out, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m) {
        float row[K > 0 ? K : 1], z[K > 0 ? K : 1];
        for (int k = 0; k < K; ++k) row[k] = bf16_to_float(x[(size_t)m * K + k]);
        oracle_hadamard32(row, sign_bits, K, z);
        oracle_quant_i8_row(z, K, q + (size_t)m * K, scale + m);
        if (z_out)
            for (int k = 0; k < K; ++k) z_out[(size_t)m * K + k] = z[k];
    }
}

/* ------------------------------------------------------------------------
 * W8A16 row-int8 GEMV (K3, "Technical approach / compute": the packed int8
 * output head, row-int8 weights with one scale per row, a weight-only
 * quantized matmul): y[m][n] = sum_k (s[n] * q[n][k]) * x[m][k], q int8,
 * s fp32, x bf16; absdot[m][n] = sum_k |w[n][k] * x[m][k]|.
 * ---------------------------------------------------------------------- */
void oracle_w8a16(const int8_t *wq, const float *scales, const uint16_t *x, int M, int N, int K,
                  double *y, double *absdot, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const double s = (double)scales[n];
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                const double w = s * (double)wq[(size_t)n * K + k];
                const double xv = (double)bf16_to_float(x[(size_t)m * K + k]);
                acc += w * xv;
                aacc += fabs(w * xv);
            }
            y[(size_t)m * N + n] = acc;
            if (absdot) absdot[(size_t)m * N + n] = aacc;
        }
    }
}

/* ------------------------------------------------------------------------
 * W8A8 int32 (UZU int8 matrix path): C[m][n] = sum_k a[m][k] * w[n][k],
 * accumulated in int64; returns 0 if every result fits in int32, else 1.
 * ---------------------------------------------------------------------- */
int oracle_w8a8(const int8_t *a, const int8_t *w, int M, int N, int K, int32_t *c,
                int nthreads) {
    set_threads(nthreads);
    int overflow = 0;
#pragma omp parallel for schedule(static) reduction(| : overflow)
    for (int n = 0; n < N; ++n) {
        for (int m = 0; m < M; ++m) {
            int64_t acc = 0;
            for (int k = 0; k < K; ++k)
                acc += (int64_t)a[(size_t)m * K + k] * (int64_t)w[(size_t)n * K + k];
            if (acc > INT32_MAX || acc < INT32_MIN) overflow = 1;
            c[(size_t)m * N + n] = (int32_t)acc;
        }
    }
    return overflow;
}
