/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the ternary linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; it decodes the packed format with its own decoder written
 * from the format definition below.
 *
 * What it computes (Neutrino-1 8B model page, intro: every transformer linear
 * is stored bit-packed and decoded inside the matrix kernels; spec table:
 * gated (SwiGLU) feed-forward, three linears per layer; "Where the bytes
 * live": per-row metadata holds row dimensions, scales and row sums):
 *
 *   y[m][r] = scale[r] * sum_k t[r][k] * x[m][k]          t in {-1, 0, +1}
 *   h[m][r] = silu(g[m][r]) * u[m][r],  silu(z) = z / (1 + exp(-z))
 *   rowsum[r] = sum_k t[r][k]
 *
 * The page calls its real bit format proprietary and never specifies it, so
 * the format decoded here is this project's own 2-bit format:
 *   - a matrix of R rows and K columns (K a multiple of 64) is R*K/16 uint32
 *     words, row-major, K-contiguous: row r owns words [r*K/16, (r+1)*K/16);
 *   - column k of row r lives in word r*K/16 + k/16, at bits 2*(k%16) (low,
 *     "b0") and 2*(k%16)+1 (high, "b1"), least significant code first;
 *   - (b1,b0) = 00 -> 0, 01 -> +1, 11 -> -1; 10 is invalid.
 *
 * Arithmetic: every activation is widened from bf16 to double exactly, every
 * product t*x is exact, the sum over k runs in increasing k in double, and the
 * fp32 scale is applied in double.  No blocking, no reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define ORC_OK 0
#define ORC_BAD_VALUE (-1) /* int8 weight outside {-1,0,+1} */
#define ORC_BAD_SHAPE (-2) /* K not a multiple of 64, or negative sizes */
#define ORC_BAD_CODE (-3)  /* a 2-bit field holds the invalid pattern 10 */

/* Value of one 2-bit field, or 2 for the invalid pattern. */
static int orc_field_value(unsigned field)
{
    switch (field & 3u) {
    case 0u: return 0;
    case 1u: return 1;
    case 3u: return -1;
    default: return 2;
    }
}

/* The 2-bit field holding column k of row r. */
static unsigned orc_field(const uint32_t *codes, int64_t k_total, int64_t r, int64_t k)
{
    const int64_t words_per_row = k_total / 16;
    const uint32_t w = codes[r * words_per_row + k / 16];
    return (unsigned)((w >> (2 * (k % 16))) & 3u);
}

double orc_bf16_to_double(uint16_t bits)
{
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)bits << 16;
    return (double)v.f;
}

/* Encode int8 weights into the 2-bit format.  Returns ORC_OK or an error. */
int orc_pack(const int8_t *t, int64_t rows, int64_t k, uint32_t *codes)
{
    if (rows < 0 || k < 0 || k % 64 != 0) return ORC_BAD_SHAPE;
    const int64_t wpr = k / 16;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < wpr; ++i) {
            uint32_t w = 0;
            for (int64_t j = 0; j < 16; ++j) {
                const int v = t[r * k + i * 16 + j];
                uint32_t field;
                if (v == 0) field = 0u;
                else if (v == 1) field = 1u;
                else if (v == -1) field = 3u;
                else return ORC_BAD_VALUE;
                w |= field << (2 * j);
            }
            codes[r * wpr + i] = w;
        }
    }
    return ORC_OK;
}

/* Decode the whole matrix back to int8.  Returns ORC_OK or ORC_BAD_CODE. */
int orc_unpack(const uint32_t *codes, int64_t rows, int64_t k, int8_t *t)
{
    if (rows < 0 || k < 0 || k % 64 != 0) return ORC_BAD_SHAPE;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < k; ++c) {
            const int v = orc_field_value(orc_field(codes, k, r, c));
            if (v == 2) return ORC_BAD_CODE;
            t[r * k + c] = (int8_t)v;
        }
    }
    return ORC_OK;
}

/*
 * Per-row sums and code counts.  rowsum[r] = sum_k t[r][k] (int64 here; the
 * stored metadata is int32), counts = {zeros, plus, minus} over the matrix.
 */
int orc_stats(const uint32_t *codes, int64_t rows, int64_t k,
              int64_t *rowsum, int64_t counts[3])
{
    if (rows < 0 || k < 0 || k % 64 != 0) return ORC_BAD_SHAPE;
    counts[0] = counts[1] = counts[2] = 0;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t s = 0;
        for (int64_t c = 0; c < k; ++c) {
            const int v = orc_field_value(orc_field(codes, k, r, c));
            if (v == 2) return ORC_BAD_CODE;
            s += v;
            counts[v == 0 ? 0 : (v == 1 ? 1 : 2)] += 1;
        }
        rowsum[r] = s;
    }
    return ORC_OK;
}

/*
 * y[mi*rows + r] = scale[r] * sum_k t[r][k] * x[mi*k + k']  for rows in
 * [row_begin, row_end) and every activation row mi < m.  x holds bf16 bit
 * patterns.  An invalid field aborts with ORC_BAD_CODE.
 */
int orc_gemm(const uint32_t *codes, const float *scale, int64_t rows, int64_t k,
             const uint16_t *x, int64_t m, double *y,
             int64_t row_begin, int64_t row_end)
{
    if (rows < 0 || k < 0 || k % 64 != 0 || m < 0) return ORC_BAD_SHAPE;
    for (int64_t mi = 0; mi < m; ++mi) {
        for (int64_t r = row_begin; r < row_end; ++r) {
            double acc = 0.0;
            for (int64_t c = 0; c < k; ++c) {
                const int v = orc_field_value(orc_field(codes, k, r, c));
                if (v == 2) return ORC_BAD_CODE;
                acc += (double)v * orc_bf16_to_double(x[mi * k + c]);
            }
            y[mi * rows + r] = (double)scale[r] * acc;
        }
    }
    return ORC_OK;
}

/* silu(z) = z * sigmoid(z) = z / (1 + exp(-z)), in double. */
double orc_silu(double z)
{
    return z / (1.0 + exp(-z));
}

/*
 * Gated feed-forward activation: h = silu(gate) * up, where gate and up are
 * the two projections of the same activations, each with its own scale.
 */
int orc_swiglu(const uint32_t *gate_codes, const float *gate_scale,
               const uint32_t *up_codes, const float *up_scale,
               int64_t rows, int64_t k, const uint16_t *x, int64_t m, double *h,
               int64_t row_begin, int64_t row_end)
{
    if (rows < 0 || k < 0 || k % 64 != 0 || m < 0) return ORC_BAD_SHAPE;
    for (int64_t mi = 0; mi < m; ++mi) {
        for (int64_t r = row_begin; r < row_end; ++r) {
            double g = 0.0, u = 0.0;
            for (int64_t c = 0; c < k; ++c) {
                const int vg = orc_field_value(orc_field(gate_codes, k, r, c));
                const int vu = orc_field_value(orc_field(up_codes, k, r, c));
                if (vg == 2 || vu == 2) return ORC_BAD_CODE;
                const double xv = orc_bf16_to_double(x[mi * k + c]);
                g += (double)vg * xv;
                u += (double)vu * xv;
            }
            g *= (double)gate_scale[r];
            u *= (double)up_scale[r];
            h[mi * rows + r] = orc_silu(g) * u;
        }
    }
    return ORC_OK;
}

/*
 * RMSNorm ahead of a projection (Neutrino-1 8B model page, spec table:
 * RMSNorm with eps 1e-6 before the attention and feed-forward blocks, whose
 * first linears are q/k/v and gate/up).  For each activation row i the page
 * gives only the textbook operation
 *
 *     xn[i][k] = g[k] * x[i][k] / sqrt(mean_k x[i][k]^2 + eps)
 *
 * with a learned per-channel weight g (fp32 here).  The projection consumes
 * bf16 activations, so xn is rounded to bf16 once, and this project fixes
 * the precision of every step, because that rounding is a quantisation the
 * CUDA path must reach bit for bit:
 *   - the mean square in double, summing x^2 in increasing k (each bf16
 *     square is exact in double), divided by K;
 *   - the row factor r = 1 / sqrt(mean + eps) in double, rounded to fp32;
 *   - per element, fp32 products in this order: v = x * r, then g * v;
 *   - v rounded to bf16, round to nearest even (finite inputs).
 */
static uint16_t orc_float_to_bf16_rne(float f)
{
    union { float f; uint32_t u; } v;
    v.f = f;
    const uint32_t lsb = (v.u >> 16) & 1u;
    return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

int orc_rmsnorm(const uint16_t *x, const float *g, int64_t m, int64_t k, double eps,
                uint16_t *xn, float *r_out)
{
    if (m < 0 || k <= 0 || eps < 0.0) return ORC_BAD_SHAPE;
    for (int64_t mi = 0; mi < m; ++mi) {
        const uint16_t *xr = x + mi * k;
        double ss = 0.0;
        for (int64_t c = 0; c < k; ++c) {
            const double v = orc_bf16_to_double(xr[c]);
            ss += v * v;
        }
        const float r = (float)(1.0 / sqrt(ss / (double)k + eps));
        if (r_out) r_out[mi] = r;
        for (int64_t c = 0; c < k; ++c) {
            volatile float xv = (float)orc_bf16_to_double(xr[c]);
            volatile float v = xv * r;   /* fp32 product, rounded */
            volatile float w = g[c] * v; /* fp32 product, rounded */
            xn[mi * k + c] = orc_float_to_bf16_rne(w);
        }
    }
    return ORC_OK;
}

/*
 * The normalised projection: y = scale * (T @ rmsnorm(x)), i.e. orc_rmsnorm
 * followed by orc_gemm on its bf16 output, for rows [row_begin, row_end).
 * xn_scratch: m * k uint16 of caller memory.
 */
int orc_rmsnorm_gemm(const uint32_t *codes, const float *scale, int64_t rows, int64_t k,
                     const uint16_t *x, const float *g, double eps, int64_t m,
                     uint16_t *xn_scratch, double *y, int64_t row_begin, int64_t row_end)
{
    const int rc = orc_rmsnorm(x, g, m, k, eps, xn_scratch, (float *)0);
    if (rc != ORC_OK) return rc;
    return orc_gemm(codes, scale, rows, k, xn_scratch, m, y, row_begin, row_end);
}

/*
 * int8 LM head (Neutrino-1 8B model page, "Where the bytes live": the output
 * head is a 151,936 x 4,096 int8 matrix with per-row scales, read once per
 * generated token; the speculative-decoding paragraph: the verifier accepts
 * draft tokens greedily, i.e. by the argmax of each position's logits):
 *
 *     logit[m][r] = scale[r] * sum_k w[r][k] * x[m][k],   w int8, x bf16
 *
 * in double (every product is exact, the sum runs in increasing k), for rows
 * [row_begin, row_end).  abs_out (may be NULL) receives
 * scale[r] * sum_k |w[r][k] * x[m][k]|, the size an fp32 evaluation's
 * rounding error is measured against.
 */
int orc_i8_gemm(const int8_t *w, const float *scale, int64_t rows, int64_t k,
                const uint16_t *x, int64_t m, double *y, double *abs_out,
                int64_t row_begin, int64_t row_end)
{
    if (rows < 0 || k < 0 || m < 0) return ORC_BAD_SHAPE;
    for (int64_t mi = 0; mi < m; ++mi) {
        for (int64_t r = row_begin; r < row_end; ++r) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t c = 0; c < k; ++c) {
                const double p = (double)w[r * k + c] * orc_bf16_to_double(x[mi * k + c]);
                acc += p;
                aacc += fabs(p);
            }
            y[mi * rows + r] = (double)scale[r] * acc;
            if (abs_out) abs_out[mi * rows + r] = fabs((double)scale[r]) * aacc;
        }
    }
    return ORC_OK;
}

/*
 * Greedy choice per activation row: the index of the largest value of
 * y[mi][0..rows), the lowest index among equal maxima.  rows > 0.
 */
int orc_argmax(const double *y, int64_t m, int64_t rows, int64_t *idx)
{
    if (m < 0 || rows <= 0) return ORC_BAD_SHAPE;
    for (int64_t mi = 0; mi < m; ++mi) {
        int64_t best = 0;
        for (int64_t r = 1; r < rows; ++r)
            if (y[mi * rows + r] > y[mi * rows + best]) best = r;
        idx[mi] = best;
    }
    return ORC_OK;
}

/*
 * Denser packing (Neutrino-1 8B model page, "Where the bytes live" and the
 * "three doors" of the format discussion: the shipped lane spends more bits
 * per weight than a ternary value needs; SURVEY's next rows name base-3
 * packing).  This project's base-3 format, defined here and nowhere on the
 * pages:
 *   - a row of K weights (K a multiple of 80, padded with zero weights) is
 *     K/5 bytes; byte j holds weights 5j .. 5j+4;
 *   - byte value b = sum_{i<5} (t[5j+i] + 1) * 3^i  (least significant digit
 *     first), so b is in [0, 242]; bytes 243..255 are invalid;
 *   - 1.6 bits per weight against 2 for the 2-bit format.
 */
int orc_pack5(const int8_t *t, int64_t rows, int64_t k, uint8_t *codes)
{
    if (rows < 0 || k < 0 || k % 80 != 0) return ORC_BAD_SHAPE;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < k / 5; ++j) {
            unsigned b = 0, p = 1;
            for (int i = 0; i < 5; ++i) {
                const int v = t[r * k + 5 * j + i];
                if (v < -1 || v > 1) return ORC_BAD_VALUE;
                b += (unsigned)(v + 1) * p;
                p *= 3u;
            }
            codes[r * (k / 5) + j] = (uint8_t)b;
        }
    return ORC_OK;
}

int orc_unpack5(const uint8_t *codes, int64_t rows, int64_t k, int8_t *t)
{
    if (rows < 0 || k < 0 || k % 80 != 0) return ORC_BAD_SHAPE;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < k / 5; ++j) {
            unsigned b = codes[r * (k / 5) + j];
            if (b > 242u) return ORC_BAD_CODE;
            for (int i = 0; i < 5; ++i) {
                t[r * k + 5 * j + i] = (int8_t)((int)(b % 3u) - 1);
                b /= 3u;
            }
        }
    return ORC_OK;
}

/* y[mi*rows + r] = scale[r] * sum_k t[r][k] * x[mi*k + k'] from base-3 codes,
 * in double, for rows [row_begin, row_end). */
int orc_gemm5(const uint8_t *codes, const float *scale, int64_t rows, int64_t k,
              const uint16_t *x, int64_t m, double *y, int64_t row_begin, int64_t row_end)
{
    if (rows < 0 || k < 0 || k % 80 != 0 || m < 0) return ORC_BAD_SHAPE;
    for (int64_t mi = 0; mi < m; ++mi)
        for (int64_t r = row_begin; r < row_end; ++r) {
            double acc = 0.0;
            for (int64_t j = 0; j < k / 5; ++j) {
                unsigned b = codes[r * (k / 5) + j];
                if (b > 242u) return ORC_BAD_CODE;
                for (int i = 0; i < 5; ++i) {
                    acc += (double)((int)(b % 3u) - 1) * orc_bf16_to_double(x[mi * k + 5 * j + i]);
                    b /= 3u;
                }
            }
            y[mi * rows + r] = (double)scale[r] * acc;
        }
    return ORC_OK;
}
