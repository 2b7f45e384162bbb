/*
 * w8_oracle.c -- CPU oracle for the FP8 weight-only (w8a16) decode GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, __graft_entry__.smoke() and the cpu_baseline
 * leg of bench.py use it.  It shares no code, header, table or constant with
 * the CUDA path under fp8_weight_only_w8a16_gb300/csrc.
 *
 * What it computes (ATOM pull request #2980, sections
 * Summary and Changes): for every output row n and decode token m
 *
 *     y[m,n] = bf16_rne( scale[n] * sum_k widen(W[n,k]) * x[m,k] )
 *
 * with W an E4M3fn plane (one fp32 factor for each output row, applied once
 * the row's sum is complete and ahead of the one bf16 rounding), x bf16 activations and
 * fp32 accumulation.  A bf16 plane runs through the same computation with no
 * scale (the PR leaves bf16 weights on their existing path).  Each E4M3 code
 * has an exact bf16 value, so the widening is the exact value of the code.
 *
 * Everything here is the plain definition: scalar loops, ascending k, fp32
 * accumulation, one fp32 multiply by the scale, one round-to-nearest-even to
 * bf16.  Build with -ffp-contract=off and without -ffast-math.  An fp64
 * recompute and a brute-force E4M3 encoder (the ptpc_fp8 quantizer's rounding)
 * are included for the tolerance checks and pins.
 *
 * Pins (tests/test_oracle_*.py) hold each function to something other than
 * itself: the 256 codes against their closed-form values and against
 * torch.float8_e4m3fn, bf16 rounding against torch.bfloat16, the GEMV against
 * a numpy fp64 matmul on tiny inputs, one-hot and exact-sum inputs against
 * exact rational results, and power-of-two scale invariance; the SiLU-and-
 * multiply against torch's float64 silu, the odd-part identity
 * silu(v) - silu(-v) = v and its limits, and the one-step fp64 -> bf16
 * rounding against the fp32 rounding and on exact bf16 midpoints; the
 * block-scaled GEMV against an fp64 brute force, one-hot tokens over
 * distinct block factors, Fraction sums, and its one-column-block case
 * against the row-scaled GEMV.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_DT_E4M3FN 1
#define ORC_DT_BF16 2

/* ------------------------------------------------------------------ */
/* Codecs                                                              */
/* ------------------------------------------------------------------ */

/* E4M3fn code -> value, bit by bit from the OCP 8-bit floating point format
 * (E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; exponent field 0 is subnormal).  The PR page
 * (Summary) relies on every such value widening exactly to bf16. */
float orc_e4m3_to_f32(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    float v;
    if (e == 15 && m == 7) {
        v = NAN;
        return s ? -v : v;
    }
    if (e == 0)
        v = ldexpf((float)m, -9);                 /* m/8 * 2^(1-7)  */
    else
        v = ldexpf(1.0f + (float)m / 8.0f, e - 7); /* 1.m * 2^(e-7) */
    return s ? -v : v;
}

/* bf16 bits -> fp32: a bf16 is the upper half of an fp32. */
float orc_bf16_to_f32(uint16_t u)
{
    uint32_t b = (uint32_t)u << 16;
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even.  NaN stays NaN (quieted,
 * sign kept); values past the largest bf16 round to infinity. */
uint16_t orc_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;          /* truncation toward zero      */
    uint32_t dropped = u & 0xFFFFu;   /* the 16 bits that are cut    */
    int up;
    if (dropped > 0x8000u)
        up = 1;                       /* more than half an ulp       */
    else if (dropped < 0x8000u)
        up = 0;                       /* less than half an ulp       */
    else
        up = (int)(kept & 1u);        /* exactly half: go to even    */
    /* bf16 patterns of one sign are ordered by magnitude, so adding one to
     * the kept pattern steps to the next larger magnitude (or to inf). */
    return (uint16_t)(kept + (uint32_t)up);
}

/* fp32 -> E4M3fn code, round to nearest with ties to even mantissa,
 * saturating at +-448.  A brute-force nearest search over the 127
 * non-negative finite codes; used by the ptpc_fp8 quantizer below. */
uint8_t orc_f32_to_e4m3_sat(float v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_d = a; /* distance to code 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs((double)orc_e4m3_to_f32((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* ptpc_fp8 row quantizer (weight side of "per-token per-channel"): one fp32
 * scale per output row, scale = amax_row / 448, codes = E4M3(W / scale)
 * clamped to +-448.  An all-zero row gets scale 1 and zero codes.  This is
 * input preparation for the tests, not part of the GEMV. */
void orc_quantize_rows(const float *w, int64_t n, int64_t k, int64_t ldw,
                       uint8_t *q, int64_t ldq, float *scale)
{
    for (int64_t r = 0; r < n; ++r) {
        float amax = 0.0f;
        for (int64_t j = 0; j < k; ++j) {
            float a = fabsf(w[r * ldw + j]);
            if (a > amax)
                amax = a;
        }
        float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        scale[r] = s;
        for (int64_t j = 0; j < k; ++j) {
            float t = w[r * ldw + j] / s;
            if (t > 448.0f)
                t = 448.0f;
            if (t < -448.0f)
                t = -448.0f;
            q[r * ldq + j] = orc_f32_to_e4m3_sat(t);
        }
    }
}

/* ------------------------------------------------------------------ */
/* GEMV                                                                */
/* ------------------------------------------------------------------ */

static float weight_value(const void *w, int dtype, int64_t idx)
{
    if (dtype == ORC_DT_E4M3FN)
        return orc_e4m3_to_f32(((const uint8_t *)w)[idx]);
    return orc_bf16_to_f32(((const uint16_t *)w)[idx]);
}

/* The method, as the plain definition.  W is [n][ldw] (logical k columns),
 * x is [m][ldx] bf16, y is [m][ldy] bf16.  For dtype E4M3FN, scale[n] is the
 * fp32 row scale; for BF16 it is ignored (may be NULL).  `threads` > 1
 * splits the output rows over OpenMP threads; every row is still summed in
 * ascending k by one thread, so the result does not depend on it.
 * Returns 0, or -1 on a bad argument. */
int orc_gemv(const void *w, int dtype, int64_t n, int64_t k, int64_t ldw,
             const float *scale, const uint16_t *x, int64_t ldx, int64_t m,
             uint16_t *y, int64_t ldy, int threads)
{
    if (!w || !x || !y || n < 0 || k < 0 || m < 0 || ldw < k || ldx < k || ldy < n)
        return -1;
    if (dtype != ORC_DT_E4M3FN && dtype != ORC_DT_BF16)
        return -1;
    if (dtype == ORC_DT_E4M3FN && !scale)
        return -1;
#ifdef _OPENMP
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(threads)
#endif
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t j = 0; j < k; ++j) {
                float wv = weight_value(w, dtype, r * ldw + j);
                float xv = orc_bf16_to_f32(x[i * ldx + j]);
                float p = wv * xv; /* exact: 4 x 8 significant bits */
                acc = acc + p;
            }
            float t = (dtype == ORC_DT_E4M3FN) ? scale[r] * acc : acc;
            y[i * ldy + r] = orc_f32_to_bf16_rne(t);
        }
    }
    (void)threads;
    return 0;
}

/* fp64 recompute of the same widened inputs, for the tolerance checks:
 *   y64[i][r]   = scale[r] * sum_k W[r,k] * x[i,k]      (in double)
 *   mag64[i][r] = sum_k |scale[r] * W[r,k] * x[i,k]|    (in double)
 * Both arrays are [m][n]. */
int orc_gemv_f64(const void *w, int dtype, int64_t n, int64_t k, int64_t ldw,
                 const float *scale, const uint16_t *x, int64_t ldx, int64_t m,
                 double *y64, double *mag64, int threads)
{
    if (!w || !x || !y64 || !mag64 || n < 0 || k < 0 || m < 0 || ldw < k || ldx < k)
        return -1;
    if (dtype != ORC_DT_E4M3FN && dtype != ORC_DT_BF16)
        return -1;
    if (dtype == ORC_DT_E4M3FN && !scale)
        return -1;
#ifdef _OPENMP
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(threads)
#endif
    for (int64_t r = 0; r < n; ++r) {
        double s = (dtype == ORC_DT_E4M3FN) ? (double)scale[r] : 1.0;
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0, mag = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                double p = (double)weight_value(w, dtype, r * ldw + j) *
                           (double)orc_bf16_to_f32(x[i * ldx + j]);
                acc += p;
                mag += fabs(s * p);
            }
            y64[i * n + r] = s * acc;
            mag64[i * n + r] = mag;
        }
    }
    (void)threads;
    return 0;
}

/* Number of threads OpenMP would use (1 without OpenMP). */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* SiLU-and-multiply of a merged gate_up projection                    */
/* ------------------------------------------------------------------ */

/* fp64 -> bf16, round to nearest, ties to even, in one step (no detour
 * through fp32, whose own rounding could move a value onto a bf16 midpoint).
 * bf16 keeps 8 significant bits with fp32's exponent range: a value in
 * [2^(e-1), 2^e) has spacing 2^(e-8), and below 2^-126 the spacing stays
 * 2^-133 (subnormals).  Dividing by that spacing is exact, nearbyint rounds
 * to the nearest integer with ties to even (the default rounding mode), and
 * a result of 2^128 or more is infinity.  NaN stays NaN (quiet, sign kept). */
uint16_t orc_f64_to_bf16_rne(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    double a = fabs(v);
    uint16_t sign = signbit(v) ? 0x8000u : 0x0000u;
    if (a == 0.0)
        return sign;
    if (isinf(a) || a >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    if (e < -125)
        e = -125;
    double q = ldexp(1.0, e - 8);
    double r = nearbyint(a / q) * q;
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* The MLP activation between a merged gate_up projection and the down
 * projection (ATOM Model Support Guide, Model architecture details, Llama:
 * one merged column-parallel projection for gate and up, then SiLU and
 * multiply, then down; Adding a new model, Step 5: gate_proj is shard 0 and
 * up_proj shard 1 of gate_up_proj):
 *
 *     h = silu(g) * u,   silu(v) = v * sigmoid(v) = v / (1 + exp(-v))
 *
 * elementwise over `count` pairs, in fp64, unrounded.  g and u are the values
 * the projection produced (the GEMV's bf16 outputs, widened by the caller).
 * At v = -inf the quotient is -inf / inf = NaN, as the formula gives. */
int orc_silu_mul_f64(const double *g, const double *u, int64_t count, double *h)
{
    if (!g || !u || !h || count < 0)
        return -1;
    for (int64_t i = 0; i < count; ++i) {
        double s = g[i] / (1.0 + exp(-g[i]));
        h[i] = s * u[i];
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* w4a16: MXFP4 weights (E2M1 elements, E8M0 block scales)             */
/* ------------------------------------------------------------------ */

/* The ATOM Model Support Guide (Model-specific optimizations, DeepSeek
 * V2/V3: FP4 support) names MXFP4 GEMMs with 16-bit activations
 * ("a16wfp4"), and the GLM-5.2 anatomy page's verified deployments serve a
 * GLM-5.2-MXFP4 checkpoint.  MXFP4 is the OCP
 * microscaling format: 4-bit E2M1 elements, 32 consecutive elements along K
 * sharing one 8-bit E8M0 scale.  This file's readings of what the pages leave
 * open: two elements per byte, column 2i in the low nibble and 2i+1 in the
 * high nibble; the block scales are a row-major [n][ldb] byte array, block
 * j covering columns 32j .. 32j+31; no per-row scale on top. */

/* E2M1 code (low 4 bits) -> value: sign bit 3, exponent bits 2..1 (bias 1),
 * mantissa bit 0; exponent 0 is subnormal (m * 0.5); no infinity or NaN. */
float orc_e2m1_to_f32(uint8_t c)
{
    int s = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    float v = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
    return s ? -v : v;
}

/* E8M0 scale -> value: 2^(e - 127); 255 is NaN. */
float orc_e8m0_to_f32(uint8_t e)
{
    if (e == 255)
        return NAN;
    return ldexpf(1.0f, (int)e - 127);
}

/* Element (r, j) of an MXFP4 plane: code from its nibble times its block's
 * scale.  The product is exact in fp32 (2 significant bits) unless it
 * leaves fp32's range. */
static float mxfp4_value(const uint8_t *w, int64_t ldw_bytes, const uint8_t *bs, int64_t ldb,
                         int64_t r, int64_t j)
{
    uint8_t byte = w[r * ldw_bytes + j / 2];
    uint8_t code = (j & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
    return orc_e2m1_to_f32(code) * orc_e8m0_to_f32(bs[r * ldb + j / 32]);
}

/* The w4a16 GEMV as the plain definition: y[i][r] = bf16_rne(sum_j
 * W[r][j] x[i][j]), W[r][j] = e2m1(code) * e8m0(scale of block j / 32), fp32
 * accumulation in ascending j.  w: [n][ldw_bytes] packed codes, bs: [n][ldb]
 * E8M0 bytes (ldb >= ceil(k / 32)).  Returns 0, or -1 on a bad argument. */
int orc_gemv_mxfp4(const uint8_t *w, int64_t n, int64_t k, int64_t ldw_bytes, const uint8_t *bs,
                   int64_t ldb, const uint16_t *x, int64_t ldx, int64_t m, uint16_t *y,
                   int64_t ldy, int threads)
{
    if (!w || !bs || !x || !y || n < 0 || k < 0 || m < 0 || 2 * ldw_bytes < k ||
        32 * ldb < k || ldx < k || ldy < n)
        return -1;
#ifdef _OPENMP
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(threads)
#endif
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t j = 0; j < k; ++j) {
                float p = mxfp4_value(w, ldw_bytes, bs, ldb, r, j) * orc_bf16_to_f32(x[i * ldx + j]);
                acc = acc + p;
            }
            y[i * ldy + r] = orc_f32_to_bf16_rne(acc);
        }
    }
    (void)threads;
    return 0;
}

/* fp64 recompute of the same dequantized inputs for the tolerance checks:
 * y64[i][r] = sum_j W x, mag64[i][r] = sum_j |W x| (both [m][n]). */
int orc_gemv_mxfp4_f64(const uint8_t *w, int64_t n, int64_t k, int64_t ldw_bytes,
                       const uint8_t *bs, int64_t ldb, const uint16_t *x, int64_t ldx, int64_t m,
                       double *y64, double *mag64, int threads)
{
    if (!w || !bs || !x || !y64 || !mag64 || n < 0 || k < 0 || m < 0 || 2 * ldw_bytes < k ||
        32 * ldb < k || ldx < k)
        return -1;
#ifdef _OPENMP
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(threads)
#endif
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0, mag = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                double p = (double)mxfp4_value(w, ldw_bytes, bs, ldb, r, j) *
                           (double)orc_bf16_to_f32(x[i * ldx + j]);
                acc += p;
                mag += fabs(p);
            }
            y64[i * n + r] = acc;
            mag64[i * n + r] = mag;
        }
    }
    (void)threads;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Block-scaled FP8: one fp32 factor per 128 x 128 block of weights    */
/* ------------------------------------------------------------------ */

/* The GLM-5.2 anatomy page (fused_qkv_a_proj) has that projection run
 * AITER's preshuffle blockscale GEMM, and the ATOM Model Support Guide
 * (Weight loading, Loading flow) loads a checkpoint's weight_scale_inv
 * tensors as the layer's weight scales.  The pages give neither the block
 * shape nor where the factor enters the sum; the readings taken here:
 *   - a factor covers 128 rows x 128 columns of W, so bs is
 *     [ceil(n / 128)][ldb] fp32 with ldb >= ceil(k / 128);
 *   - as the PR applies its row factor to a finished sum, a block's factor
 *     multiplies the finished sum of that block's 128 columns: per row and
 *     token, each block's partial sum p (fp32, ascending k) is multiplied by
 *     its factor (one fp32 multiply) and added to the row's fp32 total (one
 *     fp32 add), blocks in ascending order; the total is rounded to bf16
 *     once.  There is no row factor. */
#define ORC_BLOCK 128

static int b128_args_ok(const uint8_t *w, int64_t n, int64_t k, int64_t ldw, const float *bs,
                        int64_t ldb, const uint16_t *x, int64_t ldx, int64_t m)
{
    return w && bs && x && n >= 0 && k >= 0 && m >= 0 && ldw >= k && ldx >= k &&
           ldb * ORC_BLOCK >= k;
}

int orc_gemv_e4m3_b128(const uint8_t *w, int64_t n, int64_t k, int64_t ldw, const float *bs,
                       int64_t ldb, const uint16_t *x, int64_t ldx, int64_t m, uint16_t *y,
                       int64_t ldy, int threads)
{
    if (!b128_args_ok(w, n, k, ldw, bs, ldb, x, ldx, m) || !y || ldy < n)
        return -1;
#ifdef _OPENMP
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(threads)
#endif
    for (int64_t r = 0; r < n; ++r) {
        const float *row_factors = bs + (r / ORC_BLOCK) * ldb;
        for (int64_t i = 0; i < m; ++i) {
            float acc = 0.0f;
            for (int64_t j0 = 0; j0 < k; j0 += ORC_BLOCK) {
                const int64_t j1 = j0 + ORC_BLOCK < k ? j0 + ORC_BLOCK : k;
                float part = 0.0f;
                for (int64_t j = j0; j < j1; ++j) {
                    float wv = orc_e4m3_to_f32(w[r * ldw + j]);
                    float xv = orc_bf16_to_f32(x[i * ldx + j]);
                    float p = wv * xv; /* exact */
                    part = part + p;
                }
                float scaled = row_factors[j0 / ORC_BLOCK] * part;
                acc = acc + scaled;
            }
            y[i * ldy + r] = orc_f32_to_bf16_rne(acc);
        }
    }
    (void)threads;
    return 0;
}

/* fp64 recompute of the same inputs for the tolerance checks:
 *   y64[i][r]   = sum_j bs[r/128][j/128] * W[r,j] * x[i,j]      (double)
 *   mag64[i][r] = sum_j |bs[r/128][j/128] * W[r,j] * x[i,j]|    (double)
 * Both arrays are [m][n]. */
int orc_gemv_e4m3_b128_f64(const uint8_t *w, int64_t n, int64_t k, int64_t ldw,
                           const float *bs, int64_t ldb, const uint16_t *x, int64_t ldx,
                           int64_t m, double *y64, double *mag64, int threads)
{
    if (!b128_args_ok(w, n, k, ldw, bs, ldb, x, ldx, m) || !y64 || !mag64)
        return -1;
#ifdef _OPENMP
    if (threads < 1)
        threads = 1;
#pragma omp parallel for schedule(dynamic, 16) num_threads(threads)
#endif
    for (int64_t r = 0; r < n; ++r) {
        const float *row_factors = bs + (r / ORC_BLOCK) * ldb;
        for (int64_t i = 0; i < m; ++i) {
            double acc = 0.0, mag = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                double p = (double)row_factors[j / ORC_BLOCK] *
                           (double)orc_e4m3_to_f32(w[r * ldw + j]) *
                           (double)orc_bf16_to_f32(x[i * ldx + j]);
                acc += p;
                mag += fabs(p);
            }
            y64[i * n + r] = acc;
            mag64[i * n + r] = mag;
        }
    }
    (void)threads;
    return 0;
}
