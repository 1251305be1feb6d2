/*
 * RMSNorm forward oracle: plain, slow, fp64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library; the product path
 * never does. It shares no code, header, table or constant with the CUDA
 * library: it has its own bf16/fp16/fp32 decoders and its own
 * round-to-nearest-even encoders, written from the IEEE-754 binary16, binary32
 * and bfloat16 formats.
 *
 * Activations and weights are bf16, fp16 or fp32 (x, w and y share one
 * dtype; the kernel listing casts y back to the dtype of X, whatever it is).
 *
 * What it computes, for each row i of a row-major [M, N] activation x and a
 * weight vector w[N]:
 *
 *   s_i    = sum over j < N of x_ij^2                    (fp64, index order)
 *   ms_i   = s_i / N                                     (the true N)
 *   r_i    = 1 / sqrt(ms_i + eps)                        (eps inside the root)
 *   y_ij   = RNE_dtype( x_ij * r_i * (offset + w_j) )    (one rounding)
 *
 * Sources (web pages the method is taken from):
 *   - "Why cutile's rmsnorm required full register" (TileGym issue #169),
 *     kernel listing: the fp32 cast before squaring, the row sum of squares,
 *     division by N, eps added to the mean, rsqrt, the fp32 rstd kept for
 *     backward, y = x_normalised * (offset + w) with offset 0 for Llama and 1
 *     for Gemma3, and a single cast to the activation dtype at the end.
 *     Zero-padded columns beyond N never enter the sum.
 *   - "RMSNorm Kernel Optimization" (skillmd), Overview and Verification:
 *     out = x / sqrt(mean(x^2) + eps) * weight, and the correctness reference
 *     x * rsqrt(mean(x^2) + eps) * weight.
 * The pages leave the rounding of y unstated; this oracle reads it as IEEE
 * round-to-nearest-even, applied once to the exact-as-possible fp64 value.
 *
 * Parity pins (tests that tie this file to something other than itself):
 * 16-bit decoders against torch/numpy for all 65536 bit patterns and the fp32
 * decoder against numpy's float32 on every exponent and a million patterns;
 * encoders against exact rational rounding and numpy's float64 -> float16 and
 * float64 -> float32 conversions; the constant-row closed form; power-of-two
 * scale invariance; the textbook expression in torch float64; the Gemma
 * identity; hand-derived closed-form fixtures; brute force in 60-digit decimal
 * on tiny shapes; and the backward against torch float64 autograd and central
 * differences. No function here is "parity unpinned".
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math, no
 * fused multiply-add contraction, so x86-64 and aarch64 give the same bits).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define ORACLE_BF16 0
#define ORACLE_FP16 1
#define ORACLE_FP32 2

/* ---- decoders: exact bit pattern -> double ------------------------------ */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xFF;
    int frac = b & 0x7F;
    double mag;
    if (expo == 0xFF) {
        mag = frac ? NAN : INFINITY;
    } else if (expo == 0) {
        mag = ldexp((double)frac, -126 - 7);             /* subnormal */
    } else {
        mag = ldexp((double)(128 + frac), expo - 127 - 7); /* normal */
    }
    return sign ? -mag : mag;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double mag;
    if (expo == 0x1F) {
        mag = frac ? NAN : INFINITY;
    } else if (expo == 0) {
        mag = ldexp((double)frac, -14 - 10);
    } else {
        mag = ldexp((double)(1024 + frac), expo - 15 - 10);
    }
    return sign ? -mag : mag;
}

/* IEEE binary32: 1 sign bit, 8 exponent bits (bias 127), 23 fraction bits. */
double oracle_f32_to_f64(uint32_t b)
{
    int sign = (int)((b >> 31) & 1u);
    int expo = (int)((b >> 23) & 0xFFu);
    int32_t frac = (int32_t)(b & 0x7FFFFFu);
    double mag;
    if (expo == 0xFF) {
        mag = frac ? NAN : INFINITY;
    } else if (expo == 0) {
        mag = ldexp((double)frac, -126 - 23);
    } else {
        mag = ldexp((double)((1 << 23) + frac), expo - 127 - 23);
    }
    return sign ? -mag : mag;
}

/* ---- encoders: double -> nearest representable, ties to even ------------ */

/*
 * Generic binary-float rounding for a format with `mbits` fraction bits,
 * minimum normal exponent `emin`, and all-ones exponent field `emax_field`,
 * whose sign is bit `sign_bit`. Returns the bit pattern (sign, exponent
 * field, fraction).
 */
static uint32_t round_to_binary(double v, int mbits, int emin, int bias, int emax_field,
                                int sign_bit)
{
    uint32_t sign = signbit(v) ? (1u << sign_bit) : 0u;
    uint32_t quiet_nan = ((uint32_t)emax_field << mbits) | (1u << (mbits - 1));
    uint32_t inf = (uint32_t)emax_field << mbits;
    if (isnan(v)) return sign | quiet_nan;
    double a = fabs(v);
    if (isinf(a)) return sign | inf;
    if (a == 0.0) return sign;

    int e2;
    frexp(a, &e2);          /* a = f * 2^e2 with f in [0.5, 1) */
    int e = e2 - 1;         /* 2^e <= a < 2^(e+1) */
    if (e < emin) e = emin; /* subnormal range shares the minimum quantum */
    int qexp = e - mbits;   /* value of one unit in the last place */

    double scaled = ldexp(a, -qexp); /* exact: power-of-two scaling */
    double n = floor(scaled);
    double rem = scaled - n;         /* exact: scaled < 2^(mbits+1) */
    if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;

    int64_t k = (int64_t)n;          /* 0 .. 2^(mbits+1) */
    int64_t hidden = (int64_t)1 << mbits;
    if (k == 0) return sign;
    if (k >= 2 * hidden) {           /* carry into the next binade */
        k >>= 1;
        e += 1;
    }
    int field;
    if (k < hidden) {
        field = 0;                   /* stays subnormal (only when e == emin) */
    } else {
        field = e + bias;
        k -= hidden;
    }
    if (field >= emax_field) return sign | inf;
    return sign | ((uint32_t)field << mbits) | (uint32_t)k;
}

uint16_t oracle_f64_to_bf16(double v) { return (uint16_t)round_to_binary(v, 7, -126, 127, 0xFF, 15); }
uint16_t oracle_f64_to_f16(double v) { return (uint16_t)round_to_binary(v, 10, -14, 15, 0x1F, 15); }
uint32_t oracle_f64_to_f32(double v) { return round_to_binary(v, 23, -126, 127, 0xFF, 31); }

static int dtype_ok(int dtype)
{
    return dtype == ORACLE_BF16 || dtype == ORACLE_FP16 || dtype == ORACLE_FP32;
}

/* Element k of an array of `dtype` bit patterns, widened exactly to double. */
static double load_elem(int dtype, const void* p, int64_t k)
{
    if (dtype == ORACLE_FP32) return oracle_f32_to_f64(((const uint32_t*)p)[k]);
    if (dtype == ORACLE_BF16) return oracle_bf16_to_f64(((const uint16_t*)p)[k]);
    return oracle_f16_to_f64(((const uint16_t*)p)[k]);
}

/* Stores the `dtype` value nearest to v (ties to even) as element k. */
static void store_elem(int dtype, void* p, int64_t k, double v)
{
    if (dtype == ORACLE_FP32)
        ((uint32_t*)p)[k] = oracle_f64_to_f32(v);
    else if (dtype == ORACLE_BF16)
        ((uint16_t*)p)[k] = oracle_f64_to_bf16(v);
    else
        ((uint16_t*)p)[k] = oracle_f64_to_f16(v);
}

/* Array forms, so tests can sweep whole bit spaces in one call. Bit patterns
 * are uint16 for bf16/fp16 and uint32 for fp32. */
int oracle_decode(int dtype, int64_t n, const void* bits, double* out)
{
    if (!dtype_ok(dtype)) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(dtype, bits, i);
    return 0;
}

int oracle_encode(int dtype, int64_t n, const double* v, void* out)
{
    if (!dtype_ok(dtype)) return -1;
    for (int64_t i = 0; i < n; ++i) store_elem(dtype, out, i, v[i]);
    return 0;
}

/* ---- the forward ------------------------------------------------------- */

/*
 * Rows [row0, row1) of the RMSNorm forward over x[M, N] (row-major bit
 * patterns of `dtype`) and w[N] (same dtype).
 *   y      [M, N] rounded outputs (bit patterns), may be NULL
 *   rstd   [M]    r_i in fp64, may be NULL
 *   y_f64  [M, N] the unrounded fp64 product, may be NULL
 * eps and offset arrive as the fp32 values the CUDA entry point receives and
 * are widened exactly. Returns 0, or -1 on a bad argument.
 */
int oracle_rmsnorm_fwd(const void* x, const void* w, void* y, double* rstd, double* y_f64,
                       int64_t M, int64_t N, float eps, float offset, int dtype, int64_t row0,
                       int64_t row1)
{
    if (!dtype_ok(dtype)) return -1;
    if (M < 0 || N <= 0 || row0 < 0 || row1 > M || row0 > row1) return -1;
    const double e = (double)eps;
    const double off = (double)offset;

    for (int64_t i = row0; i < row1; ++i) {
        const int64_t xi = i * N; /* first element of row i */
        double s = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double v = load_elem(dtype, x, xi + j);
            s += v * v;
        }
        double ms = s / (double)N;
        double r = 1.0 / sqrt(ms + e);
        if (rstd) rstd[i] = r;
        for (int64_t j = 0; j < N; ++j) {
            double scale = off + load_elem(dtype, w, j);
            double v = load_elem(dtype, x, xi + j) * r * scale;
            if (y_f64) y_f64[i * N + j] = v;
            if (y) store_elem(dtype, y, i * N + j, v);
        }
    }
    return 0;
}

/* ---- the backward (derived; the pages only say rstd is kept for it) ----
 *
 * For y_ij = x_ij * r_i * s_j with s_j = offset + w_j and
 * r_i = (sum_k x_ik^2 / N + eps)^(-1/2), the chain rule gives, for an
 * upstream gradient dy:
 *
 *   c_i    = sum_j dy_ij * s_j * x_ij
 *   dx_ij  = r_i * (dy_ij * s_j - x_ij * r_i^2 * c_i / N)
 *   dw_j   = sum_i dy_ij * x_ij * r_i
 *
 * (d r_i / d x_ik = -r_i^3 x_ik / N.) r_i is the saved rstd: the caller passes
 * it (as the CUDA backward receives it), or NULL to recompute it here in fp64
 * from x and eps. dx is returned rounded to the dtype (one rounding) and in
 * fp64; dw in fp64, summed over rows in index order.
 */
int oracle_rmsnorm_bwd(const void* x, const void* w, const void* dy, const double* rstd,
                       void* dx, double* dx_f64, double* dw, int64_t M, int64_t N, float eps,
                       float offset, int dtype)
{
    if (!dtype_ok(dtype)) return -1;
    if (M < 0 || N <= 0) return -1;
    const double off = (double)offset;
    if (dw)
        for (int64_t j = 0; j < N; ++j) dw[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        const int64_t base = i * N; /* first element of row i of x, dy and dx */
        double r;
        if (rstd) {
            r = rstd[i];
        } else {
            double s = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double v = load_elem(dtype, x, base + j);
                s += v * v;
            }
            r = 1.0 / sqrt(s / (double)N + (double)eps);
        }
        double c = 0.0;
        for (int64_t j = 0; j < N; ++j)
            c += load_elem(dtype, dy, base + j) * (off + load_elem(dtype, w, j)) *
                 load_elem(dtype, x, base + j);
        for (int64_t j = 0; j < N; ++j) {
            double xv = load_elem(dtype, x, base + j), gv = load_elem(dtype, dy, base + j);
            double sv = off + load_elem(dtype, w, j);
            double v = r * (gv * sv - xv * r * r * c / (double)N);
            if (dx_f64) dx_f64[base + j] = v;
            if (dx) store_elem(dtype, dx, base + j, v);
            if (dw) dw[j] += gv * xv * r;
        }
    }
    return 0;
}
