/*
 * w4_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what the weight-only INT4
 * (group 128) matrix-vector product computes.  It exists so that the CUDA
 * library can be checked against something obviously correct.  Only the test
 * suite, __graft_entry__.smoke() and the CPU-baseline leg of bench.py may load
 * it; the library (int4_weight_only_w4_gb300) never does, and the two share no
 * code, headers or tables.
 *
 * Sources (page title, section):
 *  - Storage format (the library's canonical layout): qweight[N][K/8] uint32
 *    with nibble j of word w holding k = 8w + j at bits 4j..4j+3,
 *    scales[N][K/128] fp16 and zeros[N][K/128] uint8 in 0..15; a weight is
 *    w = (q - z) * s.  The asymmetric form with a zero point per group is the
 *    AWQ form ("Custom AWQ Dequantization Kernel", section "Dead ends in
 *    profiling": the dequantisation formula there applies zeros and scales).
 *  - Group indexing: one scale per group of 128 consecutive weights per output
 *    row ("Building an LLM Inference Runtime ...", section "The Stack
 *    Architecture: A One-Page Overview"; "CodeAlign-Runtime", section
 *    "Level 3 -- Quantization Scheme").
 *  - Dequantise, multiply by the group scale and accumulate per output row
 *    ("Building an LLM Inference Runtime ...", section "Bug #3", Path B: mask
 *    the nibble, multiply by the group's scale, feed the row accumulator).
 *
 * Arithmetic: each weight is dequantised to fp32, w32 = (float)(q - z) *
 * (float)s, which is exact (|q - z| <= 15 needs 4 bits, an fp16 significand
 * 11, their product at most 15 <= 24).  The dot product is then taken in fp64
 * in increasing k: every product w32 * x is exact in fp64 (at most 24 + 8
 * significant bits), so the only rounding is that of the K additions.
 *
 * Conversions are written from the IEEE 754 encodings: binary16 is 1 sign,
 * 5 exponent (bias 15) and 10 fraction bits; bfloat16 is the upper 16 bits of
 * a binary32.  Rounding to nearest, ties to even, everywhere.
 *
 * Build with -ffp-contract=off so that no multiply-add is fused and results
 * are the same on every host.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define W4O_GROUP 128

/* ---- number formats ------------------------------------------------------ */

double w4o_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25); /* (1024 + f) * 2^(e - 15 - 10) */
    return sign ? -v : v;
}

double w4o_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;             /* bfloat16 = top half of binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to binary16, to nearest with ties to even. */
uint16_t w4o_double_to_half_rne(double v)
{
    if (isnan(v))
        return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7C00;
    int e2;
    frexp(a, &e2);                  /* a = m * 2^e2 with m in [0.5, 1) */
    int E = e2 - 1;                 /* a in [2^E, 2^(E+1)) */
    if (E < -14)
        E = -14;                    /* below the normal range the quantum stays 2^-24 */
    if (E > 15)
        return sign | 0x7C00;
    double r = nearbyint(ldexp(a, 10 - E)); /* significand in units of 2^(E-10), RNE */
    if (r >= 2048.0) {              /* rounded up into the next binade */
        r = 1024.0;
        E += 1;
        if (E > 15)
            return sign | 0x7C00;
    }
    if (r < 1024.0)                 /* subnormal (only possible when E == -14) */
        return sign | (uint16_t)r;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)r - 1024));
}

/* Round a binary32 to bfloat16, to nearest with ties to even. */
uint16_t w4o_float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x40);    /* quiet NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Elementwise binary32 -> bfloat16 over an array (same rounding as above). */
void w4o_float_to_bf16_rne_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = w4o_float_to_bf16_rne(in[i]);
}

/* ---- dequantisation ------------------------------------------------------ */

/* q of weight (n, k) in the canonical layout: word k/8 of row n, nibble k%8. */
static int w4o_q(const uint32_t *qweight, int K, int n, int k)
{
    uint32_t word = qweight[(size_t)n * (size_t)(K / 8) + (size_t)(k / 8)];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

/* w32 = (q - z) * s for weight (n, k); group g = k / 128 of row n. */
static float w4o_w32(const uint32_t *qweight, const uint16_t *scales,
                     const uint8_t *zeros, int K, int n, int k)
{
    int G = K / W4O_GROUP;
    size_t gi = (size_t)n * (size_t)G + (size_t)(k / W4O_GROUP);
    int q = w4o_q(qweight, K, n, k);
    int z = zeros[gi];
    float s = (float)w4o_half_to_double(scales[gi]);
    return (float)(q - z) * s;
}

/* w_out[N][K] = (q - z) * s in fp32 (exact). */
void w4o_dequant_f32(const uint32_t *qweight, const uint16_t *scales,
                     const uint8_t *zeros, int K, int N, float *w_out)
{
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            w_out[(size_t)n * K + k] = w4o_w32(qweight, scales, zeros, K, n, k);
}

/* w_out[N][K] = binary16 bits of (q - z) * s, rounded once to nearest-even. */
void w4o_dequant_f16(const uint32_t *qweight, const uint16_t *scales,
                     const uint8_t *zeros, int K, int N, uint16_t *w_out)
{
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            w_out[(size_t)n * K + k] = w4o_double_to_half_rne(
                (double)w4o_w32(qweight, scales, zeros, K, n, k));
}

/* ---- matrix-vector product ----------------------------------------------- */

/* y = sum_k w32(n, k) * x[m][k] in fp64, k increasing; optionally also
 * sum_k |w32(n, k) * x[m][k]| (used by tests for rounding-error bounds). */
static void w4o_dot(const uint32_t *qweight, const uint16_t *scales,
                    const uint8_t *zeros, const uint16_t *x, int K, int n, int m,
                    double *y, double *yabs)
{
    double acc = 0.0, accabs = 0.0;
    for (int k = 0; k < K; ++k) {
        double p = (double)w4o_w32(qweight, scales, zeros, K, n, k) *
                   w4o_bf16_to_double(x[(size_t)m * K + k]);
        acc += p;
        accabs += fabs(p);
    }
    *y = acc;
    if (yabs)
        *yabs = accabs;
}

/* y[M][N] (fp64) for x[M][K] (bfloat16 bits).  yabs may be NULL. */
void w4o_gemv_f64(const uint32_t *qweight, const uint16_t *scales,
                  const uint8_t *zeros, const uint16_t *x, int M, int K, int N,
                  double *y, double *yabs)
{
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n)
            w4o_dot(qweight, scales, zeros, x, K, n, m,
                    &y[(size_t)m * N + n], yabs ? &yabs[(size_t)m * N + n] : 0);
}

/* The same product restricted to the R output rows listed in rows[]:
 * y[M][R] with y[m][i] = row rows[i].  yabs may be NULL. */
void w4o_gemv_rows_f64(const uint32_t *qweight, const uint16_t *scales,
                       const uint8_t *zeros, const uint16_t *x, int M, int K,
                       const int64_t *rows, int R, double *y, double *yabs)
{
    for (int m = 0; m < M; ++m)
        for (int i = 0; i < R; ++i)
            w4o_dot(qweight, scales, zeros, x, K, (int)rows[i], m,
                    &y[(size_t)m * R + i], yabs ? &yabs[(size_t)m * R + i] : 0);
}

/* ---- quantisation: binary16 W -> canonical (q, s, z) ------------------------
 *
 * Per row n and group g of 128 weights (the grouping of the matrix-vector
 * product above), in fp32 from the exact binary16 values, every operation
 * rounded to nearest (ties to even):
 *
 *  mode 0, asymmetric (the storage format's zero point, round to nearest):
 *    lo = min(0, min w), hi = max(0, max w)   -- 0 is always representable
 *    s  = fp16((hi - lo) / 15)
 *    z  = clamp(rint(-lo / s), 0, 15)
 *    q  = clamp(rint(w / s) + z, 0, 15)
 *  mode 1, symmetric ("Building an LLM Inference Runtime ...", section "The
 *  Stack Architecture: A One-Page Overview": scale = absmax / 7;
 *  "CodeAlign-Runtime", section "Level 3 -- Quantization Scheme": values in
 *  [-8, 7]), stored with the fixed zero point 8:
 *    s  = fp16(max |w| / 7)
 *    z  = 8
 *    q  = clamp(rint(w / s), -8, 7) + 8
 *
 * The codes are computed against the stored (fp16) scale, so that (q - z) * s
 * is the value the product uses.  A group whose scale rounds to 0 (all zeros,
 * or a range below the smallest fp16 subnormal) stores s = 0 and q = z (0 in
 * mode 0, 8 in mode 1).  Inputs must be finite.
 */
static float w4o_clampf(float v, float a, float b)
{
    return v < a ? a : (v > b ? b : v);
}

void w4o_quantize(const uint16_t *w, int K, int N, int mode, uint32_t *qweight,
                  uint16_t *scales, uint8_t *zeros)
{
    const int G = K / W4O_GROUP;
    memset(qweight, 0, (size_t)N * (size_t)(K / 8) * sizeof(uint32_t));
    for (int n = 0; n < N; ++n) {
        for (int g = 0; g < G; ++g) {
            const uint16_t *wg = w + (size_t)n * K + (size_t)g * W4O_GROUP;
            float lo = 0.0f, hi = 0.0f, amax = 0.0f;
            for (int k = 0; k < W4O_GROUP; ++k) {
                const float v = (float)w4o_half_to_double(wg[k]);
                if (v < lo) lo = v;
                if (v > hi) hi = v;
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            const float s32 = mode == 0 ? (hi - lo) / 15.0f : amax / 7.0f;
            const uint16_t sh = w4o_double_to_half_rne((double)s32);
            const float s = (float)w4o_half_to_double(sh);
            int z;
            if (s == 0.0f)
                z = mode == 0 ? 0 : 8;
            else if (mode == 0)
                z = (int)w4o_clampf(rintf(-lo / s), 0.0f, 15.0f);
            else
                z = 8;
            for (int k = 0; k < W4O_GROUP; ++k) {
                int q;
                if (s == 0.0f) {
                    q = z;
                } else {
                    const float t = rintf((float)w4o_half_to_double(wg[k]) / s);
                    if (mode == 0)
                        q = (int)w4o_clampf(w4o_clampf(t, -16.0f, 16.0f) + (float)z, 0.0f,
                                            15.0f);
                    else
                        q = (int)w4o_clampf(t, -8.0f, 7.0f) + 8;
                }
                const int kk = g * W4O_GROUP + k;
                qweight[(size_t)n * (K / 8) + kk / 8] |= (uint32_t)q << (4 * (kk % 8));
            }
            scales[(size_t)n * G + g] = sh;
            zeros[(size_t)n * G + g] = (uint8_t)z;
        }
    }
}

/* ---- gate/up product with the SwiGLU activation -----------------------------
 *
 * W is the fused [2I][K] matrix of a gated MLP: rows 0..I-1 are the gate
 * projection, rows I..2I-1 the up projection.  For token m and output j:
 *   g = sum_k w32(j, k) x[m][k],  u = sum_k w32(I + j, k) x[m][k]  (fp64, as above)
 *   y[m][j] = silu(g) * u,  silu(g) = g / (1 + exp(-g))
 * ("qengine", section "How it works": gate and up projections interleaved so
 * that SwiGLU runs in registers -- the activation applied to the pair of
 * products of the same output).  fp64 throughout; exp from the C library.
 */
void w4o_gemv_swiglu_f64(const uint32_t *qweight, const uint16_t *scales,
                         const uint8_t *zeros, const uint16_t *x, int M, int K, int I,
                         double *y)
{
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < I; ++j) {
            double g, u;
            w4o_dot(qweight, scales, zeros, x, K, j, m, &g, 0);
            w4o_dot(qweight, scales, zeros, x, K, I + j, m, &u, 0);
            y[(size_t)m * I + j] = g / (1.0 + exp(-g)) * u;
        }
}
