/*
 * w4_cpu_omp.c -- the all-core CPU baseline, for timing only (not a checker).
 *
 * The oracle's matrix-vector product (w4_oracle.c) restated with its output
 * rows shared among all host cores (OpenMP), so that the GPU can be reported
 * beside the same arithmetic run on every core of the host -- the CPU
 * progression the pages show for a decode engine (single thread, then
 * OpenMP over rows, then wider SIMD).  Each row is computed exactly as the
 * oracle computes it -- w32 = (float)(q - z) * (float)s, exact in fp32, then
 * the fp64 dot product in increasing k -- so the results are bit-identical
 * to the oracle's; only the rows are spread over threads.  Only bench.py's
 * CPU-baseline leg and the tests load it.  Build with -fopenmp
 * -ffp-contract=off.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <string.h>

/* binary16 bits -> value (IEEE 754: 1 sign, 5 exponent bits with bias 15,
 * 10 fraction bits; subnormals have exponent field 0). */
static double half_value(uint16_t h)
{
    const int e = (h >> 10) & 0x1F, f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);
    return (h & 0x8000) ? -v : v;
}

/* bfloat16 bits -> value (the upper half of a binary32). */
static double bf16_value(uint16_t b)
{
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int w4c_threads(void) { return omp_get_max_threads(); }

/* y[M][N] (fp64) = sum_k ((q - z) * s) * x[m][k], rows shared among threads. */
void w4c_gemv_f64(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                  const uint16_t *x, int M, int K, int N, double *y)
{
    const int G = K / 128, W = K / 8;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                const int g = k / 128;
                const int q = (int)((qweight[(size_t)n * W + k / 8] >> (4 * (k % 8))) & 0xFu);
                const float w32 = (float)(q - (int)zeros[(size_t)n * G + g]) *
                                  (float)half_value(scales[(size_t)n * G + g]);
                acc += (double)w32 * bf16_value(x[(size_t)m * K + k]);
            }
            y[(size_t)m * N + n] = acc;
        }
    }
}
