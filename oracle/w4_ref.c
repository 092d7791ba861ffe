/*
 * CPU oracle for the W4 group-quantised linear layer -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code, header or table with the CUDA path.
 *
 * What it computes (TensorFold README, "What each checkpoint needs": 4-bit
 * weights in groups of 64 for the dense model and of 32 for the MoE model;
 * the quantiser is symmetric: a signed 4-bit code times one fp16 scale per
 * group, no zero point):
 *
 *     y[r][n] = sum_{g ascending} s[n][g] * ( sum_{k in group g} c[n][k] * x[r][k] )
 *
 * in fp64, with the partial sum of each group formed first and then scaled,
 * in ascending k inside the group and ascending g across groups.
 *
 * Canonical weight layout (the library's input format):
 *   codes  uint8 [N][K/2]:  k even -> low nibble, k odd -> high nibble,
 *                           each nibble a two's-complement integer in [-8, 7]
 *   scales uint16 [N][K/G]: IEEE binary16 bit patterns
 *   x      uint16 [R][K]:   bfloat16 bit patterns
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* IEEE 754 binary16 -> double, from the format's definition. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24);              /* subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), expo - 25); /* (1.mant) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Signed code of element (row, k) from the canonical packed layout. */
int oracle_code_at(const uint8_t *codes, int K, int row, int k)
{
    uint8_t byte = codes[(size_t)row * (size_t)(K / 2) + (size_t)(k / 2)];
    int nib = (k % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
    return nib >= 8 ? nib - 16 : nib;
}

/* Unpack the canonical codes into int8 [N][K] (used by the round-trip pins). */
void oracle_unpack_codes(const uint8_t *codes, int K, int N, int8_t *out)
{
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            out[(size_t)n * K + k] = (int8_t)oracle_code_at(codes, K, n, k);
}

/*
 * y[r][j] for the output columns cols[j] (all N columns when cols == NULL,
 * then ncols must equal N).  x is bf16 bits [R][K]; y is double [R][ncols].
 */
void oracle_w4_linear(const uint8_t *codes, const uint16_t *scales, const uint16_t *x,
                      int R, int K, int N, int G, const int64_t *cols, int ncols, double *y)
{
    const int n_groups = K / G;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int j = 0; j < ncols; ++j) {
        const int n = cols ? (int)cols[j] : j;
        for (int r = 0; r < R; ++r) {
            double acc = 0.0;
            for (int g = 0; g < n_groups; ++g) {
                double part = 0.0;
                for (int k = g * G; k < (g + 1) * G; ++k) {
                    double c = (double)oracle_code_at(codes, K, n, k);
                    part += c * oracle_bf16_to_double(x[(size_t)r * K + k]);
                }
                acc += oracle_half_to_double(scales[(size_t)n * n_groups + g]) * part;
            }
            y[(size_t)r * ncols + j] = acc;
        }
    }
}

/* Decoders exported for the pins (vectorised over arrays). */
void oracle_half_array(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(h[i]);
}

void oracle_bf16_array(const uint16_t *b, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(b[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
