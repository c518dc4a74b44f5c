/*
 * CPU oracle for the results of the tile pipeline.  TEST INFRASTRUCTURE ONLY:
 * the test-suite, the package smoke check and the benchmark's CPU-baseline leg
 * load this library; the GPU library neither links nor includes it.
 *
 * Plain loops, no blocking, no threads, no SIMD.  Each function states the
 * definition it writes out.
 *
 *   oracle_copy        Tile copy result.  Every in-bounds output element is the
 *                      input element at the same (row, column), bit for bit.
 *                      Source: "cute(11) Hopper TMA copy", §4 (the staged tile
 *                      is written back and compared element by element with
 *                      the input) and the row-major (M, N) : (N, 1) tensor of
 *                      §2.1.  Tiling does not change this result, so the loop
 *                      is the definition itself.
 *   oracle_rowsum      Row-sum result: out[i] = sum over j < N of x[i][j], every
 *                      element widened exactly to binary64 and added in column
 *                      order in binary64.  Optionally also sum of squares, used
 *                      by the tests to scale the row-sum tolerance.
 *   oracle_colsum      Column-sum result: out[j] = sum over i < M of x[i][j],
 *                      every element widened exactly to binary64 and added in
 *                      row order in binary64; optionally also the sum of
 *                      squares of each column.  Like the row sum, not on the
 *                      pages (their consumer only "uses" the tile): the plain
 *                      definition of a second reduction of the same tiles.
 *   oracle_f16_to_f64  Exact widening of IEEE binary16 (sign, 5-bit exponent
 *                      with bias 15, 10-bit fraction; exponent 0 = subnormal,
 *                      exponent 31 = infinity or NaN).
 *   oracle_bf16_to_f64 Exact widening of bfloat16: its 16 bits are the upper
 *                      half of an IEEE binary32 value.
 *   oracle_f32_to_f64  Exact widening of IEEE binary32.
 *   oracle_xor_fold    Checksum of a byte buffer: the bitwise XOR of all its
 *                      32-bit little-endian words.  Not on the pages: the
 *                      result of the read-bandwidth reference that states the
 *                      reductions' read-only roofline; XOR is associative and
 *                      commutative, so any grouping gives this value.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F32 = 2 };

double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 0x1f;
    int fraction = h & 0x3ff;
    double magnitude;
    if (exponent == 0) {
        /* subnormal (or zero): fraction * 2^-24 */
        magnitude = ldexp((double)fraction, -24);
    } else if (exponent == 31) {
        magnitude = fraction ? NAN : INFINITY;
    } else {
        /* normal: (1 + fraction / 1024) * 2^(exponent - 15) */
        magnitude = ldexp((double)(1024 + fraction), exponent - 25);
    }
    return sign ? -magnitude : magnitude;
}

double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t wide = (uint32_t)b << 16;
    float f;
    memcpy(&f, &wide, sizeof f);
    return (double)f;
}

double oracle_f32_to_f64(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Copy the logical M x N matrix, element by element.  esize is the element
 * size in bytes; ld_src / ld_dst are row pitches in elements.  Elements of dst
 * outside [0, M) x [0, N) are never touched. */
void oracle_copy(const void *src, void *dst, int64_t M, int64_t N,
                 int64_t ld_src, int64_t ld_dst, int esize)
{
    const unsigned char *s = (const unsigned char *)src;
    unsigned char *d = (unsigned char *)dst;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            memcpy(d + (i * ld_dst + j) * esize, s + (i * ld_src + j) * esize,
                   (size_t)esize);
        }
    }
}

static double element(const void *src, int64_t index, int dtype)
{
    if (dtype == ORACLE_F16)
        return oracle_f16_to_f64(((const uint16_t *)src)[index]);
    if (dtype == ORACLE_BF16)
        return oracle_bf16_to_f64(((const uint16_t *)src)[index]);
    return oracle_f32_to_f64(((const uint32_t *)src)[index]);
}

/* Row sums of the logical M x N matrix in binary64.  sums[i] receives the
 * sum of row i; sumsq (may be NULL) receives the sum of squares of row i. */
void oracle_rowsum(const void *src, double *sums, double *sumsq, int64_t M,
                   int64_t N, int64_t ld, int dtype)
{
    for (int64_t i = 0; i < M; ++i) {
        double s = 0.0, q = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            double x = element(src, i * ld + j, dtype);
            s += x;
            q += x * x;
        }
        sums[i] = s;
        if (sumsq)
            sumsq[i] = q;
    }
}

/* Column sums of the logical M x N matrix in binary64.  sums[j] receives the
 * sum of column j; sumsq (may be NULL) receives the sum of squares of column
 * j.  Every column's elements are added from row 0 to row M - 1; the rows
 * are visited one after the other (each row updates all N running sums), so
 * memory is read in its row-major order. */
void oracle_colsum(const void *src, double *sums, double *sumsq, int64_t M,
                   int64_t N, int64_t ld, int dtype)
{
    for (int64_t j = 0; j < N; ++j) {
        sums[j] = 0.0;
        if (sumsq)
            sumsq[j] = 0.0;
    }
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double x = element(src, i * ld + j, dtype);
            sums[j] += x;
            if (sumsq)
                sumsq[j] += x * x;
        }
    }
}

/* XOR of the n32 little-endian 32-bit words at src, one after the other. */
uint32_t oracle_xor_fold(const unsigned char *src, int64_t n32)
{
    uint32_t x = 0;
    for (int64_t k = 0; k < n32; ++k) {
        const unsigned char *b = src + 4 * k;
        uint32_t w = (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) |
                     ((uint32_t)b[3] << 24);
        x ^= w;
    }
    return x;
}
