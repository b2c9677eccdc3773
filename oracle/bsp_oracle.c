/*
 * CPU oracle for the bitmap-encoded unstructured sparse matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA library is checked against.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it; the library itself never
 * calls it and shares no code, header, table or helper with it.
 *
 * What it computes, and where each piece comes from:
 *
 *  - The format (TCA-BME), from "SpInfer: How bitmaps make sparse LLMs
 *    actually fast", sections "How TCA-BME addresses the indexing overhead"
 *    and "The Values array and why it's confusing at first":
 *      * BitmapTile (BT) = 8x8 elements, one uint64 bitmap, one bit per
 *        element, set <=> the element is nonzero;
 *      * TCTile = 16x16 = 2x2 BTs; GroupTile (GT) = several TCTiles;
 *      * Values = the nonzeros only, packed in GroupTile -> TCTile ->
 *        BitmapTile order; a value's index inside its tile is the number of
 *        nonzeros before it (masked popcount, section "Shared Memory Bitmap
 *        Decoding (SMBD)");
 *      * one 4-byte offset per GT plus one (NGT+1 entries).
 *    Readings where the page is silent (all fixed here, stated once):
 *      * GT = 64x64; GTs row-major over the (M/64)x(K/64) grid;
 *      * TCTiles row-major inside a GT (4x4);
 *      * the 4 BTs of a TCTile in mma A-register order:
 *        b=0 rows 0-7/cols 0-7, b=1 rows 8-15/cols 0-7,
 *        b=2 rows 0-7/cols 8-15, b=3 rows 8-15/cols 8-15;
 *      * global BT index g = (t*16 + tc)*4 + b;
 *      * bit p = 8*row + col inside the BT (row-major, bit 0 = top left);
 *      * "nonzero" = raw element bits != 0 (so -0.0, NaN, Inf are payload);
 *      * offsets are uint32 element counts, offsets[t] = nonzeros in GTs < t.
 *  - The product, from "Unified Static-Dynamic Pruning for Efficient LLM
 *    Inference", section 3.1 (W in R^{MxK}, X in R^{KxN}): the method
 *    reaches exactly the dense product ("load as sparse, compute as dense"),
 *    so the oracle is the dense definition Y[n][m] = sum_k W[m][k]*X[n][k],
 *    taken from the original dense W, in fp64 for fp16 inputs (every fp16
 *    product is exact in fp64) and in int64 for int8 inputs.
 *
 * X is stored [N][K] and Y [N][M] (K and M contiguous), the [tokens,
 * features] layout; this is the column-major view of the pages' KxN and MxN.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GT_DIM 64

/* IEEE 754 binary16 -> double, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Count set bits one at a time: no tricks, so it can be read at a glance. */
int oracle_popcount64(uint64_t x)
{
    int n = 0;
    for (int i = 0; i < 64; ++i)
        n += (int)((x >> i) & 1u);
    return n;
}

/* Number of set bits strictly below position p (the masked popcount). */
int oracle_rank(uint64_t bitmap, int p)
{
    uint64_t mask = (p >= 64) ? ~0ull : ((1ull << p) - 1ull);
    return oracle_popcount64(bitmap & mask);
}

/* (r, c) -> (global BT index g, bit p) under the readings above. */
void oracle_locate(int64_t K, int64_t r, int64_t c, int64_t *g, int *p)
{
    int64_t gi = r / 64, gj = c / 64;
    int64_t t = gi * (K / 64) + gj;
    int64_t rr = r % 64, cc = c % 64;
    int64_t tc = (rr / 16) * 4 + (cc / 16);
    int64_t b = ((rr % 16) / 8) + 2 * ((cc % 16) / 8);
    *g = (t * 16 + tc) * 4 + b;
    *p = (int)((rr % 8) * 8 + (cc % 8));
}

/* (g, p) -> (r, c), the inverse of oracle_locate. */
void oracle_position(int64_t K, int64_t g, int p, int64_t *r, int64_t *c)
{
    int64_t t = g / 64, tc = (g / 4) % 16, b = g % 4;
    int64_t gi = t / (K / 64), gj = t % (K / 64);
    *r = gi * 64 + (tc / 4) * 16 + (b % 2) * 8 + p / 8;
    *c = gj * 64 + (tc % 4) * 16 + (b / 2) * 8 + p % 8;
}

static int elem_nonzero(const uint8_t *W, int eb, int64_t idx)
{
    const uint8_t *e = W + idx * eb;
    for (int i = 0; i < eb; ++i)
        if (e[i]) return 1;
    return 0;
}

/*
 * Pass 1 of the encoder: bitmaps[NBT] and the nonzero count.
 * W: raw elements, row-major [M][K], eb bytes each (2 = fp16, 1 = int8).
 * Returns NNZ.
 */
uint64_t oracle_encode_bitmaps(const void *Wv, int eb, int64_t M, int64_t K,
                               uint64_t *bitmaps)
{
    const uint8_t *W = (const uint8_t *)Wv;
    int64_t NBT = M * K / 64;
    uint64_t nnz = 0;
    memset(bitmaps, 0, (size_t)NBT * sizeof(uint64_t));
    for (int64_t r = 0; r < M; ++r)
        for (int64_t c = 0; c < K; ++c)
            if (elem_nonzero(W, eb, r * K + c)) {
                int64_t g; int p;
                oracle_locate(K, r, c, &g, &p);
                bitmaps[g] |= 1ull << p;
                ++nnz;
            }
    return nnz;
}

/*
 * Pass 2 of the encoder: offsets[NGT+1] and values[NNZ].
 * Values are appended for g ascending and, inside a BT, for p ascending.
 */
void oracle_encode_values(const void *Wv, int eb, int64_t M, int64_t K,
                          const uint64_t *bitmaps, uint32_t *offsets,
                          void *valuesv)
{
    const uint8_t *W = (const uint8_t *)Wv;
    uint8_t *values = (uint8_t *)valuesv;
    int64_t NGT = (M / 64) * (K / 64);
    uint64_t k = 0;
    for (int64_t t = 0; t < NGT; ++t) {
        offsets[t] = (uint32_t)k;
        for (int64_t g = t * 64; g < (t + 1) * 64; ++g)
            for (int p = 0; p < 64; ++p)
                if ((bitmaps[g] >> p) & 1u) {
                    int64_t r, c;
                    oracle_position(K, g, p, &r, &c);
                    memcpy(values + k * eb, W + (r * K + c) * eb, (size_t)eb);
                    ++k;
                }
    }
    offsets[NGT] = (uint32_t)k;
}

/*
 * Decoder: W_out[r][c] = bit set ? values[offsets[t] + (nonzeros of the
 * earlier BTs of GT t) + rank(bitmap, p)] : 0.
 */
void oracle_decode(const uint64_t *bitmaps, const uint32_t *offsets,
                   const void *valuesv, int eb, int64_t M, int64_t K,
                   void *Woutv)
{
    const uint8_t *values = (const uint8_t *)valuesv;
    uint8_t *Wout = (uint8_t *)Woutv;
    for (int64_t r = 0; r < M; ++r)
        for (int64_t c = 0; c < K; ++c) {
            int64_t g; int p;
            oracle_locate(K, r, c, &g, &p);
            uint8_t *dst = Wout + (r * K + c) * eb;
            if (!((bitmaps[g] >> p) & 1u)) {
                memset(dst, 0, (size_t)eb);
                continue;
            }
            int64_t t = g / 64;
            uint64_t idx = offsets[t];
            for (int64_t g2 = t * 64; g2 < g; ++g2)
                idx += (uint64_t)oracle_popcount64(bitmaps[g2]);
            idx += (uint64_t)oracle_rank(bitmaps[g], p);
            memcpy(dst, values + idx * eb, (size_t)eb);
        }
}

/*
 * fp16 product in fp64: Y[n][m] = sum_k W[m][k]*X[n][k] and
 * sumabs[n][m] = sum_k |W[m][k]*X[n][k]| (for the error bound).
 * W: uint16 [M][K]; X: uint16 [N][K]; Y, sumabs: double [N][M].
 */
void oracle_spmm_f16(const uint16_t *W, const uint16_t *X, int64_t M,
                     int64_t K, int64_t N, double *Y, double *sumabs)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double prod = oracle_half_to_double(W[m * K + k]) *
                              oracle_half_to_double(X[n * K + k]);
                s += prod;
                a += fabs(prod);
            }
            Y[n * M + m] = s;
            if (sumabs) sumabs[n * M + m] = a;
        }
}

/* int8 product in int64: Y[n][m] = sum_k W[m][k]*X[n][k]. */
void oracle_spmm_i8(const int8_t *W, const int8_t *X, int64_t M, int64_t K,
                    int64_t N, int64_t *Y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k)
                s += (int64_t)W[m * K + k] * (int64_t)X[n * K + k];
            Y[n * M + m] = s;
        }
}

/*
 * Scaled int8 output: Yf[n][m] = (float)acc[n][m] * scale[m], one IEEE
 * round-to-nearest int->float conversion, then one round-to-nearest fp32
 * multiply (built with -ffp-contract=off; a single product has nothing to
 * contract anyway).
 */
void oracle_scale_i8(const int64_t *acc, const float *scale, int64_t M,
                     int64_t N, float *Yf)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) {
            volatile float a = (float)acc[n * M + m];
            volatile float p = a * scale[m];
            Yf[n * M + m] = p;
        }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
