/*
 * Blockwise-FP8 linear layer: plain CPU oracle.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. The CUDA path never
 * calls it, links it or shares a line of code with it.
 *
 * What it computes. The Puro-2B report runs the matrix multiplications of
 * its main linear layers in FP8 "following DeepSeek-V3's fine-grained block
 * quantisation", keeping sensitive state in BF16/FP32 (Puro-2B article on
 * en.roboind.com, section "FP8 takes advantage of the RTX 5090's low
 * precision efficiency"; the ainews.surl.tw article "Puro-2B Publishes a
 * Consumer-Grade GPU Pretraining Recipe ..." calls it "blockwise FP8").
 * The pages fix no further detail, so this file writes out the DeepSeek-V3
 * convention that the library adopts:
 *   - activation tiles of 1x128 along the contraction axis,
 *     weight blocks of 128x128;
 *   - codes in OCP E4M3FN (bias 7, 3 mantissa bits, largest finite 448,
 *     no infinities), rounded to nearest-even and saturated to +-448;
 *   - one FP32 scale per tile, s = amax / 448 (IEEE single division);
 *   - code = e4m3(fl32(x / s)): the quotient is rounded to FP32 first, then
 *     to e4m3 (two roundings, both to nearest-even);
 *   - an all-zero tile gets s = 0 and signed-zero codes, with no division;
 *   - GEMMs: per 128-wide chunk of the contraction axis the code products
 *     are summed, multiplied by the product of the two operands' chunk
 *     scales and accumulated; the oracle does this in FP64 and returns the
 *     FP64 result (no BF16 rounding), which the tests compare against.
 *
 * Style: every function is the definition written out, loop by loop, with
 * no blocking, fusion or reordering. Rows of the output are spread over
 * OpenMP threads, which changes no arithmetic.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -fopenmp -ffp-contract=off
 *        (no -ffast-math: IEEE division and subnormals are part of the
 *        definition; x86-64 runs with FTZ/DAZ off by default).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define TILE 128

/* ---------------------------------------------------------------------- */
/* Number formats                                                          */
/* ---------------------------------------------------------------------- */

/* bfloat16 -> binary32: a bf16 value is the top half of a binary32 word,
 * so widening is exact. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Value of an E4M3FN code, exactly, as a double.
 * Layout: sign(1) exponent(4, bias 7) mantissa(3).
 *   exponent 0       : subnormal, value = m/8 * 2^(1-7)  = m * 2^-9
 *   exponent 1..15   : normal,    value = (1+m/8) * 2^(e-7) = (8+m) * 2^(e-10)
 *   exponent 15, m 7 : NaN (the format has no infinities). */
double oracle_e4m3_value(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* Encode a finite binary32 value to E4M3FN: round to nearest, ties to even,
 * then saturate to the largest finite magnitude 448 (0x7E / 0xFE).
 * The sign of zero is kept. Written from the format: find the spacing of
 * the grid at |t|, divide by it (exact, a power of two), round the quotient
 * to an integer with ties to even, multiply back. */
uint8_t oracle_e4m3_encode(float t)
{
    uint8_t sign = signbit(t) ? 0x80 : 0x00;
    if (isnan(t))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)t);
    if (isinf(t) || a >= 448.0)
        return (uint8_t)(sign | 0x7E);

    double spacing;
    if (a < ldexp(1.0, -6)) {
        spacing = ldexp(1.0, -9);             /* subnormal range */
    } else {
        int e2;
        frexp(a, &e2);                        /* a = f * 2^e2, f in [0.5, 1) */
        spacing = ldexp(1.0, (e2 - 1) - 3);   /* binade [2^(e2-1), 2^e2): 8 steps */
    }
    double n = nearbyint(a / spacing);        /* default rounding: nearest-even */
    double v = n * spacing;
    if (v > 448.0)
        v = 448.0;                            /* satfinite */
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6))
        return (uint8_t)(sign | (uint8_t)(v / ldexp(1.0, -9)));
    int e2;
    double f = frexp(v, &e2);                 /* v = f * 2^e2 */
    int biased = (e2 - 1) + 7;
    int m = (int)((2.0 * f - 1.0) * 8.0);     /* exact: v has 3 fraction bits */
    return (uint8_t)(sign | (biased << 3) | m);
}

/* The scalar encoder applied to n values (for exhaustive format checks). */
void oracle_e4m3_encode_n(const float *t, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(t[i]);
}

/* Code value as an integer multiple of 2^-9 (every finite E4M3 value is one):
 *   subnormal: m,  normal: (8+m) * 2^(e-1).  A second, integer-only reading of
 *   the same format, used by the exact-integer GEMM below. */
int64_t oracle_e4m3_units(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 15;
    int m = c & 7;
    int64_t u = (e == 0) ? (int64_t)m : (int64_t)(8 + m) << (e - 1);
    return sign ? -u : u;
}

/* ---------------------------------------------------------------------- */
/* Quantisers                                                              */
/* ---------------------------------------------------------------------- */

/* Scale of one tile: s = fl32(amax / 448). amax is exact (a maximum of
 * bf16 magnitudes). */
static float tile_scale(float amax)
{
    return amax / 448.0f;
}

/* Code of one element given its tile's scale. s == 0 only for an all-zero
 * tile (the smallest non-zero bf16 magnitude divided by 448 is still a
 * non-zero binary32 subnormal); then the code is a signed zero. */
static uint8_t element_code(float x, float s)
{
    if (s == 0.0f)
        return signbit(x) ? 0x80 : 0x00;
    float t = x / s;                          /* IEEE binary32 division */
    return oracle_e4m3_encode(t);
}

/* 1x128 activation tiles along the columns.
 * x: bf16 [R][C] (row stride ldx elements); q: codes [R][C] (stride ldq);
 * s: [ceil(C/128)][R] chunk-major (row stride lds). A last chunk shorter
 * than 128 uses the amax of its valid elements only. */
void oracle_quantize_act(const uint16_t *x, int64_t R, int64_t C, int64_t ldx,
                         uint8_t *q, int64_t ldq, float *s, int64_t lds)
{
    int64_t nchunks = (C + TILE - 1) / TILE;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t c = 0; c < nchunks; ++c) {
            int64_t c0 = c * TILE;
            int64_t c1 = c0 + TILE < C ? c0 + TILE : C;
            float amax = 0.0f;
            for (int64_t j = c0; j < c1; ++j) {
                float v = fabsf(oracle_bf16_to_f32(x[r * ldx + j]));
                if (v > amax)
                    amax = v;
            }
            float sc = tile_scale(amax);
            s[c * lds + r] = sc;
            for (int64_t j = c0; j < c1; ++j)
                q[r * ldq + j] = element_code(oracle_bf16_to_f32(x[r * ldx + j]), sc);
        }
    }
}

/* 128x128 weight blocks. w: bf16 [N][K] (stride ldw); q: codes [N][K]
 * (stride ldq); s: [N/128][K/128] dense. N and K must be multiples of 128
 * (returns -1 otherwise). If qt is not NULL the codes are also written
 * transposed, qt[k][n] (stride ldqt); a block's scale serves both. */
int oracle_quantize_weight(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                           uint8_t *q, int64_t ldq, float *s,
                           uint8_t *qt, int64_t ldqt)
{
    if (N % TILE || K % TILE)
        return -1;
    int64_t nb = N / TILE, kb = K / TILE;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t bi = 0; bi < nb; ++bi) {
        for (int64_t bj = 0; bj < kb; ++bj) {
            float amax = 0.0f;
            for (int64_t i = bi * TILE; i < (bi + 1) * TILE; ++i)
                for (int64_t j = bj * TILE; j < (bj + 1) * TILE; ++j) {
                    float v = fabsf(oracle_bf16_to_f32(w[i * ldw + j]));
                    if (v > amax)
                        amax = v;
                }
            float sc = tile_scale(amax);
            s[bi * kb + bj] = sc;
            for (int64_t i = bi * TILE; i < (bi + 1) * TILE; ++i)
                for (int64_t j = bj * TILE; j < (bj + 1) * TILE; ++j) {
                    uint8_t code = element_code(oracle_bf16_to_f32(w[i * ldw + j]), sc);
                    q[i * ldq + j] = code;
                    if (qt)
                        qt[j * ldqt + i] = code;
                }
        }
    }
    return 0;
}

/* Transposed 1x128 tiles: the tiles run down the columns of x, i.e. along
 * the rows R, which is the contraction axis of the weight-gradient GEMM.
 * x: bf16 [R][C] (stride ldx); qt: codes [C][R128] (stride ldqt >= R128,
 * R128 = R rounded up to 128); st: [R128/128][C] (stride ldst).
 * Pad positions R <= r < R128 get code 0x00; a chunk's scale covers its
 * valid rows only. */
void oracle_quantize_transpose(const uint16_t *x, int64_t R, int64_t C, int64_t ldx,
                               uint8_t *qt, int64_t ldqt, float *st, int64_t ldst)
{
    int64_t nchunks = (R + TILE - 1) / TILE;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t rb = 0; rb < nchunks; ++rb) {
            int64_t r0 = rb * TILE;
            int64_t r1 = r0 + TILE < R ? r0 + TILE : R;
            float amax = 0.0f;
            for (int64_t r = r0; r < r1; ++r) {
                float v = fabsf(oracle_bf16_to_f32(x[r * ldx + c]));
                if (v > amax)
                    amax = v;
            }
            float sc = tile_scale(amax);
            st[rb * ldst + c] = sc;
            for (int64_t r = r0; r < r0 + TILE; ++r)
                qt[c * ldqt + r] = (r < R) ? element_code(oracle_bf16_to_f32(x[r * ldx + c]), sc)
                                           : (uint8_t)0x00;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* GEMMs (FP64 reference; no BF16 rounding of the result)                   */
/* ---------------------------------------------------------------------- */

/* Output rows to compute: rows[i] for i < nrows, or 0..nrows-1 if rows is NULL. */
static int64_t pick_row(const int64_t *rows, int64_t i)
{
    return rows ? rows[i] : i;
}

/* Forward, Y = X W^T:
 *   Y[m][n] = sum_kb sX[kb][m] * sW[n/128][kb] * sum_{k in kb} v(qX[m][k]) v(qW[n][k])
 * qX [M][K] (ldqx), sX [K/128][M] (ldsx), qW [N][K] (ldqw), sW [N/128][K/128].
 * y: [nrows][N], FP64. K and N multiples of 128. */
void oracle_gemm_fwd(const uint8_t *qx, int64_t ldqx, const float *sx, int64_t ldsx,
                     const uint8_t *qw, int64_t ldqw, const float *sw,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t *rows, int64_t nrows, double *y)
{
    (void)M;
    int64_t kchunks = K / TILE;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = pick_row(rows, i);
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t kb = 0; kb < kchunks; ++kb) {
                double part = 0.0;
                for (int64_t k = kb * TILE; k < (kb + 1) * TILE; ++k)
                    part += oracle_e4m3_value(qx[m * ldqx + k]) * oracle_e4m3_value(qw[n * ldqw + k]);
                double scale = (double)sx[kb * ldsx + m] * (double)sw[(n / TILE) * kchunks + kb];
                acc += scale * part;
            }
            y[i * N + n] = acc;
        }
    }
}

/* Input gradient, dX = dY W (contraction over the N outputs of the layer):
 *   dX[m][k] = sum_nb sdY[nb][m] * sW[nb][k/128] * sum_{n in nb} v(qdY[m][n]) v(qW[n][k])
 * qdY [M][N] (ldqdy), sdY [N/128][M] (ldsdy), qW [N][K] (ldqw), sW [N/128][K/128].
 * dx: [nrows][K], FP64. */
void oracle_gemm_dgrad(const uint8_t *qdy, int64_t ldqdy, const float *sdy, int64_t ldsdy,
                       const uint8_t *qw, int64_t ldqw, const float *sw,
                       int64_t M, int64_t N, int64_t K,
                       const int64_t *rows, int64_t nrows, double *dx)
{
    (void)M;
    int64_t nchunks = N / TILE, kchunks = K / TILE;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = pick_row(rows, i);
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t nb = 0; nb < nchunks; ++nb) {
                double part = 0.0;
                for (int64_t n = nb * TILE; n < (nb + 1) * TILE; ++n)
                    part += oracle_e4m3_value(qdy[m * ldqdy + n]) * oracle_e4m3_value(qw[n * ldqw + k]);
                double scale = (double)sdy[nb * ldsdy + m] * (double)sw[nb * kchunks + k / TILE];
                acc += scale * part;
            }
            dx[i * K + k] = acc;
        }
    }
}

/* Weight gradient, dW = dY^T X (contraction over the M tokens, padded to
 * M128 with zero codes):
 *   dW[n][k] = sum_mb sdYt[mb][n] * sXt[mb][k] * sum_{m in mb} v(qdYt[n][m]) v(qXt[k][m])
 * qdYt [N][M128] (ldqdyt), sdYt [M128/128][N] (ldsdyt),
 * qXt [K][M128] (ldqxt), sXt [M128/128][K] (ldsxt). dw: [nrows][K], FP64,
 * rows index n. */
void oracle_gemm_wgrad(const uint8_t *qdyt, int64_t ldqdyt, const float *sdyt, int64_t ldsdyt,
                       const uint8_t *qxt, int64_t ldqxt, const float *sxt, int64_t ldsxt,
                       int64_t M, int64_t N, int64_t K,
                       const int64_t *rows, int64_t nrows, double *dw)
{
    (void)N;
    int64_t mchunks = (M + TILE - 1) / TILE;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = pick_row(rows, i);
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t mb = 0; mb < mchunks; ++mb) {
                double part = 0.0;
                for (int64_t m = mb * TILE; m < (mb + 1) * TILE; ++m)
                    part += oracle_e4m3_value(qdyt[n * ldqdyt + m]) * oracle_e4m3_value(qxt[k * ldqxt + m]);
                double scale = (double)sdyt[mb * ldsdyt + n] * (double)sxt[mb * ldsxt + k];
                acc += scale * part;
            }
            dw[i * K + k] = acc;
        }
    }
}

/* Forward GEMM again, with every 128-term chunk summed exactly in int64 on
 * the integer reading of the codes (units of 2^-9, so a product is in units
 * of 2^-18). Used to check that the FP64 chunk sums above are exact. */
void oracle_gemm_fwd_i64(const uint8_t *qx, int64_t ldqx, const float *sx, int64_t ldsx,
                         const uint8_t *qw, int64_t ldqw, const float *sw,
                         int64_t M, int64_t N, int64_t K,
                         const int64_t *rows, int64_t nrows, double *y)
{
    (void)M;
    int64_t kchunks = K / TILE;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = pick_row(rows, i);
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t kb = 0; kb < kchunks; ++kb) {
                int64_t part = 0;
                for (int64_t k = kb * TILE; k < (kb + 1) * TILE; ++k)
                    part += oracle_e4m3_units(qx[m * ldqx + k]) * oracle_e4m3_units(qw[n * ldqw + k]);
                double scale = (double)sx[kb * ldsx + m] * (double)sw[(n / TILE) * kchunks + kb];
                acc += scale * ldexp((double)part, -18);
            }
            y[i * N + n] = acc;
        }
    }
}
