/*
 * fp8bs oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the fine-grained FP8
 * path computes.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg may load it.  It shares no code, header, table or constant
 * generator with the CUDA library; the two never import each other.
 *
 * Sources (DeepSeek-V3-style FP8 training scheme, scraped pages):
 *  - "Should Fixing Deepseek Take 60 Steps?", Figure 7 (a) passage: activations
 *    are grouped and scaled per 1x128 tile (one token, 128 channels); weights
 *    per 128x128 block (128 input x 128 output channels).
 *  - same page, max-abs scaling passage: the tensor is aligned to the FP8 range
 *    by mapping its maximum absolute value onto the largest FP8 value.
 *  - untitled page at jp-study.kr, hybrid-format passage: E4M3 (4-bit
 *    exponent, 3-bit mantissa) is used on all tensors.
 *  - page at why-be.why-be.co.kr, online-amax passage: the max-abs is computed
 *    online for every 1x128 activation tile or 128x128 weight block.
 *  - "Should Fixing Deepseek Take 60 Steps?", Figure 6 passage: the GEMMs take
 *    FP8 inputs and produce BF16 or FP32.
 *  - untitled page at jp-study.kr, Figure 7 (b) passage: partial sums are
 *    promoted to FP32 on CUDA cores, where the scales are applied.
 *
 * Readings taken where the pages are silent:
 *  - E4M3 is the OCP "E4M3FN" layout: bias 7, no infinities, S.1111.111 = NaN,
 *    largest finite 448.  Encoding rounds to nearest, ties to even, and
 *    saturates finite overflow to +-448 ("satfinite").  The sign of zero is
 *    kept.
 *  - Scale s = fl32(amax / 448) (stored, used to dequantize).  The values are
 *    brought into range by multiplying with r = fl32(448 / amax): code =
 *    enc(fl32(x * r)).  If r is not finite (amax == 0, or amax so small that
 *    448/amax overflows fp32) the tile counts as all-zero: s = r = 1.
 *  - A tile is exactly 128 elements (or 128x128); tiled extents must be
 *    multiples of 128.
 *  - The promotion interval is one 128-deep K-slab: every slab's partial sum is
 *    multiplied by the A-tile scale and the B-block scale of that slab and
 *    added into a high-precision accumulator.
 *
 * Precision: quantization uses IEEE binary32 exactly as stated above (build
 * with -ffp-contract=off, no fast-math).  The GEMM accumulates in binary64; the
 * inner 128-term sum of decoded-code products is exact in binary64 (each
 * product has at most 8 significant bits and exponents within [-18, 18]).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ E4M3 */

/* Value of an E4M3 code, from the format definition. */
double fp8bs_oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);   /* normal: 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* Round an fp32 value to the nearest E4M3 value (ties to even), saturating
 * magnitudes at or above 448 to 448.  NaN maps to the NaN code. */
uint8_t fp8bs_oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    int ex, E, field, mant;
    double quantum, steps, val;

    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;

    /* a = f * 2^ex with f in [0.5, 1): floor(log2(a)) = ex - 1. */
    frexp(a, &ex);
    E = ex - 1;
    if (E < -6)
        E = -6;                            /* subnormal range shares 2^-9 spacing */
    quantum = ldexp(1.0, E - 3);           /* spacing of representable values */
    steps = nearbyint(a / quantum);        /* exact quotient; RNE to integer */
    val = steps * quantum;
    if (val > 448.0)                       /* cannot happen below 448; kept for clarity */
        val = 448.0;
    if (val == 0.0)
        return sign;

    frexp(val, &ex);
    E = ex - 1;
    if (E < -6) {                          /* subnormal: val = mant * 2^-9 */
        field = 0;
        mant = (int)ldexp(val, 9);
    } else {                               /* normal: val = (1 + mant/8) * 2^E */
        field = E + 7;
        mant = (int)(ldexp(val, -E) * 8.0) - 8;
    }
    return (uint8_t)(sign | (field << 3) | mant);
}

/* Element-wise encode of n fp32 values (no scaling). */
void fp8bs_oracle_e4m3_encode_n(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fp8bs_oracle_e4m3_encode(v[i]);
}

/* ---------------------------------------------------------- input values */

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Element (row, col) of a row-major matrix given as fp32 or as raw bf16 bits. */
static float load_elem(const void *x, int dtype, int64_t ld, int64_t row, int64_t col)
{
    if (dtype == ORACLE_F32)
        return ((const float *)x)[row * ld + col];
    {
        uint32_t bits = (uint32_t)((const uint16_t *)x)[row * ld + col] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return f;                          /* bf16 -> fp32 is exact */
    }
}

/* --------------------------------------------------------- tile scaling */

/* Scale and multiplier for a tile whose max-abs is amax. */
static void tile_scale(float amax, float *s, float *r)
{
    volatile float rr = 448.0f / amax;     /* IEEE binary32 division, RNE */
    if (isinf(rr)) {                       /* all-zero (or numerically zero) tile */
        *s = 1.0f;
        *r = 1.0f;
        return;
    }
    *s = amax / 448.0f;
    *r = rr;
}

static uint8_t quantize_value(float x, float r)
{
    volatile float y = x * r;              /* binary32 multiply, RNE */
    return fp8bs_oracle_e4m3_encode(y);
}

/* ----------------------------------------------------------- quantizers */

/* 1x128 activation tiles: x [M x K] row-major (leading dim ldx elements).
 * q [M x K] (ldq bytes per row); s [K/128][lds] with s[kb*lds + m]. */
void fp8bs_oracle_quant_act_1x128(const void *x, int dtype, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t *q, int64_t ldq, float *s, int64_t lds)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < K / 128; ++kb) {
            float amax = 0.0f, sc, r;
            for (int c = 0; c < 128; ++c) {
                float a = fabsf(load_elem(x, dtype, ldx, m, kb * 128 + c));
                if (a > amax)
                    amax = a;
            }
            tile_scale(amax, &sc, &r);
            for (int c = 0; c < 128; ++c)
                q[m * ldq + kb * 128 + c] =
                    quantize_value(load_elem(x, dtype, ldx, m, kb * 128 + c), r);
            s[kb * lds + m] = sc;
        }
    }
}

/* 128x1 tiles (128 tokens of one channel): x [T x C] row-major.
 * Codes are written transposed: qT [C x T] with qT[c*ldq + t];
 * s [T/128][lds] with s[tb*lds + c]. */
void fp8bs_oracle_quant_act_128x1(const void *x, int dtype, int64_t T, int64_t C, int64_t ldx,
                                  uint8_t *qT, int64_t ldq, float *s, int64_t lds)
{
    for (int64_t tb = 0; tb < T / 128; ++tb) {
        for (int64_t c = 0; c < C; ++c) {
            float amax = 0.0f, sc, r;
            for (int t = 0; t < 128; ++t) {
                float a = fabsf(load_elem(x, dtype, ldx, tb * 128 + t, c));
                if (a > amax)
                    amax = a;
            }
            tile_scale(amax, &sc, &r);
            for (int t = 0; t < 128; ++t)
                qT[c * ldq + tb * 128 + t] =
                    quantize_value(load_elem(x, dtype, ldx, tb * 128 + t, c), r);
            s[tb * lds + c] = sc;
        }
    }
}

/* 128x128 weight blocks: w [R x C] row-major.  q [R x C] (ldq); optional
 * qT [C x R] (ldqT) holding the same codes transposed; s [R/128][C/128]. */
void fp8bs_oracle_quant_w_128x128(const void *w, int dtype, int64_t R, int64_t C, int64_t ldw,
                                  uint8_t *q, int64_t ldq, uint8_t *qT, int64_t ldqT, float *s)
{
    for (int64_t rb = 0; rb < R / 128; ++rb) {
        for (int64_t cb = 0; cb < C / 128; ++cb) {
            float amax = 0.0f, sc, r;
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    float a = fabsf(load_elem(w, dtype, ldw, rb * 128 + i, cb * 128 + j));
                    if (a > amax)
                        amax = a;
                }
            tile_scale(amax, &sc, &r);
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    int64_t row = rb * 128 + i, col = cb * 128 + j;
                    uint8_t code = quantize_value(load_elem(w, dtype, ldw, row, col), r);
                    q[row * ldq + col] = code;
                    if (qT)
                        qT[col * ldqT + row] = code;
                }
            s[rb * (C / 128) + cb] = sc;
        }
    }
}

/* ----------------------------------------------------------------- GEMM */

/* Layouts of the B-operand scales (the same three layouts the library takes):
 *  0 BLOCK_NK : sb[(n/128)*ldsb + k/128]   (one scale per 128 x 128 block)
 *  1 BLOCK_KN : sb[(k/128)*ldsb + n/128]
 *  2 PERCOL   : sb[(k/128)*ldsb + n]       (128x1 tiles along K, per column) */
static double b_scale(const float *sb, int mode, int64_t ldsb, int64_t kb, int64_t n)
{
    if (mode == 0)
        return (double)sb[(n / 128) * ldsb + kb];
    if (mode == 1)
        return (double)sb[kb * ldsb + n / 128];
    return (double)sb[kb * ldsb + n];
}

/* One output element of the block-scaled GEMM
 *   C[i][j] = sum over 128-deep K-slabs kb of
 *             ( sum_{k in slab} dec(A[i][k]) * dec(B[j][k]) ) * sa[kb][i] * sb(kb, j)
 * A [M x K] codes, K contiguous (lda); B [N x K] codes, K contiguous (ldb);
 * sa[kb*ldsa + i].  Also returns S_abs = sum_k |a_ik * b_kj| over the
 * dequantized operands, the scale of the tolerance bound. */
static void gemm_one(int64_t K, const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                     const uint8_t *B, int64_t ldb, const float *sb, int mode, int64_t ldsb,
                     const double *dec, int64_t i, int64_t j, double *c_out, double *abs_out)
{
    double c = 0.0, sabs = 0.0;
    for (int64_t kb = 0; kb < K / 128; ++kb) {
        double part = 0.0, part_abs = 0.0;
        double scale = (double)sa[kb * ldsa + i] * b_scale(sb, mode, ldsb, kb, j);
        for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
            double p = dec[A[i * lda + k]] * dec[B[j * ldb + k]];
            part += p;
            part_abs += fabs(p);
        }
        c += part * scale;
        sabs += part_abs * fabs(scale);
    }
    *c_out = c;
    *abs_out = sabs;
}

static void decode_table(double dec[256])
{
    for (int v = 0; v < 256; ++v)
        dec[v] = fp8bs_oracle_e4m3_decode((uint8_t)v);
}

/* Full M x N output into c_ref / s_abs (row-major, N per row). */
void fp8bs_oracle_gemm(int64_t M, int64_t N, int64_t K,
                       const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                       const uint8_t *B, int64_t ldb, const float *sb, int mode, int64_t ldsb,
                       double *c_ref, double *s_abs)
{
    double dec[256];
    decode_table(dec);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            gemm_one(K, A, lda, sa, ldsa, B, ldb, sb, mode, ldsb, dec, i, j,
                     &c_ref[i * N + j], &s_abs[i * N + j]);
}

/* Selected output elements (rows[e], cols[e]) for e < count. */
void fp8bs_oracle_gemm_elements(int64_t K,
                                const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                                const uint8_t *B, int64_t ldb, const float *sb, int mode, int64_t ldsb,
                                int64_t count, const int64_t *rows, const int64_t *cols,
                                double *c_ref, double *s_abs)
{
    double dec[256];
    decode_table(dec);
    for (int64_t e = 0; e < count; ++e)
        gemm_one(K, A, lda, sa, ldsa, B, ldb, sb, mode, ldsb, dec, rows[e], cols[e],
                 &c_ref[e], &s_abs[e]);
}

/* ------------------------------------------------- MX (microscaling) variant
 *
 * Sources: "Should Fixing Deepseek Take 60 Steps?", Figure 7 (a) passage and
 * the page at why-be.why-be.co.kr, accumulation-precision passage: both point
 * to microscaling formats, with group scaling done by the tensor cores of the
 * next GPU generation, as the direction fine-grained quantization takes.
 *
 * Readings taken where the pages are silent:
 *  - Groups are 1x32 along the contraction axis for both operands.  A group's
 *    scale is a power of two 2^e stored as an unsigned 8-bit exponent
 *    (UE8M0: byte = e + 127, e in [-127, 127]).
 *  - e is the smallest integer with amax <= 448 * 2^e (the scale rounded up to
 *    a power of two, so no element overflows), clamped to [-127, 127]; an
 *    all-zero group gets e = 0.
 *  - code = enc(fl32(x * 2^-e)): one binary32 multiply by an exact power of
 *    two, then the E4M3 rounding of the tile quantizers.
 *  - Storage of the exponent bytes: the four groups of one row inside one
 *    128-wide K block share a 32-bit word, group 4kb+j in byte j:
 *    sf[(kb*ldsf + r)*4 + j], ldsf >= rows.
 */

/* Smallest e with amax <= 448 * 2^e, searched from a log2 estimate. */
static int mx_group_exponent(float amax)
{
    int e;
    if (amax == 0.0f)
        return 0;
    e = (int)ceil(log2((double)amax / 448.0));
    while ((double)amax > ldexp(448.0, e))
        ++e;
    while ((double)amax <= ldexp(448.0, e - 1))
        --e;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* x [R x K] row-major (ldx elements) -> q [R x K] (ldq bytes per row) and the
 * exponent bytes sf as described above.  K % 128 == 0. */
void fp8bs_oracle_mx_quant_1x32(const void *x, int dtype, int64_t R, int64_t K, int64_t ldx,
                                uint8_t *q, int64_t ldq, uint8_t *sf, int64_t ldsf)
{
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t g = 0; g < K / 32; ++g) {
            float amax = 0.0f, mult;
            int e;
            for (int c = 0; c < 32; ++c) {
                float a = fabsf(load_elem(x, dtype, ldx, r, g * 32 + c));
                if (a > amax)
                    amax = a;
            }
            e = mx_group_exponent(amax);
            mult = ldexpf(1.0f, -e);       /* exact: 2^-127 .. 2^127 are binary32 values */
            for (int c = 0; c < 32; ++c) {
                volatile float y = load_elem(x, dtype, ldx, r, g * 32 + c) * mult;
                q[r * ldq + g * 32 + c] = fp8bs_oracle_e4m3_encode(y);
            }
            sf[((g / 4) * ldsf + r) * 4 + g % 4] = (uint8_t)(e + 127);
        }
    }
}

/* One output element of the MX GEMM
 *   C[i][j] = sum over 32-deep K groups g of
 *             ( sum_{k in g} dec(A[i][k]) * dec(B[j][k]) ) * 2^(ea(i,g) + eb(j,g))
 * A [M x K] codes (lda), B [N x K] codes (ldb); exponent bytes as above.
 * Also S_abs = sum_k |a_ik * b_jk| over the dequantized operands. */
static void mx_gemm_one(int64_t K, const uint8_t *A, int64_t lda, const uint8_t *sfa,
                        int64_t ldsfa, const uint8_t *B, int64_t ldb, const uint8_t *sfb,
                        int64_t ldsfb, const double *dec, int64_t i, int64_t j,
                        double *c_out, double *abs_out)
{
    double c = 0.0, sabs = 0.0;
    for (int64_t g = 0; g < K / 32; ++g) {
        double part = 0.0, part_abs = 0.0, scale;
        int ea = (int)sfa[((g / 4) * ldsfa + i) * 4 + g % 4] - 127;
        int eb = (int)sfb[((g / 4) * ldsfb + j) * 4 + g % 4] - 127;
        scale = ldexp(1.0, ea + eb);
        for (int64_t k = g * 32; k < g * 32 + 32; ++k) {
            double p = dec[A[i * lda + k]] * dec[B[j * ldb + k]];
            part += p;
            part_abs += fabs(p);
        }
        c += part * scale;
        sabs += part_abs * scale;
    }
    *c_out = c;
    *abs_out = sabs;
}

void fp8bs_oracle_mx_gemm(int64_t M, int64_t N, int64_t K,
                          const uint8_t *A, int64_t lda, const uint8_t *sfa, int64_t ldsfa,
                          const uint8_t *B, int64_t ldb, const uint8_t *sfb, int64_t ldsfb,
                          double *c_ref, double *s_abs)
{
    double dec[256];
    decode_table(dec);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            mx_gemm_one(K, A, lda, sfa, ldsfa, B, ldb, sfb, ldsfb, dec, i, j,
                        &c_ref[i * N + j], &s_abs[i * N + j]);
}

void fp8bs_oracle_mx_gemm_elements(int64_t K,
                                   const uint8_t *A, int64_t lda, const uint8_t *sfa, int64_t ldsfa,
                                   const uint8_t *B, int64_t ldb, const uint8_t *sfb, int64_t ldsfb,
                                   int64_t count, const int64_t *rows, const int64_t *cols,
                                   double *c_ref, double *s_abs)
{
    double dec[256];
    decode_table(dec);
    for (int64_t e = 0; e < count; ++e)
        mx_gemm_one(K, A, lda, sfa, ldsfa, B, ldb, sfb, ldsfb, dec, rows[e], cols[e],
                    &c_ref[e], &s_abs[e]);
}
