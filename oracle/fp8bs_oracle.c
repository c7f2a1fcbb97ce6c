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
 *
 * Threads: the quantizers hand whole tiles, the GEMMs whole output rows (or,
 * for the element lists, whole elements) to POSIX threads.  Every tile and
 * every element is still computed by the same loop, in the same order, by one
 * thread, so the results do not depend on the thread count; threads only split
 * the list of independent pieces.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

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

/* --------------------------------------------------------------- threads */

static int g_threads = 0;          /* 0: one per online CPU */

/* Number of threads the quantizers and GEMMs use (n <= 0: one per online CPU). */
void fp8bs_oracle_set_threads(int n)
{
    g_threads = n > 0 ? n : 0;
}

int fp8bs_oracle_threads(void)
{
    long n = g_threads > 0 ? g_threads : sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1)
        n = 1;
    if (n > 256)
        n = 256;
    return (int)n;
}

/* Run body(ctx, t, nt) on nt threads, t = 0 .. nt-1; thread t takes items
 * t, t + nt, t + 2 nt, ... of whatever list the body walks. */
struct thread_arg {
    void (*body)(void *, int, int);
    void *ctx;
    int t, nt;
};

static void *thread_main(void *p)
{
    struct thread_arg *a = (struct thread_arg *)p;
    a->body(a->ctx, a->t, a->nt);
    return NULL;
}

static void run_threads(void (*body)(void *, int, int), void *ctx, int64_t items)
{
    int nt = fp8bs_oracle_threads(), t, started = 0;
    pthread_t tid[256];
    struct thread_arg args[256];
    if (items < nt)
        nt = items > 0 ? (int)items : 1;
    for (t = 0; t < nt; ++t) {
        args[t].body = body;
        args[t].ctx = ctx;
        args[t].t = t;
        args[t].nt = nt;
    }
    for (t = 1; t < nt; ++t) {
        if (pthread_create(&tid[t], NULL, thread_main, &args[t]) != 0)
            break;
        started = t;
    }
    /* items of threads that could not be started run here, in this thread */
    for (t = started + 1; t < nt; ++t)
        body(ctx, t, nt);
    body(ctx, 0, nt);
    for (t = 1; t <= started; ++t)
        pthread_join(tid[t], NULL);
}

/* ----------------------------------------------------------- quantizers */

/* Arguments of one quantizer call, shared by its threads; every tile is
 * quantized whole by one thread, so the result does not depend on how many
 * threads there are. */
struct quant_job {
    const void *x;
    int dtype;
    int64_t rows, cols, ldx;
    uint8_t *q;
    int64_t ldq;
    uint8_t *qT;
    int64_t ldqT;
    float *s;
    int64_t lds;
};

/* 1x128 tiles of rows m = t, t + nt, ... */
static void quant_1x128_rows(void *p, int t, int nt)
{
    const struct quant_job *j = (const struct quant_job *)p;
    for (int64_t m = t; m < j->rows; m += nt) {
        for (int64_t kb = 0; kb < j->cols / 128; ++kb) {
            float amax = 0.0f, sc, r;
            for (int c = 0; c < 128; ++c) {
                float a = fabsf(load_elem(j->x, j->dtype, j->ldx, m, kb * 128 + c));
                if (a > amax)
                    amax = a;
            }
            tile_scale(amax, &sc, &r);
            for (int c = 0; c < 128; ++c)
                j->q[m * j->ldq + kb * 128 + c] =
                    quantize_value(load_elem(j->x, j->dtype, j->ldx, m, kb * 128 + c), r);
            j->s[kb * j->lds + m] = sc;
        }
    }
}

/* 1x128 activation tiles: x [M x K] row-major (leading dim ldx elements).
 * q [M x K] (ldq bytes per row); s [K/128][lds] with s[kb*lds + m]. */
void fp8bs_oracle_quant_act_1x128(const void *x, int dtype, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t *q, int64_t ldq, float *s, int64_t lds)
{
    struct quant_job j = {x, dtype, M, K, ldx, q, ldq, NULL, 0, s, lds};
    run_threads(quant_1x128_rows, &j, M);
}

/* 128x1 tiles of token blocks tb = t, t + nt, ... (all channels). */
static void quant_128x1_blocks(void *p, int t, int nt)
{
    const struct quant_job *j = (const struct quant_job *)p;
    for (int64_t tb = t; tb < j->rows / 128; tb += nt) {
        for (int64_t c = 0; c < j->cols; ++c) {
            float amax = 0.0f, sc, r;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(load_elem(j->x, j->dtype, j->ldx, tb * 128 + i, c));
                if (a > amax)
                    amax = a;
            }
            tile_scale(amax, &sc, &r);
            for (int i = 0; i < 128; ++i)
                j->qT[c * j->ldqT + tb * 128 + i] =
                    quantize_value(load_elem(j->x, j->dtype, j->ldx, tb * 128 + i, c), r);
            j->s[tb * j->lds + c] = sc;
        }
    }
}

/* 128x1 tiles (128 tokens of one channel): x [T x C] row-major.
 * Codes are written transposed: qT [C x T] with qT[c*ldq + t];
 * s [T/128][lds] with s[tb*lds + c]. */
void fp8bs_oracle_quant_act_128x1(const void *x, int dtype, int64_t T, int64_t C, int64_t ldx,
                                  uint8_t *qT, int64_t ldq, float *s, int64_t lds)
{
    struct quant_job j = {x, dtype, T, C, ldx, NULL, 0, qT, ldq, s, lds};
    run_threads(quant_128x1_blocks, &j, T / 128);
}

/* 128x128 blocks of block rows rb = t, t + nt, ... */
static void quant_128x128_blockrows(void *p, int t, int nt)
{
    const struct quant_job *j = (const struct quant_job *)p;
    const int64_t C = j->cols;
    for (int64_t rb = t; rb < j->rows / 128; rb += nt) {
        for (int64_t cb = 0; cb < C / 128; ++cb) {
            float amax = 0.0f, sc, r;
            for (int i = 0; i < 128; ++i)
                for (int k = 0; k < 128; ++k) {
                    float a = fabsf(load_elem(j->x, j->dtype, j->ldx, rb * 128 + i, cb * 128 + k));
                    if (a > amax)
                        amax = a;
                }
            tile_scale(amax, &sc, &r);
            for (int i = 0; i < 128; ++i)
                for (int k = 0; k < 128; ++k) {
                    int64_t row = rb * 128 + i, col = cb * 128 + k;
                    uint8_t code = quantize_value(load_elem(j->x, j->dtype, j->ldx, row, col), r);
                    j->q[row * j->ldq + col] = code;
                    if (j->qT)
                        j->qT[col * j->ldqT + row] = code;
                }
            j->s[rb * (C / 128) + cb] = sc;
        }
    }
}

/* 128x128 weight blocks: w [R x C] row-major.  q [R x C] (ldq); optional
 * qT [C x R] (ldqT) holding the same codes transposed; s [R/128][C/128]. */
void fp8bs_oracle_quant_w_128x128(const void *w, int dtype, int64_t R, int64_t C, int64_t ldw,
                                  uint8_t *q, int64_t ldq, uint8_t *qT, int64_t ldqT, float *s)
{
    struct quant_job j = {w, dtype, R, C, ldw, q, ldq, qT, ldqT, s, 0};
    run_threads(quant_128x128_blockrows, &j, R / 128);
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

struct gemm_job {
    int64_t M, N, K;
    const uint8_t *A;
    int64_t lda;
    const float *sa;
    int64_t ldsa;
    const uint8_t *B;
    int64_t ldb;
    const float *sb;
    int mode;
    int64_t ldsb;
    const int64_t *rows, *cols;    /* element lists (NULL: whole rows) */
    double *c_ref, *s_abs;
    double dec[256];
};

/* Rows t, t + nt, ... of the full output. */
static void gemm_rows(void *p, int t, int nt)
{
    const struct gemm_job *g = (const struct gemm_job *)p;
    for (int64_t i = t; i < g->M; i += nt)
        for (int64_t j = 0; j < g->N; ++j)
            gemm_one(g->K, g->A, g->lda, g->sa, g->ldsa, g->B, g->ldb, g->sb, g->mode, g->ldsb,
                     g->dec, i, j, &g->c_ref[i * g->N + j], &g->s_abs[i * g->N + j]);
}

/* Elements t, t + nt, ... of the list. */
static void gemm_list(void *p, int t, int nt)
{
    const struct gemm_job *g = (const struct gemm_job *)p;
    for (int64_t e = t; e < g->M; e += nt)
        gemm_one(g->K, g->A, g->lda, g->sa, g->ldsa, g->B, g->ldb, g->sb, g->mode, g->ldsb,
                 g->dec, g->rows[e], g->cols[e], &g->c_ref[e], &g->s_abs[e]);
}

/* Full M x N output into c_ref / s_abs (row-major, N per row). */
void fp8bs_oracle_gemm(int64_t M, int64_t N, int64_t K,
                       const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                       const uint8_t *B, int64_t ldb, const float *sb, int mode, int64_t ldsb,
                       double *c_ref, double *s_abs)
{
    struct gemm_job g = {M, N, K, A, lda, sa, ldsa, B, ldb, sb, mode, ldsb,
                         NULL, NULL, c_ref, s_abs, {0}};
    decode_table(g.dec);
    run_threads(gemm_rows, &g, M);
}

/* Selected output elements (rows[e], cols[e]) for e < count. */
void fp8bs_oracle_gemm_elements(int64_t K,
                                const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                                const uint8_t *B, int64_t ldb, const float *sb, int mode, int64_t ldsb,
                                int64_t count, const int64_t *rows, const int64_t *cols,
                                double *c_ref, double *s_abs)
{
    struct gemm_job g = {count, 0, K, A, lda, sa, ldsa, B, ldb, sb, mode, ldsb,
                         rows, cols, c_ref, s_abs, {0}};
    decode_table(g.dec);
    run_threads(gemm_list, &g, count);
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

/* MX groups of rows r = t, t + nt, ... (one whole row per thread step). */
struct mx_quant_job {
    const void *x;
    int dtype;
    int64_t R, K, ldx;
    uint8_t *q;
    int64_t ldq;
    uint8_t *sf;
    int64_t ldsf;
};

static void mx_quant_rows(void *p, int t, int nt)
{
    const struct mx_quant_job *j = (const struct mx_quant_job *)p;
    for (int64_t r = t; r < j->R; r += nt) {
        for (int64_t g = 0; g < j->K / 32; ++g) {
            float amax = 0.0f, mult;
            int e;
            for (int c = 0; c < 32; ++c) {
                float a = fabsf(load_elem(j->x, j->dtype, j->ldx, r, g * 32 + c));
                if (a > amax)
                    amax = a;
            }
            e = mx_group_exponent(amax);
            mult = ldexpf(1.0f, -e);       /* exact: 2^-127 .. 2^127 are binary32 values */
            for (int c = 0; c < 32; ++c) {
                volatile float y = load_elem(j->x, j->dtype, j->ldx, r, g * 32 + c) * mult;
                j->q[r * j->ldq + g * 32 + c] = fp8bs_oracle_e4m3_encode(y);
            }
            j->sf[((g / 4) * j->ldsf + r) * 4 + g % 4] = (uint8_t)(e + 127);
        }
    }
}

/* x [R x K] row-major (ldx elements) -> q [R x K] (ldq bytes per row) and the
 * exponent bytes sf as described above.  K % 128 == 0. */
void fp8bs_oracle_mx_quant_1x32(const void *x, int dtype, int64_t R, int64_t K, int64_t ldx,
                                uint8_t *q, int64_t ldq, uint8_t *sf, int64_t ldsf)
{
    struct mx_quant_job j = {x, dtype, R, K, ldx, q, ldq, sf, ldsf};
    run_threads(mx_quant_rows, &j, R);
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

struct mx_job {
    int64_t M, N, K;
    const uint8_t *A;
    int64_t lda;
    const uint8_t *sfa;
    int64_t ldsfa;
    const uint8_t *B;
    int64_t ldb;
    const uint8_t *sfb;
    int64_t ldsfb;
    const int64_t *rows, *cols;    /* element lists (NULL: whole rows) */
    double *c_ref, *s_abs;
    double dec[256];
};

static void mx_rows(void *p, int t, int nt)
{
    const struct mx_job *g = (const struct mx_job *)p;
    for (int64_t i = t; i < g->M; i += nt)
        for (int64_t j = 0; j < g->N; ++j)
            mx_gemm_one(g->K, g->A, g->lda, g->sfa, g->ldsfa, g->B, g->ldb, g->sfb, g->ldsfb,
                        g->dec, i, j, &g->c_ref[i * g->N + j], &g->s_abs[i * g->N + j]);
}

static void mx_list(void *p, int t, int nt)
{
    const struct mx_job *g = (const struct mx_job *)p;
    for (int64_t e = t; e < g->M; e += nt)
        mx_gemm_one(g->K, g->A, g->lda, g->sfa, g->ldsfa, g->B, g->ldb, g->sfb, g->ldsfb,
                    g->dec, g->rows[e], g->cols[e], &g->c_ref[e], &g->s_abs[e]);
}

void fp8bs_oracle_mx_gemm(int64_t M, int64_t N, int64_t K,
                          const uint8_t *A, int64_t lda, const uint8_t *sfa, int64_t ldsfa,
                          const uint8_t *B, int64_t ldb, const uint8_t *sfb, int64_t ldsfb,
                          double *c_ref, double *s_abs)
{
    struct mx_job g = {M, N, K, A, lda, sfa, ldsfa, B, ldb, sfb, ldsfb, NULL, NULL,
                       c_ref, s_abs, {0}};
    decode_table(g.dec);
    run_threads(mx_rows, &g, M);
}

void fp8bs_oracle_mx_gemm_elements(int64_t K,
                                   const uint8_t *A, int64_t lda, const uint8_t *sfa, int64_t ldsfa,
                                   const uint8_t *B, int64_t ldb, const uint8_t *sfb, int64_t ldsfb,
                                   int64_t count, const int64_t *rows, const int64_t *cols,
                                   double *c_ref, double *s_abs)
{
    struct mx_job g = {count, 0, K, A, lda, sfa, ldsfa, B, ldb, sfb, ldsfb, rows, cols,
                       c_ref, s_abs, {0}};
    decode_table(g.dec);
    run_threads(mx_list, &g, count);
}

/* ------------------------------------------------ quantize-then-dispatch
 *
 * Source: untitled page at jp-study.kr, MoE passage: the activations entering
 * the MoE up-projection are quantized to FP8 before they are dispatched to
 * the experts.
 *
 * Readings taken where the pages are silent:
 *  - Tokens are grouped by expert; inside an expert they keep increasing
 *    token order (a stable grouping, so the row of every token is unique).
 *  - Every expert's row count is padded up to a multiple of 128 (the 1x128
 *    tiles of the grouped GEMM never straddle two experts); a padding row is
 *    a quantized zero row: codes 0, scale 1, and no token.
 *  - A token whose expert id lies outside [0, E) is dropped (no row).
 *
 * Steps, in order:
 *  1. counts[e] = number of tokens routed to expert e;
 *  2. offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e] rounded up to 128;
 *  3. walking the tokens in increasing order, the next free row of the
 *     token's expert (starting at offsets[e]) becomes token_row[t], and
 *     row_token[row] = t;
 *  4. rows offsets[e] + counts[e] .. offsets[e+1] - 1 get row_token -1;
 *  5. each routed row holds the 1x128 quantization of its token's row of x;
 *     each padding row holds codes 0 and scale 1.
 * x [T x K] (ldx elements); q [M_cap x K] (ldq bytes); s[kb*lds + row];
 * row_token has M_cap entries; rows at or past offsets[E] are not written.
 * Returns the number of dropped tokens, or -1 if M_cap is too small. */
int64_t fp8bs_oracle_dispatch(const void *x, int dtype, int64_t T, int64_t K, int64_t ldx,
                              const int32_t *expert, int32_t E, int64_t M_cap,
                              uint8_t *q, int64_t ldq, float *s, int64_t lds,
                              int64_t *offsets, int64_t *counts, int64_t *token_row,
                              int64_t *row_token)
{
    int64_t dropped = 0, *next;
    const uint16_t *xb = (const uint16_t *)x;
    const float *xf = (const float *)x;

    for (int32_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t t = 0; t < T; ++t)                                    /* step 1 */
        if (expert[t] >= 0 && expert[t] < E)
            counts[expert[t]] += 1;
    offsets[0] = 0;                                                    /* step 2 */
    for (int32_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + (counts[e] + 127) / 128 * 128;
    if (offsets[E] > M_cap)
        return -1;

    next = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
    if (next == NULL)
        return -1;
    for (int32_t e = 0; e < E; ++e)
        next[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t) {                                  /* step 3 */
        int32_t e = expert[t];
        if (e < 0 || e >= E) {
            token_row[t] = -1;
            dropped += 1;
            continue;
        }
        token_row[t] = next[e];
        row_token[next[e]] = t;
        next[e] += 1;
    }
    for (int32_t e = 0; e < E; ++e)                                    /* step 4 */
        for (int64_t r = offsets[e] + counts[e]; r < offsets[e + 1]; ++r)
            row_token[r] = -1;
    free(next);

    for (int64_t r = 0; r < offsets[E]; ++r) {                         /* step 5 */
        if (row_token[r] < 0) {
            memset(q + r * ldq, 0, (size_t)K);
            for (int64_t kb = 0; kb < K / 128; ++kb)
                s[kb * lds + r] = 1.0f;
            continue;
        }
        /* the one-row 1x128 quantizer applied to row row_token[r] of x */
        if (dtype == ORACLE_F32)
            fp8bs_oracle_quant_act_1x128(xf + row_token[r] * ldx, dtype, 1, K, ldx,
                                         q + r * ldq, ldq, s + r, lds);
        else
            fp8bs_oracle_quant_act_1x128(xb + row_token[r] * ldx, dtype, 1, K, ldx,
                                         q + r * ldq, ldq, s + r, lds);
    }
    return dropped;
}
