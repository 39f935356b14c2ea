/*
 * q6_K x int8 MMQ -- CPU ORACLE.  TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded restatement of what the q6_K x int8 prefill
 * GEMM computes, used to check the CUDA library. The library never calls,
 * links or includes this file; only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Sources (pages of the minfer CUDA optimisation log on the q6_K GEMM):
 *   [r38]  "r38 -- q6_K BT-style raw-byte mma kernel"
 *          Sec. 2.1: the 210-byte super-block (ql[128], qh[64], int8 scales[16],
 *          f16 d), 16 sub-blocks of 16, dequantised value d*sc[sub]*(q-32).
 *          Sec. 2.2: single-term rescale sum += da*dsc with dsc = d*sc[sub] and
 *          no dmin term; da is the activation's per-32 quantisation scale.
 *          Sec. 3.2: the element -> (ql byte, nibble), (qh byte, 2-bit field)
 *          index map, and dsc0/dsc1 = d * (float)(int8)sc.
 *   [r41]  "r41 -- q6_K B-expand widened to uint4 group loads", Sec. 2: the
 *          in-block byte-offset table (ql 0..127, qh 128..191, sc 192..207,
 *          d 208..209).
 *   [r53]  "r53 -- q6_K bundle: W_exp pre-expansion plane + cp.async B
 *          staging", Sec. 2.3: W_exp is the dense centered-int8 plane, one byte
 *          per element, row stride K, super-block stride 256.
 *   [r42]  "r42 -- q6_K stage-wide dsc scale reads", Sec. 3.2: dsc = d*sc per
 *          (row, 16-sub-block), in f32.
 *
 * Readings taken where the pages are silent:
 *   - activation quantiser: per token and per 32-block, amax = max|x|,
 *     da = amax/127 in f32, q = clamp(round-half-away(x/da), -127, 127) with
 *     an IEEE f32 division; amax == 0 gives da = 0 and q = 0. The pages fix no
 *     precision for this integer decision, so it is taken in f32, the kernel's
 *     precision.
 *   - d is decoded exactly, subnormals included (IEEE 754 binary16).
 *   - Y is token-major, Y[n][m]; the sum is formed in double.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fexcess-precision=standard -fPIC
 *        -shared.  ORC_MUTANT=<k> plants one deliberate mistake (used only by
 *        the test that shows the pins catch it); the default build has none.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if FLT_EVAL_METHOD != 0
#error "the oracle needs float arithmetic evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

#define QK 256          /* elements per super-block            [r38 2.1] */
#define BLK 210         /* bytes per super-block               [r38 2.1] */
#define OFF_QH 128      /* qh[64] starts here                  [r41 2]   */
#define OFF_SC 192      /* int8 scales[16] start here          [r41 2]   */
#define OFF_D 208       /* f16 super-block scale d             [r41 2]   */

int orc_mutant(void) { return ORC_MUTANT; }

/* IEEE 754 binary16 -> double, exact. Sign bit, 5-bit biased exponent (bias
 * 15), 10-bit fraction; exponent 0 is the subnormal range f * 2^-24. */
double orc_f16_to_f64(uint16_t h)
{
    const int sign = h >> 15;
    const int e = (h >> 10) & 0x1F;
    const int f = h & 0x3FF;
    double v;
    if (e == 0) {
#if ORC_MUTANT == 12
        v = 0.0;                                 /* planted: subnormals flushed */
#else
        v = ldexp((double)f, -24);
#endif
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
#if ORC_MUTANT == 13
        v = ldexp((double)(1024 + f), e - 24);   /* planted: bias off by one */
#else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
#endif
    }
    return sign ? -v : v;
}

/* The 6-bit code (0..63) of element e (0..255) of one super-block [r38 3.2].
 * The block is two halves of 128 elements. Inside a half, position r:
 *   low 4 bits  <- ql byte (64*half + r mod 64): low nibble for r < 64,
 *                  high nibble for r >= 64;
 *   high 2 bits <- qh byte (32*half + r mod 32): the 2-bit field number
 *                  floor(r/32), i.e. bits 2*floor(r/32) .. +1.
 * So a ql byte serves elements r and r+64, a qh byte serves r, r+32, r+64,
 * r+96 of the same half. */
static int orc_code(const uint8_t *blk, int e)
{
#if ORC_MUTANT == 14
    /* planted: the sequential map (ql[e/2] nibble e%2, qh[e/4] field e%4) */
    return ((blk[e >> 1] >> (4 * (e & 1))) & 0x0F)
         | (((blk[OFF_QH + (e >> 2)] >> (2 * (e & 3))) & 0x3) << 4);
#else
    const int half = e >> 7;
    const int r = e & 127;
#if ORC_MUTANT == 1
    const uint8_t lo_byte = blk[64 * half + (r & 31)];      /* planted: wrong ql index */
#else
    const uint8_t lo_byte = blk[64 * half + (r & 63)];
#endif
#if ORC_MUTANT == 3
    const int lo = (r < 64) ? (lo_byte >> 4) : (lo_byte & 0x0F);  /* planted: nibbles swapped */
#else
    const int lo = (r < 64) ? (lo_byte & 0x0F) : (lo_byte >> 4);
#endif
#if ORC_MUTANT == 2
    const uint8_t hi_byte = blk[OFF_QH + 32 * half + (r >> 2)];   /* planted: wrong qh index */
#else
    const uint8_t hi_byte = blk[OFF_QH + 32 * half + (r & 31)];
#endif
    const int hi = (hi_byte >> (2 * (r >> 5))) & 0x3;
    return lo | (hi << 4);
#endif
}

/* Centered value q - 32 in [-32, 31] of element e [r38 2.1]. */
static int orc_value(const uint8_t *blk, int e)
{
#if ORC_MUTANT == 4
    return orc_code(blk, e);                     /* planted: centering dropped */
#else
    return orc_code(blk, e) - 32;
#endif
}

/* Decode one raw super-block into its 256 centered values. */
void orc_q6k_decode_block(const uint8_t *blk, int8_t *out)
{
    for (int e = 0; e < QK; ++e)
        out[e] = (int8_t)orc_value(blk, e);
}

/* W_exp [r53 2.3]: centered int8, [M][K], row stride K, super-block stride 256. */
void orc_q6k_wexp(const uint8_t *raw, int M, int K, int8_t *wexp)
{
    const int nsb = K / QK;
    for (int m = 0; m < M; ++m)
        for (int sb = 0; sb < nsb; ++sb)
            orc_q6k_decode_block(raw + ((size_t)m * nsb + sb) * BLK,
                                 wexp + (size_t)m * K + (size_t)sb * QK);
}

/* dsc[m][s] = f32(d) * sc[s] for every 16-element sub-block s of row m
 * [r42 3.2, r38 3.2]; exact in f32 (11-bit by 8-bit significands). */
void orc_q6k_dsc(const uint8_t *raw, int M, int K, float *dsc)
{
    const int nsb = K / QK;
    for (int m = 0; m < M; ++m)
        for (int sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = raw + ((size_t)m * nsb + sb) * BLK;
            const uint16_t dh = (uint16_t)(blk[OFF_D] | (blk[OFF_D + 1] << 8));
            const float d = (float)orc_f16_to_f64(dh);
            for (int s = 0; s < 16; ++s)
                dsc[(size_t)m * (K / 16) + sb * 16 + s] = d * (float)(int8_t)blk[OFF_SC + s];
        }
}

/* Activation quantiser (per token n, per 32-element block c of K):
 *   amax = max |x|;  da = amax / 127 (f32);  q = clamp(round(x / da), -127, 127),
 * rounding half away from zero; amax == 0 gives da = 0, q = 0.
 * The pages name the packed per-token scale of the activation prepass [r38 2.2]
 * but print no quantiser; this is the reading listed in the header.
 * X is [N][ldx] f32; xq is [N][K] int8; da is [N][K/32] f32. */
void orc_q8_quantize(const float *X, int N, int K, int ldx, int8_t *xq, float *da)
{
    const int nc = K / 32;
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < nc; ++c) {
            const float *x = X + (size_t)n * ldx + 32 * c;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                const float a = fabsf(x[i]);
                if (a > amax)
                    amax = a;
            }
#if ORC_MUTANT == 10
            const float d = amax / 128.0f;             /* planted: wrong divisor */
#else
            const float d = amax / 127.0f;
#endif
            da[(size_t)n * nc + c] = d;
            for (int i = 0; i < 32; ++i) {
                int q = 0;
                if (d != 0.0f) {
                    const float t = x[i] / d;
#if ORC_MUTANT == 11
                    q = (int)truncf(t);                  /* planted: truncation */
#else
                    q = (int)roundf(t);
#endif
                    if (q > 127) q = 127;
                    if (q < -127) q = -127;
                }
                xq[(size_t)n * K + 32 * c + i] = (int8_t)q;
            }
        }
}

/* The GEMM [r38 2.1, 2.2]: for every token n and weight row m,
 *   Y[n][m] = sum over super-blocks sb and sub-blocks s of
 *             d[m][sb] * sc[m][sb][s] * da[n][c(sb,s)] * P[n][m][sb][s],
 *   P[n][m][sb][s] = sum_{t<16} (q[m][256 sb + 16 s + t] - 32) * xq[n][256 sb + 16 s + t],
 * where c(sb,s) = (256 sb + 16 s) / 32 is the 32-element activation block
 * holding the sub-block. P is an exact int32; the scaling is in double.
 * raw is [M][K/256] raw super-blocks; xq [N][K]; da [N][K/32].
 * Y is [N][M] double; P (nullable) is [N][M][K/16] int32. */
void orc_mmq(const uint8_t *raw, int M, int K, const int8_t *xq, const float *da,
             int N, double *Y, int32_t *P)
{
    const int nsb = K / QK, nsub = K / 16, nc = K / 32;
    int8_t *w = (int8_t *)malloc((size_t)K);
    if (!w)
        return;
    for (int m = 0; m < M; ++m) {
        const uint8_t *row = raw + (size_t)m * nsb * BLK;
        for (int sb = 0; sb < nsb; ++sb)
            orc_q6k_decode_block(row + (size_t)sb * BLK, w + (size_t)sb * QK);
        for (int n = 0; n < N; ++n) {
            const int8_t *x = xq + (size_t)n * K;
            double y = 0.0;
            for (int sb = 0; sb < nsb; ++sb) {
                const uint8_t *blk = row + (size_t)sb * BLK;
                const uint16_t dh = (uint16_t)(blk[OFF_D] | (blk[OFF_D + 1] << 8));
#if ORC_MUTANT == 7
                const double d = 1.0;                     /* planted: d dropped */
#else
                const double d = orc_f16_to_f64(dh);
#endif
                for (int s = 0; s < 16; ++s) {
                    const int k0 = sb * QK + 16 * s;
                    int32_t p = 0;
                    for (int t = 0; t < 16; ++t)
                        p += (int32_t)w[k0 + t] * (int32_t)x[k0 + t];
                    if (P)
                        P[((size_t)n * M + m) * nsub + (size_t)sb * 16 + s] = p;
#if ORC_MUTANT == 5
                    const double sc = (double)(int8_t)blk[OFF_SC + (s ^ 1)];   /* planted: neighbour's scale */
#else
                    const double sc = (double)(int8_t)blk[OFF_SC + s];
#endif
#if ORC_MUTANT == 6
                    const int c = k0 / 16 % nc;              /* planted: sub-block used as block */
#else
                    const int c = k0 / 32;
#endif
#if ORC_MUTANT == 9
                    const double a = (double)da[((size_t)c * N + n) % ((size_t)N * nc)];  /* planted: da read as [K/32][N] */
#else
                    const double a = (double)da[(size_t)n * nc + c];
#endif
#if ORC_MUTANT == 8
                    y += (s & 1 ? -1.0 : 1.0) * d * sc * a * (double)p;   /* planted: sign flip */
#else
                    y += d * sc * a * (double)p;
#endif
                }
            }
            Y[(size_t)n * M + m] = y;
        }
    }
    free(w);
}
