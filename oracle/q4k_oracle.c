/*
 * q4_K x int8 MMQ -- CPU ORACLE.  TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded restatement of what the q4_K x int8 GEMM
 * computes, used to check the CUDA library. The library never calls, links or
 * includes this file; only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or
 * constant with the CUDA path. Built into the same shared object as the q6_K
 * oracle (q6k_oracle.c), whose activation quantiser it uses unchanged.
 *
 * Sources (pages of the minfer CUDA optimisation log):
 *   [r18]  "r18: Load-time B pre-expansion -- staging becomes a bulk copy",
 *          Sec. 1: a q4_K super-block is 144 bytes, a 16-byte header and 128
 *          bytes of packed nibbles, 256 elements in 8 sub-blocks of 32.
 *          Sec. 3.2 (the in-loop B expansion it replaces): for nibble pair p
 *          (0..3) the 32 bytes at 16 + 32 p hold sub-block 2 p in their low
 *          nibbles and sub-block 2 p + 1 in their high nibbles, in element
 *          order (raw values 0..15, not centred); the per-chunk scale parse
 *          reads d (f16) at byte 0, dmin (f16) at byte 2 and the packed
 *          6-bit scale / min of chunk c & 7 from the 12 bytes at byte 4, and
 *          forms the pair (d * sc, -(dmin * m)).
 *   [r38]  "r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2: q4_K's
 *          rescale has two terms, d and dmin both multiply the accumulator,
 *          with the activation side's per-32 scale and block sum.
 *
 * Reading taken where the pages are silent: the 12-byte packing of the eight
 * 6-bit scales and eight 6-bit mins (the pages call the helper that unpacks it
 * but do not print it) is the GGUF q4_K layout:
 *   sub-blocks j = 0..3: scale = low 6 bits of byte j,
 *                        min   = low 6 bits of byte j + 4;
 *   sub-blocks j = 4..7: scale = low nibble of byte j + 4, with the top two
 *                        bits of byte j - 4 as its bits 4 and 5;
 *                        min   = high nibble of byte j + 4, with the top two
 *                        bits of byte j as its bits 4 and 5.
 * Every bit of the 12 bytes feeds exactly one of the 16 six-bit values.
 *
 * The operation, in double: for token n and weight row m,
 *   Y[n][m] = sum over super-blocks b and sub-blocks c of
 *             da[n][8b + c] * ( d[m][b] * sc[m][b][c] * P[n][m][b][c]
 *                               - dmin[m][b] * mn[m][b][c] * S[n][b][c] ),
 *   P = sum over the 32 elements of q * xq (q the raw nibble 0..15),
 *   S = sum over the 32 elements of xq,
 * i.e. the dequantised weight d*sc*q - dmin*m times the dequantised
 * activation da*xq, summed over k.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

#define Q4_QK 256      /* elements per super-block                [r18 1]   */
#define Q4_BLK 144     /* bytes per super-block                   [r18 1]   */
#define Q4_OFF_DMIN 2  /* f16 dmin                                [r18 3.2] */
#define Q4_OFF_SC 4    /* 12 bytes of packed 6-bit scales / mins  [r18 3.2] */
#define Q4_OFF_QS 16   /* 128 bytes of nibbles                    [r18 3.2] */

double orc_f16_to_f64(uint16_t h); /* q6k_oracle.c */

/* The 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes s
 * (the reading in the header). */
void orc_q4k_scale_min(const uint8_t *s, int j, int *sc, int *mn)
{
    if (j < 4) {
        *sc = s[j] & 63;
#if ORC_MUTANT == 15
        *mn = s[j] & 63;                                   /* planted: min read from the scale byte */
#else
        *mn = s[j + 4] & 63;
#endif
    } else {
#if ORC_MUTANT == 16
        *sc = (s[j + 4] & 15) | ((s[j] >> 6) << 4);       /* planted: top bits from the min bytes */
#else
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
#endif
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* The raw nibble (0..15) of element e (0..255) of one super-block [r18 3.2]:
 * sub-block c = e / 32, nibble pair p = c / 2, byte 16 + 32 p + e % 32, low
 * nibble for even c, high nibble for odd c. */
static int orc_q4k_code(const uint8_t *blk, int e)
{
    const int c = e >> 5, t = e & 31;
    const uint8_t b = blk[Q4_OFF_QS + 32 * (c >> 1) + t];
#if ORC_MUTANT == 17
    return (c & 1) ? (b & 15) : (b >> 4);                  /* planted: nibbles swapped */
#else
    return (c & 1) ? (b >> 4) : (b & 15);
#endif
}

/* Decode one raw super-block: the 256 nibbles, the 8 scales and 8 mins, and
 * the two f16 factors as doubles. */
void orc_q4k_decode_block(const uint8_t *blk, uint8_t *codes, int *sc, int *mn, double *d,
                          double *dmin)
{
    for (int e = 0; e < Q4_QK; ++e)
        codes[e] = (uint8_t)orc_q4k_code(blk, e);
    for (int j = 0; j < 8; ++j)
        orc_q4k_scale_min(blk + Q4_OFF_SC, j, &sc[j], &mn[j]);
    *d = orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    *dmin = orc_f16_to_f64((uint16_t)(blk[Q4_OFF_DMIN] | (blk[Q4_OFF_DMIN + 1] << 8)));
}

/* The GEMM (see the header). raw is [M][K/256] raw super-blocks; xq [N][K];
 * da [N][K/32]. Y is [N][M] double; P (nullable) is [N][M][K/32] int32, the
 * exact per-sub-block sums of q * xq. */
void orc_q4k_mmq(const uint8_t *raw, int M, int K, const int8_t *xq, const float *da, int N,
                 double *Y, int32_t *P)
{
    const int nsb = K / Q4_QK, nc = K / 32;
    uint8_t *q = (uint8_t *)malloc((size_t)K);
    int *sc = (int *)malloc(sizeof(int) * (size_t)nc);
    int *mn = (int *)malloc(sizeof(int) * (size_t)nc);
    double *d = (double *)malloc(sizeof(double) * (size_t)nsb);
    double *dmin = (double *)malloc(sizeof(double) * (size_t)nsb);
    if (!q || !sc || !mn || !d || !dmin)
        goto out;
    for (int m = 0; m < M; ++m) {
        const uint8_t *row = raw + (size_t)m * nsb * Q4_BLK;
        for (int b = 0; b < nsb; ++b)
            orc_q4k_decode_block(row + (size_t)b * Q4_BLK, q + (size_t)b * Q4_QK, sc + 8 * b,
                                 mn + 8 * b, &d[b], &dmin[b]);
        for (int n = 0; n < N; ++n) {
            const int8_t *x = xq + (size_t)n * K;
            double y = 0.0;
            for (int c = 0; c < nc; ++c) {
                int32_t p = 0, s = 0;
                for (int t = 0; t < 32; ++t) {
                    p += (int32_t)q[32 * c + t] * (int32_t)x[32 * c + t];
                    s += (int32_t)x[32 * c + t];
                }
                if (P)
                    P[((size_t)n * M + m) * nc + c] = p;
                const int b = c / 8;
#if ORC_MUTANT == 19
                const double a = (double)da[(size_t)n * nc + (c ^ 1)];   /* planted: neighbour's da */
#else
                const double a = (double)da[(size_t)n * nc + c];
#endif
#if ORC_MUTANT == 18
                y += a * (d[b] * sc[c] * (double)p + dmin[b] * mn[c] * (double)s);  /* planted: min term added */
#else
                y += a * (d[b] * sc[c] * (double)p - dmin[b] * mn[c] * (double)s);
#endif
            }
            Y[(size_t)n * M + m] = y;
        }
    }
out:
    free(q);
    free(sc);
    free(mn);
    free(d);
    free(dmin);
}
