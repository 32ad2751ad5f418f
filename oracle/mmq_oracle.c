/*
 * mmq_oracle.c -- plain, slow, obviously-correct CPU oracle for block-quantized int8 MMQ.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library.  The CUDA library never links, includes or calls it, and it
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Sources (cited by page title and section):
 *   [R1]  "08 · R1 — int8 MMQ prefill GEMM (opt-in): the parity-first strategy" (minfer CUDA notes)
 *         §2.1 "The int8 tensor-core mma (s8s8s32)", §2.2 "The q8_1-style activation pipeline",
 *         §3.2 "Key code" (the CPU reference frame of the parity test).
 *   [NR]  "When the Product Won't Collapse: A Negative Result on int8 Tensor-Core MMQ",
 *         §2 "The obstruction: an opaque accumulator" (the blockwise contraction display equation).
 *   [IQ]  "CUDA: add IQ1_M to MMQ" (llama.cpp pull request #304), PR description and "Design".
 *   [W8]  "INT8 W8A8 GEMM — Prefill (M > 32) — gfx928 / SGLang TP4 + TP8", §1 "M = 3072 prefill"
 *         and §2 (int32 accumulation, scale epilogue, bf16 output, mismatch 0 / max_abs_error 0.0).
 *   [R1] §2.2 also fixes q6_K's arithmetic: a 6-bit grid 0..63 moved to the signed domain by
 *         subtracting 32, scales on 16-element sub-blocks, so each 32-k chunk carries two integer dots
 *         multiplied by (d*sc0, d*sc1) ("The K-quant signed domain"; "The q6_K per-16 loop").
 *
 * Mutation switches (MUT_*): each plants one plausible mistake.  They are never defined in a normal
 * build; the pin suite's self-test compiles each mutant and checks that some pin fails on it.
 *
 * Everything is scalar loops.  Integer dots are int32/int64; floating point is IEEE f32 in exactly the
 * order written (build with -ffp-contract=off, no fast-math), because the pages fix f32 as the
 * precision of the scale arithmetic ([R1] §3.2 reference; the activation scale is an f32 value).
 *
 * Byte layouts are this library's documented layouts (the pages give block sizes, not bit layouts):
 *   q8_1 activations : q int8 [M][K]; d f32 [M][K/32]; s f32 [M][K/32]       (separate arrays here)
 *   Q8_0  (34 B/32)  : f16 d | int8 q[32]
 *   Q4_0  (18 B/32)  : f16 d | 16 B, byte i = element i (low nibble) | element i+16 (high nibble)
 *   Q4_K  (144 B/256): f16 d | f16 dmin | 12 B = 16 six-bit fields, little-endian bit stream,
 *                      sc[0..7] then m[0..7] | 128 B nibbles, byte 32j+i = element 64j+i (low) |
 *                      element 64j+32+i (high)
 *   IQ1_M (76 B/256) : 64 B two-bit codes (element i at bits 2(i%4) of byte i/4; code 0,1,2 -> g=-1,0,+1)
 *                      | 4 B sign bits (bit j of the little-endian word: elements 8j..8j+7, 0 -> +1/8,
 *                      1 -> -1/8) | 6 B = 16 three-bit sub-scales s, little-endian bit stream (s_h for
 *                      elements 16h..16h+15) | f16 d
 *   W8A8             : int8 W [N][K] with f32 ws [N]; int8 X [M][K] with f32 xs [M]
 *   Q6_K (224 B/256) : int8 sc[16] (sc_h for elements 16h..16h+15) | f16 d | 14 B zero | four 48 B
 *                      stage records j = 0..3: 32 B low nibbles, byte i = element 64j+i (low) |
 *                      element 64j+32+i (high), then 16 B high pairs, byte i = bits 4-5 of elements
 *                      64j+i (bits 0-1), 64j+16+i (bits 2-3), 64j+32+i (bits 4-5), 64j+48+i (bits 6-7)
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_Q8_0 = 0, OR_Q4_0 = 1, OR_Q4_K = 2, OR_IQ1_M = 3, OR_W8A8 = 4, OR_Q6_K = 5 };

/* Block types of the blockwise product (W8A8 has its own entry point). */
static int block_type(int wtype) { return (wtype >= 0 && wtype <= 3) || wtype == OR_Q6_K; }

/* ---------------------------------------------------------------- scalar helpers */

/* IEEE binary16 -> binary32, exact (textbook decode of sign / 5-bit exponent / 10-bit fraction). */
static float half_to_float(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t ex = (uint32_t)(h >> 10) & 31u;
    uint32_t fr = (uint32_t)h & 1023u;
    float mag;
    if (ex == 0) {
        mag = (float)fr * (1.0f / 16777216.0f);            /* subnormal: fr * 2^-24, exact */
    } else if (ex == 31) {
        mag = fr ? NAN : INFINITY;
    } else {
#ifdef MUT_F16_BIAS
        uint32_t bits = ((ex - 14u + 127u) << 23) | (fr << 13);
#else
        uint32_t bits = ((ex - 15u + 127u) << 23) | (fr << 13);
#endif
        memcpy(&mag, &bits, 4);
    }
    return sign ? -mag : mag;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | ((uint16_t)p[1] << 8)); }

/* Read bit field [pos, pos+width) of a little-endian bit stream. */
static unsigned bits_le(const uint8_t* p, unsigned pos, unsigned width) {
    unsigned v = 0;
    for (unsigned i = 0; i < width; i++) {
        unsigned b = pos + i;
        v |= (unsigned)((p[b >> 3] >> (b & 7)) & 1u) << i;
    }
    return v;
}

/* f32 -> bf16 bit pattern, round to nearest even (non-NaN inputs; NaN maps to a quiet NaN). */
static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
#ifdef MUT_BF16_HALF_UP
    u += 0x8000u;                                           /* ties rounded up instead of to even */
    (void)lsb;
#else
    u += 0x7FFFu + lsb;
#endif
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- q8_1 quantizer */
/*
 * [R1] §2.2 and §3.2 (reference quantizer): per 32-value block, amax = max|x|, d = amax/127,
 * q = round-half-even(x/d) clamped, block sum over the codes.  The block sum this library stores is
 * the f32 value s = d * sum(q) (the llama-style q8_1 sum).  d is kept in f32.
 * Division is the correctly rounded f32 x/d.  amax == 0 gives d = 0, q = 0, s = 0.
 */
int oracle_quantize_q8_1(const float* x, int64_t M, int64_t K, int8_t* q, float* d, float* s) {
    if (K % 32 != 0 || M < 0) return 1;
    const int64_t nb = K / 32;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t b = 0; b < nb; b++) {
            const float* xb = x + m * K + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
#ifdef MUT_SCALE_RECIP
            float db = amax * (1.0f / 127.0f);              /* d from a rounded reciprocal */
#else
            float db = amax / 127.0f;
#endif
            int32_t sum = 0;
            for (int i = 0; i < 32; i++) {
                int32_t qi = 0;
                if (db != 0.0f) {
#ifdef MUT_ROUND_AWAY
                    float r = roundf(xb[i] / db);
#else
                    float r = rintf(xb[i] / db);              /* rintf: ties to even (default mode) */
#endif
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    qi = (int32_t)r;
                }
                q[m * K + b * 32 + i] = (int8_t)qi;
                sum += qi;
            }
            d[m * nb + b] = db;
#ifdef MUT_SUM_ORDER
            {   /* s as a running f32 sum of d*q instead of d times the exact integer sum */
                float acc = 0.0f;
                for (int i = 0; i < 32; i++) acc += db * (float)q[m * K + b * 32 + i];
                s[m * nb + b] = acc;
            }
#else
            s[m * nb + b] = db * (float)sum;
#endif
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- weight decoders */
/*
 * Decode one weight row into integer values and per-group scales, the way the blockwise product
 * consumes them.  G = group size of the integer dot (32, or 16 for IQ1_M).
 *   Q8_0 : wq = q,               wsc = d                         [R1] §2.1 (Q8_0 x q8_1)
 *   Q4_0 : wq = nib - 8,         wsc = d          (w = d (q - 8))
 *   Q4_K : wq = nib (unsigned),  wsc = d*sc_b, wmin = dmin*m_b   [R1] §2.2 rank-1 min term
 *   IQ1_M: wq = 8g + (+1|-1),    wsc = d*(2s+1)/8 per 16 values  [IQ] Design (exact fold)
 *   Q6_K : wq = q - 32,          wsc = d*sc_h per 16 values      [R1] §2.2 (signed domain, sub-scales)
 *   W8A8 : wq = W, one scale per row (handled by oracle_w8a8).
 */
static int group_size(int wtype) { return (wtype == OR_IQ1_M || wtype == OR_Q6_K) ? 16 : 32; }

static void decode_row(int wtype, const uint8_t* row, int64_t K, int8_t* wq, float* wsc, float* wmin) {
    if (wtype == OR_Q8_0) {
        for (int64_t b = 0; b < K / 32; b++) {
            const uint8_t* blk = row + b * 34;
            wsc[b] = half_to_float(rd16(blk));
            for (int i = 0; i < 32; i++) wq[b * 32 + i] = (int8_t)blk[2 + i];
        }
    } else if (wtype == OR_Q4_0) {
        for (int64_t b = 0; b < K / 32; b++) {
            const uint8_t* blk = row + b * 18;
            wsc[b] = half_to_float(rd16(blk));
            for (int i = 0; i < 16; i++) {
                uint8_t by = blk[2 + i];
#if defined(MUT_NIBBLE_SWAP)
                wq[b * 32 + i] = (int8_t)((int)(by >> 4) - 8);
                wq[b * 32 + i + 16] = (int8_t)((int)(by & 15) - 8);
#elif defined(MUT_Q4_0_NO_OFFSET)
                wq[b * 32 + i] = (int8_t)(by & 15);
                wq[b * 32 + i + 16] = (int8_t)(by >> 4);
#else
                wq[b * 32 + i] = (int8_t)((int)(by & 15) - 8);
                wq[b * 32 + i + 16] = (int8_t)((int)(by >> 4) - 8);
#endif
            }
        }
    } else if (wtype == OR_Q4_K) {
        for (int64_t sb = 0; sb < K / 256; sb++) {
            const uint8_t* blk = row + sb * 144;
            float dd = half_to_float(rd16(blk));
            float dmin = half_to_float(rd16(blk + 2));
            const uint8_t* packed = blk + 4;
            const uint8_t* nib = blk + 16;
            for (int j = 0; j < 8; j++) {
#ifdef MUT_Q4K_FIELD_SWAP
                unsigned mn = bits_le(packed, 6u * (unsigned)j, 6);
                unsigned sc = bits_le(packed, 6u * (unsigned)(8 + j), 6);
#else
                unsigned sc = bits_le(packed, 6u * (unsigned)j, 6);
                unsigned mn = bits_le(packed, 6u * (unsigned)(8 + j), 6);
#endif
                wsc[sb * 8 + j] = dd * (float)sc;
                wmin[sb * 8 + j] = dmin * (float)mn;
            }
            for (int j = 0; j < 4; j++)
                for (int i = 0; i < 32; i++) {
                    uint8_t by = nib[32 * j + i];
                    wq[sb * 256 + 64 * j + i] = (int8_t)(by & 15);
                    wq[sb * 256 + 64 * j + 32 + i] = (int8_t)(by >> 4);
                }
        }
    } else if (wtype == OR_IQ1_M) {
        for (int64_t sb = 0; sb < K / 256; sb++) {
            const uint8_t* blk = row + sb * 76;
            const uint8_t* codes = blk;
            const uint8_t* signs = blk + 64;
            const uint8_t* subs = blk + 68;
            float dd = half_to_float(rd16(blk + 74));
            for (int i = 0; i < 256; i++) {
                int code = (codes[i / 4] >> (2 * (i % 4))) & 3;
                int g = code - 1;                                /* code 3 never appears */
                int neg = (signs[(i / 8) / 8] >> ((i / 8) % 8)) & 1;
#ifdef MUT_SIGN_POLARITY
                wq[sb * 256 + i] = (int8_t)(8 * g + (neg ? 1 : -1));
#else
                wq[sb * 256 + i] = (int8_t)(8 * g + (neg ? -1 : 1));
#endif
            }
            for (int h = 0; h < 16; h++) {
#ifdef MUT_IQ1_SCALE_GROUP32
                unsigned sv = bits_le(subs, 3u * (unsigned)(h & ~1), 3);
#else
                unsigned sv = bits_le(subs, 3u * (unsigned)h, 3);
#endif
                wsc[sb * 16 + h] = (dd * (float)(2u * sv + 1u)) * 0.125f;
            }
        }
    } else if (wtype == OR_Q6_K) {
        for (int64_t sb = 0; sb < K / 256; sb++) {
            const uint8_t* blk = row + sb * 224;
            float dd = half_to_float(rd16(blk + 16));
            for (int h = 0; h < 16; h++) wsc[sb * 16 + h] = dd * (float)(int8_t)blk[h];
            for (int j = 0; j < 4; j++) {
                const uint8_t* lo = blk + 32 + 48 * j;
                const uint8_t* hi = lo + 32;
                for (int e = 0; e < 64; e++) {
                    int low = e < 32 ? (lo[e] & 15) : (lo[e - 32] >> 4);
#ifdef MUT_Q6K_HIGH_PAIR
                    int high = (hi[e % 16] >> (2 * (e % 4))) & 3;
#else
                    int high = (hi[e % 16] >> (2 * (e / 16))) & 3;
#endif
                    wq[sb * 256 + 64 * j + e] = (int8_t)((low | (high << 4)) - 32);
                }
            }
        }
    }
}

static int64_t row_bytes(int wtype, int64_t K) {
    switch (wtype) {
        case OR_Q8_0: return K / 32 * 34;
        case OR_Q4_0: return K / 32 * 18;
        case OR_Q4_K: return K / 256 * 144;
        case OR_IQ1_M: return K / 256 * 76;
        case OR_Q6_K: return K / 256 * 224;
        default: return K;
    }
}

static int check_k(int wtype, int64_t K) {
    if (K <= 0) return 1;
    if ((wtype == OR_Q4_K || wtype == OR_IQ1_M || wtype == OR_Q6_K) && K % 256 != 0) return 1;
    if (K % 32 != 0) return 1;
    return 0;
}

/* Decode a whole [N][K] weight matrix: wq [N][K], wsc [N][K/G], wmin [N][K/32] (Q4_K only). */
int oracle_decode(int wtype, const uint8_t* W, int64_t N, int64_t K, int8_t* wq, float* wsc, float* wmin) {
    if (!block_type(wtype) || check_k(wtype, K)) return 1;
    const int64_t G = group_size(wtype);
    for (int64_t n = 0; n < N; n++)
        decode_row(wtype, W + n * row_bytes(wtype, K), K, wq + n * K, wsc + n * (K / G),
                   wmin ? wmin + n * (K / 32) : NULL);
    return 0;
}

/* ---------------------------------------------------------------- per-group integer partials */
/*
 * I[m][n][g] = sum over k in group g of xq[m][k] * wq[n][k], exact in int32 ([R1] §2.1: the in-block
 * integer dot is exact; [NR] §2 inner sum).  wq is the decoded integer weight (int8), K-major.
 */
int oracle_partials(int wtype, const int8_t* xq, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                    int32_t* P) {
    if (wtype < 0 || wtype > 5 || check_k(wtype, K)) return 1;
    const int64_t G = group_size(wtype), ng = K / G;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            for (int64_t g = 0; g < ng; g++) {
                int32_t acc = 0;
                for (int64_t k = g * G; k < (g + 1) * G; k++)
#ifdef MUT_PARTIAL_TRANSPOSE
                    acc += (int32_t)xq[m * K + k] * (int32_t)wq[n * K + (k ^ 1)];
#else
                    acc += (int32_t)xq[m * K + k] * (int32_t)wq[n * K + k];
#endif
                P[(m * N + n) * ng + g] = acc;
            }
    return 0;
}

/* ---------------------------------------------------------------- folded 32-k block sums */
/*
 * Integer factor of each group's weight scale that is an exact integer: Q4_K's 6-bit sc_b per 32
 * ([R1] §2.2 (d*s) per sub-block), IQ1_M's (2s+1) per 16 ([IQ] Design: d(2s+1) per 16 values), q6_K's
 * int8 sc_h per 16 ([R1] §2.2).  Q8_0 / Q4_0 have none (factor 1).
 */
static void decode_row_int_scale(int wtype, const uint8_t* row, int64_t K, int32_t* isc) {
    if (wtype == OR_Q4_K) {
        for (int64_t sb = 0; sb < K / 256; sb++)
            for (int j = 0; j < 8; j++) isc[sb * 8 + j] = (int32_t)bits_le(row + sb * 144 + 4, 6u * (unsigned)j, 6);
    } else if (wtype == OR_IQ1_M) {
        for (int64_t sb = 0; sb < K / 256; sb++)
            for (int h = 0; h < 16; h++)
                isc[sb * 16 + h] = (int32_t)(2u * bits_le(row + sb * 76 + 68, 3u * (unsigned)h, 3) + 1u);
    } else if (wtype == OR_Q6_K) {
        for (int64_t sb = 0; sb < K / 256; sb++)
            for (int h = 0; h < 16; h++) isc[sb * 16 + h] = (int32_t)(int8_t)row[sb * 224 + h];
    } else {
        for (int64_t g = 0; g < K / 32; g++) isc[g] = 1;
    }
}

/*
 * A[m][n][b] = sum over k in 32-block b of xq[m][k] * wq[n][k] * isc[n][group(k)]: the exact integer
 * block sum with each group's integer scale factor folded in (the 32-k block dot of [R1] §2.1 on the
 * folded operand; for IQ1_M and q6_K the sum of the block's two per-16 dots, each times its factor).
 */
int oracle_block_sums(int wtype, const uint8_t* W, const int8_t* xq, int64_t M, int64_t N, int64_t K,
                      int32_t* A) {
    if (!block_type(wtype) || check_k(wtype, K)) return 1;
    const int64_t G = group_size(wtype), nb = K / 32;
    const int64_t ngi = (wtype == OR_Q8_0 || wtype == OR_Q4_0) ? K / 32 : K / G;
    int8_t* wq = (int8_t*)malloc((size_t)(N * K));
    float* wsc = (float*)malloc((size_t)(N * (K / G)) * sizeof(float));
    float* wmin = (float*)malloc((size_t)(N * nb) * sizeof(float));
    int32_t* isc = (int32_t*)malloc((size_t)(N * ngi) * sizeof(int32_t));
    if (!wq || !wsc || !wmin || !isc) { free(wq); free(wsc); free(wmin); free(isc); return 2; }
    oracle_decode(wtype, W, N, K, wq, wsc, wmin);
    for (int64_t n = 0; n < N; n++) decode_row_int_scale(wtype, W + n * row_bytes(wtype, K), K, isc + n * ngi);
    const int64_t gi = K / ngi;                           /* values per integer-scale group */
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            for (int64_t b = 0; b < nb; b++) {
                int64_t acc = 0;
                for (int64_t k = b * 32; k < b * 32 + 32; k++)
                    acc += (int64_t)xq[m * K + k] * (int64_t)wq[n * K + k] * (int64_t)isc[n * ngi + k / gi];
                A[(m * N + n) * nb + b] = (int32_t)acc;
            }
    free(wq); free(wsc); free(wmin); free(isc);
    return 0;
}

/* ---------------------------------------------------------------- blockwise product for one row pair */
/*
 * [NR] §2: out[m,n] = sum_kb (xs[m,kb] * wd[n,kb]) * sum_{k in kb} xq[m,k] * wq[n,k]
 * [R1] §3.2 reference frame: out += da * (ds * sum w*q + dm * sum q) per 32-block; here with the
 * library's f32 block sum s = d * sum(q), the min term is -(dmin*m_b) * s[m,b].
 * Per block b, in this order (f32, round to nearest, no fused multiply-add):
 *   Q8_0/Q4_0 : acc = acc + ((xd * wsc) * (float)I)
 *   Q4_K      : acc = acc + (((xd * wsc) * (float)I) - (wmin * s))
 *   IQ1_M,Q6_K: for h = 0, 1: acc = acc + ((xd * wsc_h) * (float)I_h)      (per-16 halves)
 */
static float block_dot_row(int wtype, const int8_t* xq, const float* xd, const float* xs,
                           const int8_t* wq, const float* wsc, const float* wmin, int64_t K) {
    float acc = 0.0f;
    for (int64_t b = 0; b < K / 32; b++) {
        if (wtype == OR_IQ1_M || wtype == OR_Q6_K) {
            for (int h = 0; h < 2; h++) {
                int32_t I = 0;
                for (int64_t k = b * 32 + 16 * h; k < b * 32 + 16 * h + 16; k++)
                    I += (int32_t)xq[k] * (int32_t)wq[k];
                float t = xd[b] * wsc[2 * b + h];
                float u = t * (float)I;
                acc = acc + u;
            }
        } else {
            int32_t I = 0;
            for (int64_t k = b * 32; k < b * 32 + 32; k++) I += (int32_t)xq[k] * (int32_t)wq[k];
#ifdef MUT_SCALE_INDEX
            float t = xd[b] * wsc[(b + 1) % (K / 32)];
#else
            float t = xd[b] * wsc[b];
#endif
            float u = t * (float)I;
#ifndef MUT_DROP_MIN
            if (wtype == OR_Q4_K) {
                float v = wmin[b] * xs[b];
#ifdef MUT_MIN_SIGN
                u = u + v;                                  /* min term added instead of subtracted */
#else
                u = u - v;
#endif
            }
#endif
            acc = acc + u;
        }
    }
    return acc;
}

/*
 * Dense blockwise GEMM: out f32 [M][N] for weights W (raw blocks, [N] rows) and q8_1 activations
 * (q [M][K], d [M][K/32], s [M][K/32]).
 */
int oracle_gemm(int wtype, const uint8_t* W, const int8_t* xq, const float* xd, const float* xs,
                int64_t M, int64_t N, int64_t K, float* out) {
    if (!block_type(wtype) || check_k(wtype, K)) return 1;
    const int64_t G = group_size(wtype);
    int8_t* wq = (int8_t*)malloc((size_t)(N * K));
    float* wsc = (float*)malloc((size_t)(N * (K / G)) * sizeof(float));
    float* wmin = (float*)malloc((size_t)(N * (K / 32)) * sizeof(float));
    if (!wq || !wsc || !wmin) { free(wq); free(wsc); free(wmin); return 2; }
    memset(wmin, 0, (size_t)(N * (K / 32)) * sizeof(float));
    oracle_decode(wtype, W, N, K, wq, wsc, wmin);
    const int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            out[m * N + n] = block_dot_row(wtype, xq + m * K, xd + m * nb, xs + m * nb, wq + n * K,
                                           wsc + n * (K / G), wmin + n * nb, K);
    free(wq); free(wsc); free(wmin);
    return 0;
}

/* Same product for a chosen subset of activation rows (rows[i] in [0, M)): out [nrows][N]. */
int oracle_gemm_rows(int wtype, const uint8_t* W, const int8_t* xq, const float* xd, const float* xs,
                     int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows, float* out) {
    if (!block_type(wtype) || check_k(wtype, K)) return 1;
    for (int64_t i = 0; i < nrows; i++)
        if (rows[i] < 0 || rows[i] >= M) return 1;
    const int64_t G = group_size(wtype);
    int8_t* wq = (int8_t*)malloc((size_t)(N * K));
    float* wsc = (float*)malloc((size_t)(N * (K / G)) * sizeof(float));
    float* wmin = (float*)malloc((size_t)(N * (K / 32)) * sizeof(float));
    if (!wq || !wsc || !wmin) { free(wq); free(wsc); free(wmin); return 2; }
    memset(wmin, 0, (size_t)(N * (K / 32)) * sizeof(float));
    oracle_decode(wtype, W, N, K, wq, wsc, wmin);
    const int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; i++) {
        int64_t m = rows[i];
        for (int64_t n = 0; n < N; n++)
            out[i * N + n] = block_dot_row(wtype, xq + m * K, xd + m * nb, xs + m * nb, wq + n * K,
                                           wsc + n * (K / G), wmin + n * nb, K);
    }
    free(wq); free(wsc); free(wmin);
    return 0;
}

/* ---------------------------------------------------------------- W8A8 per-channel */
/*
 * [W8]: int8 W [N][K] (checkpoint layout, stride K), int8 X [M][K], per-channel f32 ws [N], per-token
 * f32 xs [M]; int32 accumulation over the full K; epilogue out = bf16(((float)I * xs[m]) * ws[n]),
 * round to nearest even.  out holds bf16 bit patterns [M][N].
 */
int oracle_w8a8(const int8_t* W, const float* ws, const int8_t* X, const float* xs, int64_t M, int64_t N,
                int64_t K, uint16_t* out) {
    if (K <= 0 || K % 32 != 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            int64_t I = 0;
            for (int64_t k = 0; k < K; k++) I += (int64_t)X[m * K + k] * (int64_t)W[n * K + k];
            float f = (float)(int32_t)I;
#ifdef MUT_W8A8_SCALE_SWAP
            float t = f * xs[n % M];
            float u = t * ws[m % N];
#else
            float t = f * xs[m];
            float u = t * ws[n];
#endif
            out[m * N + n] = float_to_bf16_rne(u);
        }
    return 0;
}

/* W8A8 32-k integer partials I[m][n][k/32] (for the debug-partials comparison). */
int oracle_w8a8_partials(const int8_t* W, const int8_t* X, int64_t M, int64_t N, int64_t K, int32_t* P) {
    return oracle_partials(OR_W8A8, X, W, M, N, K, P);
}

/* ---------------------------------------------------------------- MoE (MUL_MAT_ID) */
/*
 * [IQ] PR description: MUL_MAT_ID, each token times each of its routed experts.  For token t and slot
 * j with expert e = ids[t][j]: out[t][j][:] = blockwise product of expert e's weights (rows [N], raw
 * blocks, experts stored back to back) with activation row t.  ids must lie in [0, n_experts).
 */
int oracle_gemm_id(int wtype, const uint8_t* W, int64_t n_experts, const int8_t* xq, const float* xd,
                   const float* xs, const int32_t* ids, int64_t n_slots, int64_t M, int64_t N, int64_t K,
                   float* out) {
    if (!block_type(wtype) || check_k(wtype, K) || n_experts <= 0 || n_slots <= 0) return 1;
    for (int64_t i = 0; i < M * n_slots; i++)
        if (ids[i] < 0 || ids[i] >= n_experts) return 1;
    const int64_t G = group_size(wtype), nb = K / 32, rb = row_bytes(wtype, K);
    int8_t* wq = (int8_t*)malloc((size_t)(N * K));
    float* wsc = (float*)malloc((size_t)(N * (K / G)) * sizeof(float));
    float* wmin = (float*)malloc((size_t)(N * nb) * sizeof(float));
    if (!wq || !wsc || !wmin) { free(wq); free(wsc); free(wmin); return 2; }
    for (int64_t e = 0; e < n_experts; e++) {
        int used = 0;
        for (int64_t i = 0; i < M * n_slots; i++) used |= (ids[i] == e);
        if (!used) continue;
        memset(wmin, 0, (size_t)(N * nb) * sizeof(float));
        oracle_decode(wtype, W + e * N * rb, N, K, wq, wsc, wmin);
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < M * n_slots; i++) {
            if (ids[i] != e) continue;
            int64_t t = i / n_slots;
#ifdef MUT_MOE_SLOT_MAJOR
            const int64_t orow = (i % n_slots) * M + t;      /* output rows slot-major instead of token-major */
#else
            const int64_t orow = i;
#endif
            for (int64_t n = 0; n < N; n++)
                out[orow * N + n] = block_dot_row(wtype, xq + t * K, xd + t * nb, xs + t * nb, wq + n * K,
                                                  wsc + n * (K / G), wmin + n * nb, K);
        }
    }
    free(wq); free(wsc); free(wmin);
    return 0;
}

/* ---------------------------------------------------------------- exported scalar helpers (for pins) */
float oracle_half_to_float(uint16_t h) { return half_to_float(h); }
uint16_t oracle_float_to_bf16(float f) { return float_to_bf16_rne(f); }
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
